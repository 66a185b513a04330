// kvq_noalloc.cu -- decode / verify attention for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand us a workspace: code running inside
// another framework's memory pool that forbids foreign cudaMalloc calls,
// plugins loaded into a process whose allocator they do not own, or
// real-time paths where any allocation is banned after start-up.  For them,
// paged_decode_attn_e4m3_noalloc uses a fixed scratch buffer that lives in
// this library's own device memory (a file-scope __device__ array), so the
// call itself allocates nothing.
//
// The buffer is KVQ_NOALLOC_SCRATCH_BYTES (16 MiB) per device.  Every GPU
// that loads the library holds it until the process exits.  All calls on a
// device share it: two calls whose GPU work overlaps (for example on two
// streams) race on it, so callers must order them.  The buffer keeps the
// previous call's contents; nothing in it needs to start at zero, because
// the attention kernel writes every partial result the combine then reads.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "kvq.h"

namespace {

__device__ __align__(256) unsigned char kvq_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;

// The looked-up address of the scratch buffer on one device, and the context
// it belongs to.  A device reset (cudaDeviceReset) ends the primary context;
// the runtime then loads the module again in a new context, where the buffer
// may sit elsewhere, so an address is used only in the context it was looked
// up in.
struct ScratchEntry {
    unsigned long long ctx_id;
    void *ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Driver calls resolved through the runtime (no link against the driver
// library): the current context and its process-unique id.
using CtxGetCurrentFn = int (*)(void **);
using CtxGetIdFn = int (*)(void *, unsigned long long *);
std::once_flag g_driver_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

bool current_context_id(unsigned long long *id)
{
    std::call_once(g_driver_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(fn);
    });
    void *ctx = nullptr;
    if (!g_ctx_get_current || !g_ctx_get_id) return false;
    if (g_ctx_get_current(&ctx) != 0 || !ctx) return false;
    return g_ctx_get_id(ctx, id) == 0;
}

// Device address of the scratch buffer on the current device.  The name
// kvq_noalloc_scratch in host code is only a handle for the runtime, not an
// address a kernel may use; the address comes from cudaGetSymbolAddress,
// looked up with the device current, once per device and context (the
// first call on a device, and the first after a device reset).
int scratch_for_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx)) {
        // no context current on this thread yet: cudaSetDevice makes the
        // device's primary context current (and allocates nothing)
        if (cudaSetDevice(dev) != cudaSuccess || !current_context_id(&ctx)) return KVQ_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    ScratchEntry &e = g_scratch[dev];
    if (!e.ptr || e.ctx_id != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, kvq_noalloc_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
        e.ptr = p;
        e.ctx_id = ctx;
    }
    *out = e.ptr;
    return KVQ_OK;
}

}  // namespace

extern "C" int paged_decode_attn_e4m3_noalloc(const void *q, const uint8_t *k_cache,
                                              const uint8_t *v_cache, int64_t num_pages,
                                              const int32_t *block_tables,
                                              const int32_t *context_lens, float k_scale,
                                              float v_scale, const int32_t *topk_idx,
                                              const int32_t *topk_lens, void *out,
                                              const kvq_attn_params *p, int32_t *err_flag,
                                              void *stream)
{
    const int32_t splits = kvq_attn_num_splits(p);        // validates the parameters
    if (splits < 0) return splits;
    const size_t need = kvq_attn_workspace_bytes(p);
    if (need > KVQ_NOALLOC_SCRATCH_BYTES) return KVQ_ERR_WORKSPACE;   // too big for the buffer
    void *scratch = nullptr;
    const int st = scratch_for_current_device(&scratch);
    if (st != KVQ_OK) return st;
    return paged_decode_attn_e4m3(q, k_cache, v_cache, num_pages, block_tables, context_lens,
                                  k_scale, v_scale, topk_idx, topk_lens,
                                  static_cast<float *>(scratch), KVQ_NOALLOC_SCRATCH_BYTES, out, p,
                                  err_flag, stream);
}
