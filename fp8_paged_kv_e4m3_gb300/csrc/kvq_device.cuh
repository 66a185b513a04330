// kvq_device.cuh -- sm_103a device primitives used by the kvq kernels:
// mbarriers, 1-D bulk TMA copies, ldmatrix / movmatrix / mma.sync fragments,
// the bitcast E4M3 -> fp16 decoder, and bounded waits.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "kvq.h"

namespace kvq {

// ---------------------------------------------------------------------------
// error reporting

__device__ __forceinline__ void report(int32_t *err_flag, int bits)
{
    if (err_flag) atomicOr(err_flag, bits);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start before the previous kernel in the stream has
// finished; it must call grid_dependency_wait() before touching any memory
// that earlier work writes.  launch_dependents() lets the next kernel start
// its own prologue early.  Both are no-ops when there is no such dependency.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// shared-memory addresses and mbarriers

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of an mbarrier, but never forever: after
// `limit_ns` of wall time (or once another warp has raised *abort) it gives
// up, raises *abort, reports KVQ_DEV_TIMEOUT and returns false.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort, int32_t *err_flag,
                                                  uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0u) {
            if (abort && *abort) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                if (abort) *abort = 1;
                report(err_flag, KVQ_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// 1-D bulk TMA: global -> shared, completion counted on an mbarrier.
// Both addresses 16-byte aligned, size a multiple of 16.

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_1d(uint32_t dst_smem, const void *src, uint32_t bytes,
                                            uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst_smem),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// ---------------------------------------------------------------------------
// warp-level matrix fragments (mma.sync m16n8k16, fp16 x fp16 -> fp32)

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// two fp32 -> packed f16x2 (lo in the low half), round to nearest even
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// two fp32 lanes per instruction (sm_100 and later): d = a * b + c and
// d = a + b, each lane rounded to nearest as its scalar form
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b)
{
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// maximum of three (sm_100 and later), NaN handling as fmaxf's
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// Bitcast E4M3 -> fp16 decoder ([P2] Changes: "exact bitcast E4M3 software
// decoder").  An E4M3 byte s.eeee.mmm placed as the fp16 bit pattern
// s.0eeee.mmm0000000 is the same number times 2^-8, exactly, for every
// finite code (normals and subnormals alike, since both formats keep the
// mantissa bits in the same place below the exponent).  The 2^8 is folded
// into the hoisted per-layer scale.  Codes 0x7F / 0xFF (NaN) become the
// finite fp16 value 1.875; the quantiser never writes them for finite input.
//
// A 32-bit word of four bytes b3.b2.b1.b0 yields two f16x2 words:
//   dec_lo -> (b0 in the low half, b2 in the high half)
//   dec_hi -> (b1 in the low half, b3 in the high half)
// i.e. each output half takes the byte sitting in the high byte of that
// half, after an 8-bit shift for dec_lo.
__device__ __forceinline__ uint32_t dec_hi(uint32_t x)
{
    return ((x >> 1) & 0x3F803F80u) | (x & 0x80008000u);
}

__device__ __forceinline__ uint32_t dec_lo(uint32_t x)
{
    return dec_hi(x << 8);
}

// Hardware E4M3 -> fp16 conversion (exact: every E4M3 value is an fp16
// value).  cvt_lo takes bytes 0,1 of x, cvt_hi bytes 2,3; the lower byte
// becomes the lower half.  Unlike the bitcast decoder the result is the
// value itself, not value * 2^-8.
__device__ __forceinline__ uint32_t cvt_lo(uint32_t x)
{
    uint32_t d;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, l;\n\t}"
        : "=r"(d) : "r"(x));
    return d;
}

__device__ __forceinline__ uint32_t cvt_hi(uint32_t x)
{
    uint32_t d;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, h;\n\t}"
        : "=r"(d) : "r"(x));
    return d;
}

}  // namespace kvq
