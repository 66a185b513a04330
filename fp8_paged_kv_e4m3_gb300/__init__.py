"""GB300-native calibrated E4M3 paged KV cache for decode / MTP-verify attention.

The compute path is the CUDA library ``libkvq.so`` (built from ``csrc/``);
this package is its thin Python binding.  The library is loaded on first use
and its absence is an error: there is no CPU fallback.
"""
