"""GB300 (sm_103a) causal grouped-query attention: forward and backward.

The compute lives in libattn_gqa.so (hand-written CUDA kernels behind the C
ABI of include/attn_gqa.h); this package is its thin Python binding plus the
seeded synthetic-input generators (``synth``).  Build the library with
``build_ext.build()``.
"""
from .binding import (ALGOS, MASKS, ATTN_ALGO_AUTO, ATTN_ALGO_DECODE, ATTN_ALGO_GENERIC,
                      ATTN_ALGO_TCGEN05, ATTN_BF16, ATTN_F16, ATTN_F32, EXPORTED, AttnError,
                      attn_bwd, attn_bwd_varlen, attn_fwd, attn_fwd_decode_noalloc,
                      attn_fwd_masked, attn_fwd_paged, attn_fwd_staged, attn_fwd_varlen,
                      attn_lse_combine, device_status, kernel_launches, last_error,
                      library_path, load_library, pack_mask, set_wait_limit)

__all__ = ["ALGOS", "MASKS", "ATTN_ALGO_AUTO", "ATTN_ALGO_DECODE", "ATTN_ALGO_GENERIC",
           "ATTN_ALGO_TCGEN05", "ATTN_BF16", "ATTN_F16", "ATTN_F32", "EXPORTED", "AttnError",
           "attn_bwd", "attn_bwd_varlen", "attn_fwd", "attn_fwd_decode_noalloc",
           "attn_fwd_masked", "attn_fwd_paged", "attn_fwd_staged", "attn_fwd_varlen",
           "attn_lse_combine", "device_status", "kernel_launches", "last_error",
           "library_path", "load_library", "pack_mask", "set_wait_limit"]
