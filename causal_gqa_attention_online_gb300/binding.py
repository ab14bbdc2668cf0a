"""Thin ctypes binding of libattn_gqa (the C ABI in include/attn_gqa.h).

Argument marshalling only: torch tensors are used as device memory and
streams, their data pointers are handed to the C entry points, and every step
of the attention runs in the library's CUDA kernels.  There is no CPU path:
if the library or a CUDA device is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import build_ext

ATTN_F32, ATTN_F16, ATTN_BF16 = 0, 1, 2
ATTN_ALGO_AUTO, ATTN_ALGO_GENERIC, ATTN_ALGO_TCGEN05, ATTN_ALGO_DECODE = 0, 1, 2, 3
ATTN_ALGO_MMA = 4
ALGOS = {"auto": 0, "generic": 1, "tcgen05": 2, "decode": 3, "mma": 4}
# bottom-right causal (the pages' rule), top-left causal, none
MASKS = {"causal": 0, "causal_top_left": 1, "none": 2}
_DTYPE_CODE = {torch.float32: ATTN_F32, torch.float16: ATTN_F16, torch.bfloat16: ATTN_BF16}

EXPORTED = ("attn_fwd", "attn_fwd_varlen", "attn_fwd_algo", "attn_fwd_varlen_algo",
            "attn_fwd_ex", "attn_fwd_varlen_ex", "attn_fwd_paged", "attn_fwd_masked",
            "attn_bwd", "attn_bwd_varlen", "attn_lse_combine", "attn_lse_combine_ex",
            "attn_fwd_decode_noalloc", "attn_fwd_staged", "attn_last_error",
            "attn_device_status", "attn_set_wait_limit", "attn_kernel_launches", "attn_version")

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    """A non-zero status from the library."""

    def __init__(self, status: int, message: str):
        super().__init__(f"attn status {status}: {message}")
        self.status = status


def library_path() -> str:
    return build_ext.LIB_PATH


def load_library(path: str | None = None):
    """Load libattn_gqa.so (built in-tree by ``build_ext.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or build_ext.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with causal_gqa_attention_online_gb300.build_ext."
                "build() (no CPU fallback exists)")
        lib = ctypes.CDLL(path)
        vp, ip, fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        common = [vp, vp, vp, vp, vp] + [ip] * 7 + [vp, vp, ip, fp, ip]
        varlen = [vp, vp, vp, vp, vp] + [ip] * 9 + [vp, vp, ip, fp, ip]
        lib.attn_fwd.argtypes = common + [vp]
        lib.attn_fwd_varlen.argtypes = varlen + [vp]
        lib.attn_fwd_algo.argtypes = common + [ip, vp]
        lib.attn_fwd_varlen_algo.argtypes = varlen + [ip, vp]
        lib.attn_fwd_ex.argtypes = common[:-1] + [ip, ip, ip, vp]
        lib.attn_fwd_varlen_ex.argtypes = varlen[:-1] + [ip, ip, ip, vp]
        lib.attn_fwd_ex.restype = ip
        lib.attn_fwd_paged.argtypes = [vp] * 5 + [ip] * 6 + [vp, ip, ip, ip, vp, vp, ip, fp, ip,
                                                             ip, ip, vp]
        lib.attn_fwd_paged.restype = ip
        lib.attn_fwd_masked.argtypes = [vp] * 5 + [ip] * 7 + [vp, vp, vp, ip, ip, ip, fp, ip, ip,
                                                             ip, vp]
        lib.attn_fwd_masked.restype = ip
        lib.attn_fwd_varlen_ex.restype = ip
        lib.attn_fwd_decode_noalloc.argtypes = common + [vp]
        lib.attn_fwd_decode_noalloc.restype = ip
        for f in (lib.attn_fwd, lib.attn_fwd_varlen, lib.attn_fwd_algo, lib.attn_fwd_varlen_algo):
            f.restype = ip
        ullp = ctypes.POINTER(ctypes.c_ulonglong)
        lib.attn_fwd_staged.argtypes = ([vp] * 10 + [ip] * 7 + [vp] * 4 + [ip, fp, ip, ip] +
                                        [ullp, ullp, vp])
        lib.attn_fwd_staged.restype = ip
        lib.attn_bwd.argtypes = [vp] * 9 + [ip] * 7 + [vp, vp, ip, fp, ip, ip, ip, vp]
        lib.attn_bwd_varlen.argtypes = [vp] * 9 + [ip] * 9 + [vp, vp, ip, fp, ip, ip, ip, vp]
        lib.attn_lse_combine.argtypes = [vp, vp, vp, vp, ip, ctypes.c_longlong, ip, ip, vp]
        lib.attn_lse_combine.restype = ip
        lib.attn_lse_combine_ex.argtypes = [vp, vp, vp, vp, ip, ctypes.c_longlong, ip, ip, ip, vp]
        lib.attn_lse_combine_ex.restype = ip
        lib.attn_last_error.argtypes = []
        lib.attn_last_error.restype = ctypes.c_char_p
        lib.attn_device_status.argtypes = [ctypes.POINTER(ctypes.c_int)]
        lib.attn_device_status.restype = ip
        lib.attn_set_wait_limit.argtypes = [ctypes.c_ulonglong]
        lib.attn_set_wait_limit.restype = ctypes.c_ulonglong
        lib.attn_kernel_launches.argtypes = []
        lib.attn_kernel_launches.restype = ctypes.c_ulonglong
        lib.attn_version.argtypes = []
        lib.attn_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def last_error() -> str:
    return load_library().attn_last_error().decode()


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load_library().attn_kernel_launches())


def device_status() -> tuple[int, int]:
    """(status, detail) of the current device's status word (synchronises)."""
    d = ctypes.c_int(0)
    st = load_library().attn_device_status(ctypes.byref(d))
    return st, d.value


def set_wait_limit(ns: int) -> int:
    """Limit (ns) of the tcgen05 kernels' mbarrier waits for later launches;
    0 restores the default (2 s).  Returns the previous limit.  A diagnostic
    aid: a short limit makes a launch time out, reported by device_status()."""
    return int(load_library().attn_set_wait_limit(int(ns)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int):
    if rc != 0:
        raise AttnError(rc, last_error())


def _check_tensor(name, t, dtype, numel, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected {numel}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def attn_fwd(q, k, v, o=None, lse=None, *, seqlens_q=None, seqlens_k=None, window=0,
             scale=None, algo="auto", mask="causal", stream=None, want_lse=True):
    """Padded layout: q [B,Q,Hq,D], k [B,K,Hkv,D], v [B,K,Hkv,Dv] CUDA tensors.
    ``mask``: "causal" (bottom-right, the default), "causal_top_left" or "none".

    Returns (o [B,Q,Hq,Dv], lse [B,Q,Hq] float32 or None)."""
    lib = load_library()
    B, Q, Hq, D = q.shape
    K, Hkv = k.shape[1], k.shape[2]
    Dv = v.shape[3]
    dev = q.device
    if o is None:
        o = torch.empty((B, Q, Hq, Dv), dtype=q.dtype, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, Q, Hq), dtype=torch.float32, device=dev)
    for name, t, n in (("q", q, B * Q * Hq * D), ("k", k, B * K * Hkv * D),
                       ("v", v, B * K * Hkv * Dv), ("o", o, B * Q * Hq * Dv)):
        _check_tensor(name, t, q.dtype, n, dev)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, B * Q * Hq, dev)
    for name, t in (("seqlens_q", seqlens_q), ("seqlens_k", seqlens_k)):
        if t is not None:
            _check_tensor(name, t, torch.int32, B, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib.attn_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Q, K, D, Dv,
                         _ptr(seqlens_q), _ptr(seqlens_k), int(window), float(scale), MASKS[mask],
                         _DTYPE_CODE[q.dtype], ALGOS[algo], _stream_ptr(stream))
    _check(rc)
    return o, lse


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_q, max_k, o=None, lse=None, *,
                    window=0, scale=None, algo="auto", mask="causal", stream=None,
                    want_lse=True):
    """Packed layout: q [Tq,Hq,D], k [Tk,Hkv,D], v [Tk,Hkv,Dv], int32
    cumulative lengths [B+1] on the device.  ``mask`` as in attn_fwd.
    Returns (o [Tq,Hq,Dv], lse [Tq,Hq])."""
    lib = load_library()
    Tq, Hq, D = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    Dv = v.shape[2]
    B = cu_seqlens_q.numel() - 1
    dev = q.device
    if o is None:
        o = torch.empty((Tq, Hq, Dv), dtype=q.dtype, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=dev)
    for name, t, n in (("q", q, Tq * Hq * D), ("k", k, Tk * Hkv * D), ("v", v, Tk * Hkv * Dv),
                       ("o", o, Tq * Hq * Dv)):
        _check_tensor(name, t, q.dtype, n, dev)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, Tq * Hq, dev)
    _check_tensor("cu_seqlens_q", cu_seqlens_q, torch.int32, B + 1, dev)
    _check_tensor("cu_seqlens_k", cu_seqlens_k, torch.int32, B + 1, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib.attn_fwd_varlen_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                Tq, Tk, int(max_q), int(max_k), D, Dv, _ptr(cu_seqlens_q),
                                _ptr(cu_seqlens_k), int(window), float(scale), MASKS[mask],
                                _DTYPE_CODE[q.dtype], ALGOS[algo], _stream_ptr(stream))
    _check(rc)
    return o, lse


def attn_bwd(q, k, v, o, lse, dout, dq=None, dk=None, dv=None, *, seqlens_q=None,
             seqlens_k=None, window=0, scale=None, algo="auto", mask="causal", stream=None):
    """Gradients of attn_fwd (padded layout) for the output gradient ``dout``
    [B,Q,Hq,Dv]; ``o`` and ``lse`` are attn_fwd's outputs for q, k, v with the
    same seqlens / window / scale / mask.  ``algo``: "auto", "generic" (CUDA
    cores), "mma" (mma.sync tensor cores) or "tcgen05" (tcgen05 dQ and dK/dV
    kernels).  Returns (dq, dk, dv)."""
    lib = load_library()
    B, Q, Hq, D = q.shape
    K, Hkv = k.shape[1], k.shape[2]
    Dv = v.shape[3]
    dev = q.device
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, n in (("q", q, B * Q * Hq * D), ("k", k, B * K * Hkv * D),
                       ("v", v, B * K * Hkv * Dv), ("o", o, B * Q * Hq * Dv),
                       ("dout", dout, B * Q * Hq * Dv), ("dq", dq, B * Q * Hq * D),
                       ("dk", dk, B * K * Hkv * D), ("dv", dv, B * K * Hkv * Dv)):
        _check_tensor(name, t, q.dtype, n, dev)
    _check_tensor("lse", lse, torch.float32, B * Q * Hq, dev)
    for name, t in (("seqlens_q", seqlens_q), ("seqlens_k", seqlens_k)):
        if t is not None:
            _check_tensor(name, t, torch.int32, B, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                      _ptr(dk), _ptr(dv), B, Hq, Hkv, Q, K, D, Dv, _ptr(seqlens_q),
                      _ptr(seqlens_k), int(window), float(scale), MASKS[mask],
                      _DTYPE_CODE[q.dtype], ALGOS[algo], _stream_ptr(stream))
    _check(rc)
    return dq, dk, dv


def attn_bwd_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_q, max_k, dq=None,
                    dk=None, dv=None, *, window=0, scale=None, algo="auto", mask="causal",
                    stream=None):
    """attn_bwd on the packed layout of attn_fwd_varlen.  Returns (dq, dk, dv);
    rows outside every sequence are left as they were (zeros when the
    outputs are allocated here)."""
    lib = load_library()
    Tq, Hq, D = q.shape
    Tk, Hkv = k.shape[0], k.shape[1]
    Dv = v.shape[2]
    B = cu_seqlens_q.numel() - 1
    dev = q.device
    dq = torch.zeros_like(q) if dq is None else dq
    dk = torch.zeros_like(k) if dk is None else dk
    dv = torch.zeros_like(v) if dv is None else dv
    for name, t, n in (("q", q, Tq * Hq * D), ("k", k, Tk * Hkv * D), ("v", v, Tk * Hkv * Dv),
                       ("o", o, Tq * Hq * Dv), ("dout", dout, Tq * Hq * Dv),
                       ("dq", dq, Tq * Hq * D), ("dk", dk, Tk * Hkv * D),
                       ("dv", dv, Tk * Hkv * Dv)):
        _check_tensor(name, t, q.dtype, n, dev)
    _check_tensor("lse", lse, torch.float32, Tq * Hq, dev)
    _check_tensor("cu_seqlens_q", cu_seqlens_q, torch.int32, B + 1, dev)
    _check_tensor("cu_seqlens_k", cu_seqlens_k, torch.int32, B + 1, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib.attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                             _ptr(dk), _ptr(dv), B, Hq, Hkv, Tq, Tk, int(max_q), int(max_k), D,
                             Dv, _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(window),
                             float(scale), MASKS[mask], _DTYPE_CODE[q.dtype], ALGOS[algo],
                             _stream_ptr(stream))
    _check(rc)
    return dq, dk, dv


def attn_fwd_decode_noalloc(q, k, v, o, lse=None, *, seqlens_q=None, seqlens_k=None, window=0,
                            scale=None, stream=None):
    """attn_fwd's split-KV decode with its scratch in the library's fixed
    device array: the call allocates nothing (``o`` and ``lse`` are the
    caller's).  For callers that may not allocate device memory while
    attention runs.  Calls that overlap on one GPU race on the shared array."""
    lib = load_library()
    B, Q, Hq, D = q.shape
    K, Hkv = k.shape[1], k.shape[2]
    Dv = v.shape[3]
    dev = q.device
    for name, t, n in (("q", q, B * Q * Hq * D), ("k", k, B * K * Hkv * D),
                       ("v", v, B * K * Hkv * Dv), ("o", o, B * Q * Hq * Dv)):
        _check_tensor(name, t, q.dtype, n, dev)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, B * Q * Hq, dev)
    for name, t in (("seqlens_q", seqlens_q), ("seqlens_k", seqlens_k)):
        if t is not None:
            _check_tensor(name, t, torch.int32, B, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib.attn_fwd_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                     Q, K, D, Dv, _ptr(seqlens_q), _ptr(seqlens_k), int(window),
                                     float(scale), _DTYPE_CODE[q.dtype], _stream_ptr(stream))
    _check(rc)
    return o, lse


def attn_lse_combine(o_parts, lse_parts, o=None, lse=None, *, dtype=torch.float32, stream=None):
    """Merge split-KV partials: o_parts [S,rows,Dv] fp32, lse_parts [S,rows] fp32."""
    lib = load_library()
    S, rows, Dv = o_parts.shape
    dev = o_parts.device
    if o is None:
        o = torch.empty((rows, Dv), dtype=dtype, device=dev)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=dev)
    _check_tensor("o_parts", o_parts, torch.float32, S * rows * Dv, dev)
    _check_tensor("lse_parts", lse_parts, torch.float32, S * rows, dev)
    _check_tensor("o", o, o.dtype, rows * Dv, dev)
    rc = lib.attn_lse_combine(_ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse), S, rows, Dv,
                              _DTYPE_CODE[o.dtype], _stream_ptr(stream))
    _check(rc)
    return o, lse


def attn_lse_combine_parts(o_parts, lse_parts, o=None, lse=None, *, stream=None):
    """Merge partials [S, rows, Dv] in their storage dtype (fp32, fp16 or bf16;
    as attn_fwd wrote them) by their LSE [S, rows]; o is in that dtype."""
    lib = load_library()
    S, rows, Dv = o_parts.shape
    dev = o_parts.device
    if o is None:
        o = torch.empty((rows, Dv), dtype=o_parts.dtype, device=dev)
    if lse is None:
        lse = torch.empty((rows,), dtype=torch.float32, device=dev)
    _check_tensor("o_parts", o_parts, o_parts.dtype, S * rows * Dv, dev)
    _check_tensor("lse_parts", lse_parts, torch.float32, S * rows, dev)
    _check_tensor("o", o, o_parts.dtype, rows * Dv, dev)
    code = _DTYPE_CODE[o_parts.dtype]
    rc = lib.attn_lse_combine_ex(_ptr(o_parts), _ptr(lse_parts), _ptr(o), _ptr(lse), S, rows, Dv,
                                 code, code, _stream_ptr(stream))
    _check(rc)
    return o, lse


def attn_fwd_staged(hq, hk, hv, q, k, v, o, lse=None, ho=None, hlse=None, *, seqlens_q=None,
                    seqlens_k=None, seqlens_q_dev=None, seqlens_k_dev=None, window=0, scale=None,
                    chunks=0, stream=None):
    """attn_fwd on host tensors (padded layout; page-locked for overlap): per
    group of sequences, copy in the valid rows, run attention, copy the
    outputs back, the copies of one group overlapping the attention of the
    next.  ``q, k, v, o, lse`` are device staging buffers of the same shapes.
    ``seqlens_q/k`` are int32 CPU tensors; their device copies may be given
    as ``seqlens_q_dev/k_dev`` (else they are copied here, on ``stream``).
    Returns (ho, hlse, bytes_in, bytes_out); the host outputs are complete
    once ``stream`` reaches this point."""
    lib = load_library()
    B, Q, Hq, D = hq.shape
    K, Hkv = hk.shape[1], hk.shape[2]
    Dv = hv.shape[3]
    dev = q.device
    if ho is None:
        ho = torch.empty((B, Q, Hq, Dv), dtype=hq.dtype).pin_memory()
    if hlse is None and lse is not None:
        hlse = torch.empty((B, Q, Hq), dtype=torch.float32).pin_memory()
    cpu = torch.device("cpu")
    for name, t, n in (("hq", hq, B * Q * Hq * D), ("hk", hk, B * K * Hkv * D),
                       ("hv", hv, B * K * Hkv * Dv), ("ho", ho, B * Q * Hq * Dv)):
        _check_tensor(name, t, hq.dtype, n, cpu)
    for name, t, n in (("q", q, B * Q * Hq * D), ("k", k, B * K * Hkv * D),
                       ("v", v, B * K * Hkv * Dv), ("o", o, B * Q * Hq * Dv)):
        _check_tensor(name, t, hq.dtype, n, dev)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, B * Q * Hq, dev)
        _check_tensor("hlse", hlse, torch.float32, B * Q * Hq, cpu)
    dsq, dsk = seqlens_q_dev, seqlens_k_dev
    st = stream if stream is not None else torch.cuda.current_stream()
    if seqlens_q is not None:
        _check_tensor("seqlens_q", seqlens_q, torch.int32, B, cpu)
        if dsq is None:
            with torch.cuda.stream(st):
                dsq = seqlens_q.to(dev, non_blocking=True)
        _check_tensor("seqlens_q_dev", dsq, torch.int32, B, dev)
    if seqlens_k is not None:
        _check_tensor("seqlens_k", seqlens_k, torch.int32, B, cpu)
        if dsk is None:
            with torch.cuda.stream(st):
                dsk = seqlens_k.to(dev, non_blocking=True)
        _check_tensor("seqlens_k_dev", dsk, torch.int32, B, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    bin_, bout = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    rc = lib.attn_fwd_staged(_ptr(hq), _ptr(hk), _ptr(hv), _ptr(ho), _ptr(hlse), _ptr(q), _ptr(k),
                             _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Q, K, D, Dv, _ptr(dsq),
                             _ptr(dsk), _ptr(seqlens_q), _ptr(seqlens_k), int(window),
                             float(scale), _DTYPE_CODE[hq.dtype], int(chunks),
                             ctypes.byref(bin_), ctypes.byref(bout), _stream_ptr(st))
    _check(rc)
    return ho, hlse, bin_.value, bout.value


def pack_mask(allow: torch.Tensor) -> torch.Tensor:
    """Bit-pack a boolean mask [B, Hm, Q, K] into the int32 words attn_fwd_masked
    reads: bit k % 32 of word k / 32 of a row is key k, rows padded to a
    multiple of 128 keys.  Returns [B, Hm, Q, 4 * ceil(K / 128)] int32 on the
    mask's device."""
    B, Hm, Q, K = allow.shape
    kp = (K + 127) // 128 * 128
    bits = torch.zeros((B, Hm, Q, kp), dtype=torch.int64, device=allow.device)
    bits[..., :K] = allow.to(torch.int64)
    bits = bits.view(B, Hm, Q, kp // 32, 32)
    weights = torch.ones(32, dtype=torch.int64, device=allow.device) << torch.arange(
        32, device=allow.device)
    words = (bits * weights).sum(dim=-1)
    words = torch.where(words >= 2**31, words - 2**32, words)
    return words.to(torch.int32).contiguous()


def attn_fwd_masked(q, k, v, mask_words, o=None, lse=None, *, seqlens_q=None, seqlens_k=None,
                    window=0, scale=None, algo="auto", mask="none", stream=None, want_lse=True):
    """Padded layout with an arbitrary mask: ``mask_words`` int32 [B, Hm, Q, W]
    (``pack_mask`` of a boolean [B, Hm, Q, K]; Hm = 1 or Hq), ANDed with
    ``mask`` ("none" by default, or a causal mode) and ``window``.
    Returns (o, lse)."""
    lib = load_library()
    B, Q, Hq, D = q.shape
    K, Hkv = k.shape[1], k.shape[2]
    Dv = v.shape[3]
    dev = q.device
    Hm, W = mask_words.shape[1], mask_words.shape[3]
    if o is None:
        o = torch.empty((B, Q, Hq, Dv), dtype=q.dtype, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, Q, Hq), dtype=torch.float32, device=dev)
    for name, t, n in (("q", q, B * Q * Hq * D), ("k", k, B * K * Hkv * D),
                       ("v", v, B * K * Hkv * Dv), ("o", o, B * Q * Hq * Dv)):
        _check_tensor(name, t, q.dtype, n, dev)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, B * Q * Hq, dev)
    _check_tensor("mask_words", mask_words, torch.int32, B * Hm * Q * W, dev)
    for name, t in (("seqlens_q", seqlens_q), ("seqlens_k", seqlens_k)):
        if t is not None:
            _check_tensor(name, t, torch.int32, B, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib.attn_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Q, K, D,
                             Dv, _ptr(seqlens_q), _ptr(seqlens_k), _ptr(mask_words), W, Hm,
                             int(window), float(scale), MASKS[mask], _DTYPE_CODE[q.dtype],
                             ALGOS[algo], _stream_ptr(stream))
    _check(rc)
    return o, lse


def attn_fwd_paged(q, k_pages, v_pages, block_table, seqlens_k, o=None, lse=None, *,
                   seqlens_q=None, window=0, scale=None, algo="auto", mask="causal",
                   stream=None, want_lse=True):
    """Paged K/V: q [B,Q,Hq,D]; k_pages [P,page,Hkv,D], v_pages [P,page,Hkv,Dv];
    block_table int32 [B,max_pages] (key j of sequence b: row j % page of page
    block_table[b, j // page]); seqlens_k int32 [B].  All CUDA tensors.
    Returns (o [B,Q,Hq,Dv], lse [B,Q,Hq] or None)."""
    lib = load_library()
    B, Q, Hq, D = q.shape
    P, page, Hkv = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    Dv = v_pages.shape[3]
    max_pages = block_table.shape[1]
    dev = q.device
    if o is None:
        o = torch.empty((B, Q, Hq, Dv), dtype=q.dtype, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, Q, Hq), dtype=torch.float32, device=dev)
    for name, t, n in (("q", q, B * Q * Hq * D), ("k_pages", k_pages, P * page * Hkv * D),
                       ("v_pages", v_pages, P * page * Hkv * Dv), ("o", o, B * Q * Hq * Dv)):
        _check_tensor(name, t, q.dtype, n, dev)
    if lse is not None:
        _check_tensor("lse", lse, torch.float32, B * Q * Hq, dev)
    _check_tensor("block_table", block_table, torch.int32, B * max_pages, dev)
    _check_tensor("seqlens_k", seqlens_k, torch.int32, B, dev)
    if seqlens_q is not None:
        _check_tensor("seqlens_q", seqlens_q, torch.int32, B, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib.attn_fwd_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(o), _ptr(lse), B, Hq, Hkv,
                            Q, D, Dv, _ptr(block_table), max_pages, page, P, _ptr(seqlens_q),
                            _ptr(seqlens_k), int(window), float(scale), MASKS[mask],
                            _DTYPE_CODE[q.dtype], ALGOS[algo], _stream_ptr(stream))
    _check(rc)
    return o, lse
