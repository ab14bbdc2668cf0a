"""TEST INFRASTRUCTURE ONLY: the fp64 two-pass CPU oracle.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product package never imports it
and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it with the host C compiler and exposes numpy-facing
wrappers.  What it computes is the plain softmax-attention definition that the
online method reaches exactly in exact arithmetic:

* "Attention execution mapping: 现状、缺口与有界实验" (LuisaCompute), §1:
  bottom-right causal GQA, ``kh = h / (Hq/Hkv)``, legal keys ``k <= q + K - Q``.
* "快速後端" (Laya fast backends), "數值校驗": sliding window, per-sequence
  int32 lengths, empty sequences, finite padded output.

Inputs are float32 arrays holding the exact values the device consumes; the
oracle widens them to double and returns double outputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile an oracle C source (by default ``attn_oracle.c``) into a shared
    library (by default ``oracle/_build/liboracle.so``)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _i32(a):
    if a is None:
        return None, None
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _f64p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


class OracleLib:
    """The oracle entry points bound to one compiled library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        ci, cd, cl = ctypes.c_int, ctypes.c_double, ctypes.c_long
        lib.oracle_attn_padded.argtypes = [f32p, f32p, f32p, f64p, f64p] + [ci] * 7 + [
            i32p, i32p, ci, ci, cd, ci]
        lib.oracle_attn_padded.restype = ci
        lib.oracle_attn_packed.argtypes = [f32p, f32p, f32p, f64p, f64p] + [ci] * 5 + [
            i32p, i32p, ci, ci, cd, ci]
        lib.oracle_attn_packed.restype = ci
        lib.oracle_attn_padded_rows.argtypes = [f32p, f32p, f32p] + [ci] * 7 + [
            i32p, i32p, ci, ci, cd, i32p, i32p, i32p, cl, f64p, f64p, ci]
        lib.oracle_attn_padded_rows.restype = ci
        lib.oracle_attn_bwd_padded.argtypes = [f32p, f32p, f32p, f32p, f64p, f64p, f64p] + [
            ci] * 7 + [i32p, i32p, ci, ci, cd, ci]
        lib.oracle_attn_bwd_padded.restype = ci
        lib.oracle_attn_bwd_sampled.argtypes = [f32p, f32p, f32p, f32p] + [ci] * 7 + [
            i32p, i32p, ci, ci, cd, i32p, ctypes.c_long, f64p, ci, ci, ci, ci, f64p, f64p, ci]
        lib.oracle_attn_bwd_sampled.restype = ci
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_attn_padded_allow.argtypes = [f32p, f32p, f32p, f64p, f64p] + [ci] * 7 + [
            i32p, i32p, u8p, ci, ci, ci, cd, ci]
        lib.oracle_attn_padded_allow.restype = ci
        lib.oracle_legal_pairs.argtypes = [ci, ci, ci, ci]
        lib.oracle_legal_pairs.restype = ctypes.c_longlong
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ci
        self.lib = lib
        self.path = path

    def attn_padded(self, q, k, v, *, B, Hq, Hkv, Q, K, D, Dv, seqlens_q=None,
                    seqlens_k=None, window=0, scale=None, nthreads=0, mask=0):
        """Padded layout q [B,Q,Hq,D], k [B,K,Hkv,D], v [B,K,Hkv,Dv].
        ``mask``: 0 bottom-right causal (the pages' rule), 1 top-left causal,
        2 none.

        Returns (o [B,Q,Hq,Dv] float64, lse [B,Q,Hq] float64)."""
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        q, qp = _f32(q)
        k, kp = _f32(k)
        v, vp = _f32(v)
        if q.size != B * Q * Hq * D or k.size != B * K * Hkv * D or v.size != B * K * Hkv * Dv:
            raise ValueError("oracle_attn_padded: array sizes do not match the dims")
        sq, sqp = _i32(seqlens_q)
        sk, skp = _i32(seqlens_k)
        o = np.empty((B, Q, Hq, Dv), np.float64)
        lse = np.empty((B, Q, Hq), np.float64)
        rc = self.lib.oracle_attn_padded(qp, kp, vp, _f64p(o), _f64p(lse), B, Hq, Hkv, Q, K,
                                         D, Dv, sqp, skp, int(window), int(mask), float(scale),
                                         int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_padded failed with status {rc}")
        return o, lse

    def attn_packed(self, q, k, v, *, B, Hq, Hkv, D, Dv, cu_seqlens_q, cu_seqlens_k,
                    window=0, scale=None, nthreads=0, mask=0):
        """Packed layout q [Tq,Hq,D], k [Tk,Hkv,D], v [Tk,Hkv,Dv] with int32
        cumulative lengths [B+1].  Returns (o [Tq,Hq,Dv], lse [Tq,Hq]) float64."""
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        cq, cqp = _i32(cu_seqlens_q)
        ck, ckp = _i32(cu_seqlens_k)
        Tq, Tk = int(cq[B]), int(ck[B])
        q, qp = _f32(q)
        k, kp = _f32(k)
        v, vp = _f32(v)
        if q.size != Tq * Hq * D or k.size != Tk * Hkv * D or v.size != Tk * Hkv * Dv:
            raise ValueError("oracle_attn_packed: array sizes do not match the dims")
        o = np.empty((Tq, Hq, Dv), np.float64)
        lse = np.empty((Tq, Hq), np.float64)
        rc = self.lib.oracle_attn_packed(qp, kp, vp, _f64p(o), _f64p(lse), B, Hq, Hkv, D, Dv,
                                         cqp, ckp, int(window), int(mask), float(scale),
                                         int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_packed failed with status {rc}")
        return o, lse

    def attn_padded_allow(self, q, k, v, allow, *, B, Hq, Hkv, Q, K, D, Dv, seqlens_q=None,
                          seqlens_k=None, window=0, scale=None, nthreads=0, mask=0):
        """Padded layout with an arbitrary boolean mask ``allow`` [B, Hm, Q, K]
        (Hm = 1: one mask for every head; Hm = Hq: one per query head), ANDed
        with the ``mask`` mode and the window.  Returns (o, lse) float64."""
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        q, qp = _f32(q)
        k, kp = _f32(k)
        v, vp = _f32(v)
        allow = np.ascontiguousarray(allow, dtype=bool).astype(np.uint8)
        if allow.ndim != 4 or allow.shape[0] != B or allow.shape[2:] != (Q, K):
            raise ValueError("oracle_attn_padded_allow: allow must be [B, Hm, Q, K]")
        Hm = allow.shape[1]
        if q.size != B * Q * Hq * D or k.size != B * K * Hkv * D or v.size != B * K * Hkv * Dv:
            raise ValueError("oracle_attn_padded_allow: array sizes do not match the dims")
        sq, sqp = _i32(seqlens_q)
        sk, skp = _i32(seqlens_k)
        o = np.empty((B, Q, Hq, Dv), np.float64)
        lse = np.empty((B, Q, Hq), np.float64)
        ap = allow.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))
        rc = self.lib.oracle_attn_padded_allow(qp, kp, vp, _f64p(o), _f64p(lse), B, Hq, Hkv, Q,
                                               K, D, Dv, sqp, skp, ap, int(Hm), int(window),
                                               int(mask), float(scale), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_padded_allow failed with status {rc}")
        return o, lse

    def attn_padded_rows(self, q, k, v, rows, *, B, Hq, Hkv, Q, K, D, Dv, seqlens_q=None,
                         seqlens_k=None, window=0, scale=None, nthreads=0, mask=0):
        """Selected rows of the padded layout.  ``rows`` is an int array [n,3]
        of (b, q, h).  Returns (o [n,Dv], lse [n]) float64."""
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
        rb, rbp = _i32(rows[:, 0])
        rq, rqp = _i32(rows[:, 1])
        rh, rhp = _i32(rows[:, 2])
        q, qp = _f32(q)
        k, kp = _f32(k)
        v, vp = _f32(v)
        if q.size != B * Q * Hq * D or k.size != B * K * Hkv * D or v.size != B * K * Hkv * Dv:
            raise ValueError("oracle_attn_padded_rows: array sizes do not match the dims")
        sq, sqp = _i32(seqlens_q)
        sk, skp = _i32(seqlens_k)
        n = rows.shape[0]
        o = np.empty((n, Dv), np.float64)
        lse = np.empty((n,), np.float64)
        rc = self.lib.oracle_attn_padded_rows(qp, kp, vp, B, Hq, Hkv, Q, K, D, Dv, sqp, skp,
                                              int(window), int(mask), float(scale), rbp, rqp,
                                              rhp, n,
                                              _f64p(o), _f64p(lse), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_padded_rows failed with status {rc}")
        return o, lse

    def attn_bwd_padded(self, q, k, v, dout, *, B, Hq, Hkv, Q, K, D, Dv, seqlens_q=None,
                        seqlens_k=None, window=0, scale=None, mask=0, nthreads=0):
        """Gradients (dq [B,Q,Hq,D], dk [B,K,Hkv,D], dv [B,K,Hkv,Dv], float64)
        of the padded-layout attention for the output gradient ``dout``
        [B,Q,Hq,Dv]; the forward is recomputed from its definition."""
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        q, qp = _f32(q)
        k, kp = _f32(k)
        v, vp = _f32(v)
        g, gp = _f32(dout)
        if (q.size != B * Q * Hq * D or k.size != B * K * Hkv * D or
                v.size != B * K * Hkv * Dv or g.size != B * Q * Hq * Dv):
            raise ValueError("oracle_attn_bwd_padded: array sizes do not match the dims")
        sq, sqp = _i32(seqlens_q)
        sk, skp = _i32(seqlens_k)
        dq = np.empty((B, Q, Hq, D), np.float64)
        dk = np.empty((B, K, Hkv, D), np.float64)
        dv = np.empty((B, K, Hkv, Dv), np.float64)
        rc = self.lib.oracle_attn_bwd_padded(qp, kp, vp, gp, _f64p(dq), _f64p(dk), _f64p(dv), B,
                                             Hq, Hkv, Q, K, D, Dv, sqp, skp, int(window),
                                             int(mask), float(scale), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd_padded failed with status {rc}")
        return dq, dk, dv

    def attn_bwd_sampled(self, q, k, v, dout, *, B, Hq, Hkv, Q, K, D, Dv, rows=None,
                         key_block=None, seqlens_q=None, seqlens_k=None, window=0, scale=None,
                         mask=0, nthreads=0):
        """Parts of the padded-layout gradients: dq of ``rows`` (int [n,3] of
        (b, q, h)) and dk, dv of ``key_block`` = (b, kh, k0, k1).  Returns
        (dq [n,D], dk [k1-k0,D], dv [k1-k0,Dv]) float64."""
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        q, qp = _f32(q)
        k, kp = _f32(k)
        v, vp = _f32(v)
        g, gp = _f32(dout)
        if (q.size != B * Q * Hq * D or k.size != B * K * Hkv * D or
                v.size != B * K * Hkv * Dv or g.size != B * Q * Hq * Dv):
            raise ValueError("oracle_attn_bwd_sampled: array sizes do not match the dims")
        sq, sqp = _i32(seqlens_q)
        sk, skp = _i32(seqlens_k)
        rows = np.zeros((0, 3), np.int32) if rows is None else np.ascontiguousarray(rows, np.int32)
        rp = rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
        kb, kh, k0, k1 = key_block if key_block is not None else (0, 0, 0, 0)
        dq = np.zeros((rows.shape[0], D), np.float64)
        dk = np.zeros((max(k1 - k0, 0), D), np.float64)
        dv = np.zeros((max(k1 - k0, 0), Dv), np.float64)
        rc = self.lib.oracle_attn_bwd_sampled(qp, kp, vp, gp, B, Hq, Hkv, Q, K, D, Dv, sqp, skp,
                                              int(window), int(mask), float(scale), rp,
                                              rows.shape[0], _f64p(dq), kb, kh, k0, k1,
                                              _f64p(dk), _f64p(dv), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_attn_bwd_sampled failed with status {rc}")
        return dq, dk, dv

    def legal_pairs(self, Qb: int, Kb: int, window: int = 0, mask: int = 0) -> int:
        """Legal (query, key) pairs of one sequence and head, by enumeration."""
        return int(self.lib.oracle_legal_pairs(int(Qb), int(Kb), int(window), int(mask)))

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())


def _default() -> OracleLib:
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
        return _lib


def attn_padded(*args, **kw):
    return _default().attn_padded(*args, **kw)


def attn_packed(*args, **kw):
    return _default().attn_packed(*args, **kw)


def attn_padded_rows(*args, **kw):
    return _default().attn_padded_rows(*args, **kw)


def attn_padded_allow(*args, **kw):
    return _default().attn_padded_allow(*args, **kw)


def attn_bwd_padded(*args, **kw):
    return _default().attn_bwd_padded(*args, **kw)


def attn_bwd_sampled(*args, **kw):
    return _default().attn_bwd_sampled(*args, **kw)


def legal_pairs(Qb: int, Kb: int, window: int = 0, mask: int = 0) -> int:
    return _default().legal_pairs(Qb, Kb, window, mask)


def max_threads() -> int:
    return _default().max_threads()


SOURCE = _SRC
