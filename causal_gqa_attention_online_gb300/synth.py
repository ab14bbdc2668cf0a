"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and rounds them to the storage dtype; it holds
none of the attention arithmetic, so the CPU oracle and the CUDA path can both
be fed from it without sharing any of the method.

* Normals: N(0,1) float32 from numpy's PCG64, drawn in fixed chunks of 2**22
  values, chunk ``i`` of stream ``s`` seeded by ``SeedSequence([seed, s, i])``;
  the result does not depend on the thread count.  Streams: 0 = Q, 1 = K,
  2 = V, 3 = lengths.
* Storage dtypes: bf16 / fp16 are round-to-nearest-even from float32 (torch's
  conversion); the float32 upcast of the rounded value is exact, which is what
  the oracle receives.
* Lengths: int32 uniform on an inclusive range, e.g. [0, 8192] including 0.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}
TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}

_CHUNK = 1 << 22
STREAM_Q, STREAM_K, STREAM_V, STREAM_LEN, STREAM_DO = 0, 1, 2, 3, 4


def _fill_chunk(args):
    seed, stream, idx, out = args
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, idx])))
    g.standard_normal(out=out, dtype=np.float32)


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` N(0,1) float32 values of stream ``stream`` under ``seed``."""
    out = np.empty(int(n), np.float32)
    jobs = [(int(seed), int(stream), i, out[i * _CHUNK:(i + 1) * _CHUNK])
            for i in range((out.size + _CHUNK - 1) // _CHUNK)]
    if len(jobs) <= 1:
        for j in jobs:
            _fill_chunk(j)
    else:
        with ThreadPoolExecutor(min(len(jobs), os.cpu_count() or 1)) as ex:
            list(ex.map(_fill_chunk, jobs))
    return out


def lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` int32 lengths uniform on the inclusive range [lo, hi]."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), STREAM_LEN])))
    return g.integers(lo, hi, size=int(n), endpoint=True).astype(np.int32)


def to_storage(x: np.ndarray, dtype: str) -> torch.Tensor:
    """Round float32 values to the storage dtype (a CPU torch tensor)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(TORCH_DTYPES[dtype]).contiguous()


def exact_f32(t: torch.Tensor) -> np.ndarray:
    """The exact float32 values a storage tensor holds (CPU numpy)."""
    return t.detach().to("cpu").float().numpy()


@dataclass
class Inputs:
    """One seeded problem.  ``q/k/v`` are CPU torch tensors in the storage
    dtype; ``seqlens_*`` (padded) or ``cu_seqlens_*`` (packed) are int32 numpy
    arrays or None."""
    layout: str                      # "padded" or "packed"
    dtype: str
    B: int
    Hq: int
    Hkv: int
    Q: int                           # padded capacity, or max query length
    K: int                           # padded capacity, or max key length
    D: int
    Dv: int
    window: int
    scale: float
    q: torch.Tensor = field(repr=False)
    k: torch.Tensor = field(repr=False)
    v: torch.Tensor = field(repr=False)
    seqlens_q: np.ndarray | None = None
    seqlens_k: np.ndarray | None = None
    cu_seqlens_q: np.ndarray | None = None
    cu_seqlens_k: np.ndarray | None = None


def make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype="bf16", seed=1234, seqlens_q=None,
                seqlens_k=None, window=0, scale=None, pad_value=0.0) -> Inputs:
    """Padded layout q [B,Q,Hq,D], k [B,K,Hkv,D], v [B,K,Hkv,Dv].

    Rows past a sequence's length (query rows >= Qb, key rows >= Kb) hold
    ``pad_value`` (e.g. NaN, to show that they are never read) instead of
    random values; only the valid rows consume the random streams, in
    (b, row) order."""
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    sq = None if seqlens_q is None else np.asarray(seqlens_q, np.int32)
    sk = None if seqlens_k is None else np.asarray(seqlens_k, np.int32)
    qb = np.full(B, Q, np.int64) if sq is None else np.clip(sq, 0, Q).astype(np.int64)
    kb = np.full(B, K, np.int64) if sk is None else np.clip(sk, 0, K).astype(np.int64)

    def fill(stream, rows_per_b, cap, width):
        out = np.full((B, cap, width), pad_value, np.float32)
        vals = normal(seed, stream, int(rows_per_b.sum()) * width)
        off = 0
        for b in range(B):
            n = int(rows_per_b[b])
            out[b, :n] = vals[off:off + n * width].reshape(n, width)
            off += n * width
        return out

    q = fill(STREAM_Q, qb, Q, Hq * D).reshape(B, Q, Hq, D)
    k = fill(STREAM_K, kb, K, Hkv * D).reshape(B, K, Hkv, D)
    v = fill(STREAM_V, kb, K, Hkv * Dv).reshape(B, K, Hkv, Dv)
    return Inputs("padded", dtype, B, Hq, Hkv, Q, K, D, Dv, int(window), float(scale),
                  to_storage(q, dtype), to_storage(k, dtype), to_storage(v, dtype),
                  seqlens_q=sq, seqlens_k=sk)


def make_packed(seqlens_q, seqlens_k, Hq, Hkv, D, Dv, dtype="bf16", seed=1234, window=0,
                scale=None) -> Inputs:
    """Packed (varlen) layout q [Tq,Hq,D], k [Tk,Hkv,D], v [Tk,Hkv,Dv] with
    int32 cumulative lengths [B+1] starting at 0."""
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    sq = np.asarray(seqlens_q, np.int64)
    sk = np.asarray(seqlens_k, np.int64)
    B = int(sq.size)
    cq = np.concatenate([[0], np.cumsum(sq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(sk)]).astype(np.int32)
    Tq, Tk = int(cq[-1]), int(ck[-1])
    q = normal(seed, STREAM_Q, Tq * Hq * D).reshape(Tq, Hq, D)
    k = normal(seed, STREAM_K, Tk * Hkv * D).reshape(Tk, Hkv, D)
    v = normal(seed, STREAM_V, Tk * Hkv * Dv).reshape(Tk, Hkv, Dv)
    return Inputs("packed", dtype, B, Hq, Hkv, int(sq.max(initial=0)), int(sk.max(initial=0)),
                  D, Dv, int(window), float(scale), to_storage(q, dtype), to_storage(k, dtype),
                  to_storage(v, dtype), cu_seqlens_q=cq, cu_seqlens_k=ck)


def make_dout(inp: Inputs, seed: int = 1234, pad_value=0.0) -> torch.Tensor:
    """An output gradient dO shaped like the problem's O (padded [B,Q,Hq,Dv]
    or packed [Tq,Hq,Dv]), N(0,1) in the storage dtype; padded rows past a
    sequence's query length hold ``pad_value``."""
    if inp.layout == "packed":
        Tq = int(inp.cu_seqlens_q[-1])
        x = normal(seed, STREAM_DO, Tq * inp.Hq * inp.Dv).reshape(Tq, inp.Hq, inp.Dv)
        return to_storage(x, inp.dtype)
    qb = (np.full(inp.B, inp.Q) if inp.seqlens_q is None
          else np.clip(inp.seqlens_q, 0, inp.Q)).astype(np.int64)
    w = inp.Hq * inp.Dv
    out = np.full((inp.B, inp.Q, w), pad_value, np.float32)
    vals = normal(seed, STREAM_DO, int(qb.sum()) * w)
    off = 0
    for b in range(inp.B):
        n = int(qb[b])
        out[b, :n] = vals[off:off + n * w].reshape(n, w)
        off += n * w
    return to_storage(out.reshape(inp.B, inp.Q, inp.Hq, inp.Dv), inp.dtype)


# ---------------------------------------------------------------------------
# The named synthetic workloads.  Each builder returns an Inputs.

def prefill_f32_b1_h4x2_q64_k128_d64(seed=1234):
    """fp32 prefill, B=1 Hq=4 Hkv=2 Q=64 K=128 D=Dv=64, bottom-right causal."""
    return make_padded(1, 4, 2, 64, 128, 64, 64, "f32", seed)


def decode_f32_b1_h8x2_k2053_d80x96(seed=1234):
    """fp32 decode, B=1 Hq=8 Hkv=2 Q=1 K=2053 (ragged KV tail), D=80 Dv=96."""
    return make_padded(1, 8, 2, 1, 2053, 80, 96, "f32", seed)


def decode_bf16_b64_h32x8_k8192_d128(seed=1234, B=64, Kcap=8192, pad_value=0.0):
    """bf16 batched decode, B=64 Hq=32 Hkv=8 Q=1 D=Dv=128, per-sequence key
    lengths uniform on [0, 8192] (0 included), KV buffer padded to 8192."""
    sk = lengths(seed, B, 0, Kcap)
    return make_padded(B, 32, 8, 1, Kcap, 128, 128, "bf16", seed, seqlens_k=sk,
                       pad_value=pad_value)


def prefill_bf16_b4_h32x8_s4096_d128(seed=1234, B=4, S=4096):
    """bf16 causal prefill, B=4 Hq=32 Hkv=8 Q=K=4096 D=Dv=128."""
    return make_padded(B, 32, 8, S, S, 128, 128, "bf16", seed)


def varlen_bf16_16seq_h16x4_k4096_q512_w1024(seed=1234, nseq=16, Kmax=4096, Qmax=512,
                                               window=1024):
    """bf16 varlen chunked prefill: 16 packed sequences, key lengths uniform on
    [0, 4096] (empty included), each query chunk the last min(512, Kb) tokens,
    Hq=16 Hkv=4 D=Dv=128, sliding window 1024."""
    sk = lengths(seed, nseq, 0, Kmax)
    sq = np.minimum(sk, Qmax)
    return make_packed(sq, sk, 16, 4, 128, 128, "bf16", seed, window=window)
