"""Helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the CPU oracle on the same seeded inputs, compare element by element.

Tolerances (fixed by the method's stated bar):
* fp32 storage: max-abs 1e-4 on O and on LSE;
* bf16 / fp16 storage: max-abs 2e-2 on O, 1e-3 on LSE;
* rows with no legal key and padded rows: bit-exact O = +0.0, LSE = -inf.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from causal_gqa_attention_online_gb300 import attn_fwd, attn_fwd_varlen, synth

TOL = {"f32": (1e-4, 1e-4), "f16": (2e-2, 1e-3), "bf16": (2e-2, 1e-3)}
GUARD = 256  # elements of canary after every output buffer


def _guarded(shape, dtype, fill, device):
    n = int(np.prod(shape))
    buf = torch.full((n + GUARD,), fill, dtype=dtype, device=device)
    return buf, buf[:n].view(shape)


def _bits(t):
    """Bit pattern of a tensor (NaN canaries compare equal to themselves)."""
    return t.view(torch.int32 if t.element_size() == 4 else torch.int16)


MASK_NAMES = {0: "causal", 1: "causal_top_left", 2: "none"}


def run_gpu(inp: synth.Inputs, algo="auto", device="cuda", mask=0):
    """Run the library on ``inp``.  Outputs start as NaN canaries and are
    followed by guard regions; both are checked.  Returns numpy (o, lse)."""
    q = inp.q.to(device)
    k = inp.k.to(device)
    v = inp.v.to(device)
    q0, k0, v0 = q.clone(), k.clone(), v.clone()
    if inp.layout == "padded":
        oshape = (inp.B, inp.Q, inp.Hq, inp.Dv)
        lshape = (inp.B, inp.Q, inp.Hq)
    else:
        Tq = int(inp.cu_seqlens_q[-1])
        oshape = (Tq, inp.Hq, inp.Dv)
        lshape = (Tq, inp.Hq)
    obuf, o = _guarded(oshape, q.dtype, float("nan"), device)
    lbuf, lse = _guarded(lshape, torch.float32, float("nan"), device)
    if inp.layout == "padded":
        sq = None if inp.seqlens_q is None else torch.from_numpy(inp.seqlens_q).to(device)
        sk = None if inp.seqlens_k is None else torch.from_numpy(inp.seqlens_k).to(device)
        attn_fwd(q, k, v, o, lse, seqlens_q=sq, seqlens_k=sk, window=inp.window,
                 scale=inp.scale, algo=algo, mask=MASK_NAMES[mask])
    else:
        cq = torch.from_numpy(inp.cu_seqlens_q).to(device)
        ck = torch.from_numpy(inp.cu_seqlens_k).to(device)
        attn_fwd_varlen(q, k, v, cq, ck, inp.Q, inp.K, o, lse, window=inp.window,
                        scale=inp.scale, algo=algo, mask=MASK_NAMES[mask])
    torch.cuda.synchronize()
    assert torch.isnan(obuf[-GUARD:].float()).all(), "write past the end of o"
    assert torch.isnan(lbuf[-GUARD:]).all(), "write past the end of lse"
    for a, a0 in ((q, q0), (k, k0), (v, v0)):
        assert torch.equal(_bits(a), _bits(a0)), "inputs modified"
    return o.float().cpu().numpy(), lse.cpu().numpy()


def run_oracle(inp: synth.Inputs, nthreads=0, mask=0):
    q = synth.exact_f32(inp.q)
    k = synth.exact_f32(inp.k)
    v = synth.exact_f32(inp.v)
    if inp.layout == "padded":
        return oracle.attn_padded(q, k, v, B=inp.B, Hq=inp.Hq, Hkv=inp.Hkv, Q=inp.Q, K=inp.K,
                                  D=inp.D, Dv=inp.Dv, seqlens_q=inp.seqlens_q,
                                  seqlens_k=inp.seqlens_k, window=inp.window, scale=inp.scale,
                                  nthreads=nthreads, mask=mask)
    return oracle.attn_packed(q, k, v, B=inp.B, Hq=inp.Hq, Hkv=inp.Hkv, D=inp.D, Dv=inp.Dv,
                              cu_seqlens_q=inp.cu_seqlens_q, cu_seqlens_k=inp.cu_seqlens_k,
                              window=inp.window, scale=inp.scale, nthreads=nthreads,
                              mask=mask)


def compare(dtype, o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Element-by-element check; returns (max O error, max LSE error)."""
    tol_o, tol_l = TOL[dtype]
    o_gpu = np.asarray(o_gpu, np.float64).reshape(o_ref.shape)
    lse_gpu = np.asarray(lse_gpu, np.float64).reshape(lse_ref.shape)
    empty = lse_ref == -math.inf
    # rows with no legal key (and padded rows): exact +0.0 and -inf
    if empty.any():
        oe = o_gpu[empty]
        assert np.all(oe == 0.0) and not np.any(np.signbit(oe)), f"{what}: empty rows not +0"
        assert np.all(lse_gpu[empty] == -math.inf), f"{what}: empty rows LSE not -inf"
    full = ~empty
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite output"
    assert np.all(np.isfinite(lse_gpu[full])), f"{what}: non-finite LSE on a row with keys"
    eo = float(np.max(np.abs(o_gpu[full] - o_ref[full]))) if full.any() else 0.0
    el = float(np.max(np.abs(lse_gpu[full] - lse_ref[full]))) if full.any() else 0.0
    assert eo <= tol_o, f"{what}: max |dO| = {eo:.3g} > {tol_o}"
    assert el <= tol_l, f"{what}: max |dLSE| = {el:.3g} > {tol_l}"
    return eo, el


def check(inp: synth.Inputs, algo="auto", what="", mask=0):
    o, lse = run_gpu(inp, algo, mask=mask)
    ro, rl = run_oracle(inp, mask=mask)
    return compare(inp.dtype, o, lse, ro, rl, what or algo)


def sample_rows(inp: synth.Inputs, n: int, seed: int = 0):
    """(b, q, h) rows of a padded problem for sampled checks: random rows plus
    the first and last valid row of sampled sequences and some padded rows."""
    g = np.random.default_rng(seed)
    rows = []
    qb = np.full(inp.B, inp.Q) if inp.seqlens_q is None else np.clip(inp.seqlens_q, 0, inp.Q)
    for _ in range(n):
        b = int(g.integers(inp.B))
        rows.append((b, int(g.integers(inp.Q)), int(g.integers(inp.Hq))))
    for b in g.choice(inp.B, size=min(inp.B, 8), replace=False):
        h = int(g.integers(inp.Hq))
        if qb[b] > 0:
            rows.append((int(b), 0, h))
            rows.append((int(b), int(qb[b]) - 1, h))
        if qb[b] < inp.Q:
            rows.append((int(b), int(qb[b]), h))
    return np.array(rows, np.int32)


def check_sampled_padded(inp: synth.Inputs, o_gpu, lse_gpu, rows, what=""):
    """Compare sampled rows of a full-size padded run with the oracle, one
    sequence at a time (so only that sequence is widened to float32)."""
    errs = []
    for b in np.unique(rows[:, 0]):
        sel = rows[rows[:, 0] == b]
        local = sel.copy()
        local[:, 0] = 0
        q = synth.exact_f32(inp.q[b:b + 1])
        k = synth.exact_f32(inp.k[b:b + 1])
        v = synth.exact_f32(inp.v[b:b + 1])
        sq = None if inp.seqlens_q is None else inp.seqlens_q[b:b + 1]
        sk = None if inp.seqlens_k is None else inp.seqlens_k[b:b + 1]
        ro, rl = oracle.attn_padded_rows(q, k, v, local, B=1, Hq=inp.Hq, Hkv=inp.Hkv, Q=inp.Q,
                                         K=inp.K, D=inp.D, Dv=inp.Dv, seqlens_q=sq,
                                         seqlens_k=sk, window=inp.window, scale=inp.scale)
        og = o_gpu[sel[:, 0], sel[:, 1], sel[:, 2]]
        lg = lse_gpu[sel[:, 0], sel[:, 1], sel[:, 2]]
        errs.append(compare(inp.dtype, og, lg, ro, rl, f"{what} b={b}"))
    return max(e[0] for e in errs), max(e[1] for e in errs)
