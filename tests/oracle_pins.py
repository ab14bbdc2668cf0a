"""Checks that pin the CPU oracle to facts outside itself.

Each ``pin_*`` function takes an ``oracle.OracleLib`` and raises
AssertionError when the oracle disagrees with:

* hand-derived closed forms (``tests/golden/*.json``, each citing its passage);
* ``torch.nn.functional.scaled_dot_product_attention`` in fp64 with a boolean
  mask built by ``numpy.tril`` / ``numpy.triu`` (a library routine and a mask
  construction independent of the oracle's explicit key enumeration);
* invariants the definition fixes (constant V, a single legal key, identical
  keys, probabilities summing to one, empty rows, window >= K, scale 0,
  MHA/MQA equivalence, thread-count invariance).

``tests/test_oracle.py`` runs them against the real oracle and
``tests/test_oracle_mutants.py`` checks that every planted mistake in a copy
of the oracle fails at least one of them.
"""
from __future__ import annotations

import glob
import json
import math
import os
from fractions import Fraction

import numpy as np
import torch

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# helpers

def parse_value(s) -> float:
    """A fixture scalar: a number, "a/b", "log(n)" or "-inf"."""
    if isinstance(s, (int, float)):
        return float(s)
    s = s.strip()
    if s == "-inf":
        return -math.inf
    if s.startswith("log(") and s.endswith(")"):
        return math.log(float(Fraction(s[4:-1])))
    return float(Fraction(s))


def parse_array(a) -> np.ndarray:
    return np.vectorize(parse_value, otypes=[np.float64])(np.array(a, dtype=object))


def golden_files():
    return sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.json")))


def mask_matrix(Qb: int, Kb: int, window: int, mask: int = 0) -> np.ndarray:
    """Legal-key mask built from numpy's triangle routines: np.tril keeps
    j - i <= Kb - Qb (bottom-right causal; j - i <= 0 for the top-left mask),
    np.triu keeps the window; mask 2 keeps every key."""
    if mask == 2:
        return np.ones((Qb, Kb), dtype=bool)
    off = Kb - Qb if mask == 0 else 0
    m = np.tril(np.ones((Qb, Kb), dtype=bool), k=off)
    if window > 0:
        m &= np.triu(np.ones((Qb, Kb), dtype=bool), k=off - window + 1)
    return m


def sdpa_reference(q, k, v, Qb, Kb, Hq, Hkv, window, scale, mask=0):
    """fp64 torch SDPA with an explicit boolean mask for one sequence.

    q [Qb,Hq,D], k [Kb,Hkv,D], v [Kb,Hkv,Dv] float arrays.  Returns
    (o [Qb,Hq,Dv], lse [Qb,Hq], has_key [Qb]) with o/lse only meaningful where
    the row has a legal key.  KV heads are expanded with repeat_interleave,
    which maps query head h to KV head h // (Hq/Hkv)."""
    G = Hq // Hkv
    qt = torch.from_numpy(np.asarray(q, np.float64)).permute(1, 0, 2)       # [Hq,Qb,D]
    kt = torch.from_numpy(np.asarray(k, np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
    vt = torch.from_numpy(np.asarray(v, np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
    m = mask_matrix(Qb, Kb, window, mask)
    has = m.any(axis=1)
    mt = torch.from_numpy(m)
    safe = mt.clone()
    safe[~torch.from_numpy(has)] = True      # keep SDPA finite on rows we ignore
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.unsqueeze(0), kt.unsqueeze(0), vt.unsqueeze(0), attn_mask=safe, scale=scale)[0]
    s = torch.matmul(qt, kt.transpose(1, 2)) * scale
    s = s.masked_fill(~mt, -math.inf)
    lse = torch.logsumexp(s, dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy(), has


def rng_inputs(seed, B, Hq, Hkv, Q, K, D, Dv):
    g = np.random.default_rng(seed)
    q = g.standard_normal((B, Q, Hq, D)).astype(np.float32)
    k = g.standard_normal((B, K, Hkv, D)).astype(np.float32)
    v = g.standard_normal((B, K, Hkv, Dv)).astype(np.float32)
    return q, k, v


# ---------------------------------------------------------------------------
# pins

def pin_golden(ol):
    files = golden_files()
    assert files, "no golden fixtures found"
    for path in files:
        with open(path) as f:
            g = json.load(f)
        q = parse_array(g["q"]).astype(np.float32)
        k = parse_array(g["k"]).astype(np.float32)
        v = parse_array(g["v"]).astype(np.float32)
        scale = parse_value(g["scale"])
        exp_o = parse_array(g["expected_o"])
        exp_l = parse_array(g["expected_lse"])
        if g["layout"] == "padded":
            o, lse = ol.attn_padded(q, k, v, B=g["B"], Hq=g["Hq"], Hkv=g["Hkv"], Q=g["Q"],
                                    K=g["K"], D=g["D"], Dv=g["Dv"],
                                    seqlens_q=g.get("seqlens_q"), seqlens_k=g.get("seqlens_k"),
                                    window=g["window"], scale=scale)
        else:
            o, lse = ol.attn_packed(q, k, v, B=g["B"], Hq=g["Hq"], Hkv=g["Hkv"], D=g["D"],
                                    Dv=g["Dv"], cu_seqlens_q=g["cu_seqlens_q"],
                                    cu_seqlens_k=g["cu_seqlens_k"], window=g["window"],
                                    scale=scale)
        lse = lse.reshape(exp_l.shape)
        o = o.reshape(exp_o.shape)
        assert np.allclose(o, exp_o, atol=g["atol"], rtol=0), (g["name"], o, exp_o)
        fin = np.isfinite(exp_l)
        assert np.array_equal(np.isfinite(lse), fin), (g["name"], lse, exp_l)
        assert np.all(lse[~fin] == -math.inf), (g["name"], lse)
        assert np.allclose(lse[fin], exp_l[fin], atol=g["atol"], rtol=0), (g["name"], lse, exp_l)
        # rows with no legal key hold +0.0 exactly (sign bit clear)
        zero_rows = ~fin
        if zero_rows.any():
            oz = o[zero_rows]
            assert np.all(oz == 0.0) and not np.any(np.signbit(oz)), (g["name"], oz)


SDPA_CASES = [
    # B, Hq, Hkv, Q, K, D, Dv, window, seqlens_q, seqlens_k
    (1, 4, 2, 16, 37, 8, 8, 0, None, None),
    (2, 6, 3, 9, 9, 5, 7, 0, None, None),
    (1, 8, 2, 1, 53, 16, 12, 0, None, None),        # decode
    (2, 4, 1, 13, 40, 8, 8, 5, None, None),         # MQA + window
    (1, 3, 3, 20, 20, 4, 4, 3, None, None),         # MHA + window
    (3, 4, 2, 12, 16, 8, 6, 0, [12, 5, 0], [16, 3, 9]),
    (2, 2, 1, 10, 4, 4, 4, 0, None, None),          # Q > K: leading rows empty
    (2, 4, 2, 7, 30, 6, 6, 4, [7, 3], [30, 0]),
]


def pin_sdpa(ol):
    for ci, (B, Hq, Hkv, Q, K, D, Dv, w, sq, sk) in enumerate(SDPA_CASES):
        q, k, v = rng_inputs(100 + ci, B, Hq, Hkv, Q, K, D, Dv)
        scale = 1.0 / math.sqrt(D) * (1.0 + 0.25 * ci)
        o, lse = ol.attn_padded(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv,
                                seqlens_q=sq, seqlens_k=sk, window=w, scale=scale)
        for b in range(B):
            Qb = Q if sq is None else sq[b]
            Kb = K if sk is None else sk[b]
            # padded rows
            assert np.all(o[b, Qb:] == 0.0) and np.all(lse[b, Qb:] == -math.inf), (ci, b)
            if Qb == 0:
                continue
            if Kb == 0:
                assert np.all(o[b, :Qb] == 0.0) and np.all(lse[b, :Qb] == -math.inf), (ci, b)
                continue
            ro, rl, has = sdpa_reference(q[b, :Qb], k[b, :Kb], v[b, :Kb], Qb, Kb, Hq, Hkv, w,
                                         scale)
            assert np.allclose(o[b, :Qb][has], ro[has], atol=1e-12, rtol=1e-10), (ci, b)
            assert np.allclose(lse[b, :Qb][has], rl[has], atol=1e-12, rtol=1e-12), (ci, b)
            assert np.all(o[b, :Qb][~has] == 0.0), (ci, b)
            assert np.all(lse[b, :Qb][~has] == -math.inf), (ci, b)


def pin_invariants(ol):
    B, Hq, Hkv, Q, K, D, Dv = 2, 4, 2, 11, 19, 8, 5
    q, k, v = rng_inputs(7, B, Hq, Hkv, Q, K, D, Dv)
    kw = dict(B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv)
    G = Hq // Hkv

    # constant V -> that constant on every row
    vc = np.full_like(v, 0.375)
    o, lse = ol.attn_padded(q, k, vc, **kw)
    assert np.allclose(o, 0.375, atol=1e-14), "constant V"

    # window 1 -> the diagonal key's V row, LSE = its score
    o, lse = ol.attn_padded(q, k, v, window=1, **kw)
    scale = 1.0 / math.sqrt(D)
    for b in range(B):
        for i in range(Q):
            kd = i + K - Q
            for h in range(Hq):
                assert np.allclose(o[b, i, h], v[b, kd, h // G], atol=1e-14), "single key"
                s = scale * float(np.dot(q[b, i, h].astype(np.float64), k[b, kd, h // G]))
                assert abs(lse[b, i, h] - s) < 1e-12, "single key lse"

    # identical keys -> mean of the legal V rows
    ks = np.broadcast_to(k[:, :1], k.shape).copy()
    for w in (0, 4):
        o, lse = ol.attn_padded(q, ks, v, window=w, **kw)
        m = mask_matrix(Q, K, w)
        for b in range(B):
            for i in range(Q):
                for h in range(Hq):
                    mean = v[b][m[i], h // G].astype(np.float64).mean(axis=0)
                    assert np.allclose(o[b, i, h], mean, atol=1e-12), "identical keys"

    # probabilities sum to one: sum_{legal k} exp(s_k - LSE) == 1
    for w in (0, 6):
        o, lse = ol.attn_padded(q, k, v, window=w, **kw)
        m = mask_matrix(Q, K, w)
        for b in range(B):
            for h in range(Hq):
                s = scale * (q[b, :, h].astype(np.float64) @ k[b, :, h // G].astype(np.float64).T)
                tot = np.where(m, np.exp(s - lse[b, :, h][:, None]), 0.0).sum(axis=1)
                assert np.allclose(tot, 1.0, atol=1e-12), "sum p = 1"

    # scale 0 -> uniform weights -> mean of legal V rows, LSE = ln(#legal)
    o, lse = ol.attn_padded(q, k, v, scale=0.0, window=3, **kw)
    m = mask_matrix(Q, K, 3)
    for b in range(B):
        for i in range(Q):
            for h in range(Hq):
                mean = v[b][m[i], h // G].astype(np.float64).mean(axis=0)
                assert np.allclose(o[b, i, h], mean, atol=1e-12), "scale 0"
                assert abs(lse[b, i, h] - math.log(m[i].sum())) < 1e-12, "scale 0 lse"

    # window >= K is the same as no window
    o0, l0 = ol.attn_padded(q, k, v, window=0, **kw)
    o1, l1 = ol.attn_padded(q, k, v, window=K, **kw)
    o2, l2 = ol.attn_padded(q, k, v, window=K + 100, **kw)
    assert np.array_equal(o0, o1) and np.array_equal(o0, o2), "window >= K"
    assert np.array_equal(l0, l1) and np.array_equal(l0, l2), "window >= K lse"

    # GQA == MHA with every KV head repeated G times (numpy.repeat)
    kr = np.repeat(k, G, axis=2)
    vr = np.repeat(v, G, axis=2)
    om, lm = ol.attn_padded(q, kr, vr, B=B, Hq=Hq, Hkv=Hq, Q=Q, K=K, D=D, Dv=Dv)
    assert np.array_equal(o0, om) and np.array_equal(l0, lm), "GQA == MHA"
    # MQA: a single KV head
    o_mqa, _ = ol.attn_padded(q, k[:, :, :1].copy(), v[:, :, :1].copy(), B=B, Hq=Hq, Hkv=1,
                              Q=Q, K=K, D=D, Dv=Dv)
    om2, _ = ol.attn_padded(q, np.repeat(k[:, :, :1], Hq, axis=2), np.repeat(v[:, :, :1], Hq, axis=2),
                            B=B, Hq=Hq, Hkv=Hq, Q=Q, K=K, D=D, Dv=Dv)
    assert np.array_equal(o_mqa, om2), "MQA == MHA"

    # empty KV (Kb = 0) and Q > K leading rows: +0 and -inf exactly
    o, lse = ol.attn_padded(q, k, v, seqlens_k=[0, 3], **kw)
    assert np.all(o[0] == 0.0) and not np.any(np.signbit(o[0])) and np.all(lse[0] == -math.inf)
    # sequence 1 has Qb = 11 > Kb = 3: rows 0..7 have no legal key
    assert np.all(o[1, :8] == 0.0) and np.all(lse[1, :8] == -math.inf), "Q > K rows"
    assert np.all(np.isfinite(lse[1, 8:])), "Q > K rows with keys"

    # thread count does not change a single bit
    oa, la = ol.attn_padded(q, k, v, window=5, nthreads=1, **kw)
    ob, lb = ol.attn_padded(q, k, v, window=5, nthreads=4, **kw)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb), "thread invariance"


def pin_packed_matches_padded(ol):
    Hq, Hkv, D, Dv = 4, 2, 8, 6
    sq = np.array([5, 0, 3, 9, 1], np.int32)
    sk = np.array([5, 4, 0, 12, 7], np.int32)
    cq = np.concatenate([[0], np.cumsum(sq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(sk)]).astype(np.int32)
    g = np.random.default_rng(11)
    q = g.standard_normal((cq[-1], Hq, D)).astype(np.float32)
    k = g.standard_normal((ck[-1], Hkv, D)).astype(np.float32)
    v = g.standard_normal((ck[-1], Hkv, Dv)).astype(np.float32)
    for w in (0, 3):
        o, lse = ol.attn_packed(q, k, v, B=sq.size, Hq=Hq, Hkv=Hkv, D=D, Dv=Dv,
                                cu_seqlens_q=cq, cu_seqlens_k=ck, window=w)
        for b in range(sq.size):
            Qb, Kb = int(sq[b]), int(sk[b])
            if Qb == 0:
                continue
            if Kb == 0:
                assert np.all(o[cq[b]:cq[b + 1]] == 0.0)
                assert np.all(lse[cq[b]:cq[b + 1]] == -math.inf)
                continue
            ro, rl, has = sdpa_reference(q[cq[b]:cq[b + 1]], k[ck[b]:ck[b + 1]],
                                         v[ck[b]:ck[b + 1]], Qb, Kb, Hq, Hkv, w,
                                         1.0 / math.sqrt(D))
            ob, lb = o[cq[b]:cq[b + 1]], lse[cq[b]:cq[b + 1]]
            assert np.allclose(ob[has], ro[has], atol=1e-12), ("packed", b)
            assert np.allclose(lb[has], rl[has], atol=1e-12), ("packed lse", b)
            assert np.all(ob[~has] == 0.0) and np.all(lb[~has] == -math.inf)


def pin_rows_match_full(ol):
    B, Hq, Hkv, Q, K, D, Dv = 2, 4, 2, 9, 14, 8, 8
    q, k, v = rng_inputs(5, B, Hq, Hkv, Q, K, D, Dv)
    kw = dict(B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv, seqlens_q=[9, 4], seqlens_k=[14, 2],
              window=5)
    o, lse = ol.attn_padded(q, k, v, **kw)
    rows = np.array([[0, 0, 0], [0, 8, 3], [1, 3, 1], [1, 6, 2], [0, 4, 2]], np.int32)
    ro, rl = ol.attn_padded_rows(q, k, v, rows, **kw)
    for i, (b, qi, h) in enumerate(rows):
        assert np.array_equal(ro[i], o[b, qi, h]) and rl[i] == lse[b, qi, h], ("rows", i)


def pin_legal_pairs(ol):
    for (Qb, Kb, w) in [(4096, 4096, 0), (1, 8192, 0), (512, 4000, 1024), (3, 1, 0),
                        (0, 5, 0), (7, 0, 0), (10, 20, 3), (64, 128, 0)]:
        for mask in (0, 1, 2):
            ww = 0 if mask == 2 else w
            n = int(mask_matrix(Qb, Kb, ww, mask).sum())
            got = ol.legal_pairs(Qb, Kb, ww, mask)
            assert got == n, ("pairs", Qb, Kb, ww, mask, got, n)
    assert ol.legal_pairs(4096, 4096, 0) == 4096 * 4097 // 2
    # closed forms of the two extension masks
    assert ol.legal_pairs(300, 700, 0, 2) == 300 * 700
    assert ol.legal_pairs(700, 300, 0, 1) == 300 * 301 // 2 + 400 * 300


# (B, Hq, Hkv, Q, K, D, Dv, window, seqlens_q, seqlens_k, mask) for the two
# masks beyond the pages' bottom-right rule
MASK_CASES = [
    (1, 4, 2, 16, 37, 8, 8, 0, None, None, 1),        # top-left, Q < K
    (2, 4, 1, 30, 12, 8, 6, 0, None, None, 1),        # top-left, Q > K
    (1, 6, 3, 20, 25, 5, 7, 4, None, None, 1),        # top-left + window
    (3, 4, 2, 12, 16, 8, 6, 0, [12, 5, 0], [16, 3, 9], 1),
    (1, 4, 2, 16, 37, 8, 8, 0, None, None, 2),        # no mask
    (2, 8, 2, 1, 53, 16, 12, 0, None, None, 2),       # no mask, decode
    (3, 4, 2, 12, 16, 8, 6, 0, [12, 5, 3], [16, 0, 9], 2),
]


def pin_sdpa_masks(ol):
    for ci, (B, Hq, Hkv, Q, K, D, Dv, w, sq, sk, mask) in enumerate(MASK_CASES):
        q, k, v = rng_inputs(300 + ci, B, Hq, Hkv, Q, K, D, Dv)
        scale = 1.0 / math.sqrt(D) * (1.0 + 0.25 * ci)
        o, lse = ol.attn_padded(q, k, v, B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv,
                                seqlens_q=sq, seqlens_k=sk, window=w, scale=scale, mask=mask)
        for b in range(B):
            Qb = Q if sq is None else sq[b]
            Kb = K if sk is None else sk[b]
            assert np.all(o[b, Qb:] == 0.0) and np.all(lse[b, Qb:] == -math.inf), (ci, b)
            if Qb == 0:
                continue
            if Kb == 0:
                assert np.all(o[b, :Qb] == 0.0) and np.all(lse[b, :Qb] == -math.inf), (ci, b)
                continue
            ro, rl, has = sdpa_reference(q[b, :Qb], k[b, :Kb], v[b, :Kb], Qb, Kb, Hq, Hkv, w,
                                         scale, mask)
            assert np.allclose(o[b, :Qb][has], ro[has], atol=1e-12, rtol=1e-10), (ci, b)
            assert np.allclose(lse[b, :Qb][has], rl[has], atol=1e-12, rtol=1e-12), (ci, b)
            assert np.all(o[b, :Qb][~has] == 0.0), (ci, b)
            assert np.all(lse[b, :Qb][~has] == -math.inf), (ci, b)
    # relations between the masks: with Q = K the two causal masks agree; a
    # causal row that sees every key is the unmasked row
    B, Hq, Hkv, Q, K, D, Dv = 2, 4, 2, 9, 9, 8, 8
    q, k, v = rng_inputs(400, B, Hq, Hkv, Q, K, D, Dv)
    kw = dict(B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv)
    o0, l0 = ol.attn_padded(q, k, v, mask=0, **kw)
    o1, l1 = ol.attn_padded(q, k, v, mask=1, **kw)
    o2, l2 = ol.attn_padded(q, k, v, mask=2, **kw)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1), "Q = K: causal masks differ"
    assert np.array_equal(o0[:, -1], o2[:, -1]) and np.array_equal(l0[:, -1], l2[:, -1]), \
        "last causal row != unmasked row"
    assert not np.allclose(o0[:, 0], o2[:, 0]), "unmasked first row sees only key 0"
    # a window is rejected without a causal mask
    try:
        ol.attn_padded(q, k, v, mask=2, window=3, **kw)
    except ValueError:
        pass
    else:
        raise AssertionError("window accepted with no mask")


# ---------------------------------------------------------------------------
# backward pins: the gradients of the forward definition

BWD_CASES = [
    # B, Hq, Hkv, Q, K, D, Dv, window, seqlens_q, seqlens_k, mask
    (2, 4, 2, 7, 11, 8, 8, 0, None, None, 0),
    (3, 6, 2, 9, 9, 8, 12, 3, [9, 4, 0], [9, 7, 5], 0),
    (2, 4, 1, 6, 10, 16, 8, 0, [6, 5], [10, 0], 1),
    (2, 2, 2, 5, 8, 4, 4, 0, [5, 3], [8, 6], 2),
    (1, 8, 2, 12, 5, 8, 8, 2, None, None, 0),
]


def autograd_reference(q, k, v, dout, Qb, Kb, Hq, Hkv, window, scale, mask=0):
    """torch fp64 autograd of sum(O * dO) for one sequence, O the masked
    softmax attention built from torch ops (softmax, matmul) and the numpy
    mask.  Rows without a legal key are left out of the loss.  KV heads are
    expanded with repeat_interleave, so autograd sums each KV head's
    gradient over its query heads."""
    G = Hq // Hkv
    qt = torch.tensor(np.asarray(q, np.float64), requires_grad=True)
    kt = torch.tensor(np.asarray(k, np.float64), requires_grad=True)
    vt = torch.tensor(np.asarray(v, np.float64), requires_grad=True)
    m = torch.from_numpy(mask_matrix(Qb, Kb, window, mask))
    has = m.any(dim=1)
    safe = m.clone()
    safe[~has] = True
    qh = qt.permute(1, 0, 2)
    kh = kt.permute(1, 0, 2).repeat_interleave(G, 0)
    vh = vt.permute(1, 0, 2).repeat_interleave(G, 0)
    s = torch.matmul(qh, kh.transpose(1, 2)) * scale
    p = torch.softmax(s.masked_fill(~safe, -math.inf), dim=-1)
    o = torch.matmul(p, vh).permute(1, 0, 2)                          # [Qb,Hq,Dv]
    g = torch.from_numpy(np.asarray(dout, np.float64)) * has[:, None, None]
    (o * g).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def _bwd_inputs(seed, B, Hq, Hkv, Q, K, D, Dv):
    q, k, v = rng_inputs(seed, B, Hq, Hkv, Q, K, D, Dv)
    g = np.random.default_rng(seed + 1)
    dout = g.standard_normal((B, Q, Hq, Dv)).astype(np.float32)
    return q, k, v, dout


def pin_bwd_autograd(ol):
    for ci, (B, Hq, Hkv, Q, K, D, Dv, w, sq, sk, mask) in enumerate(BWD_CASES):
        q, k, v, dout = _bwd_inputs(500 + ci, B, Hq, Hkv, Q, K, D, Dv)
        scale = 1.0 / math.sqrt(D) * (1.0 + 0.3 * ci)
        dq, dk, dv = ol.attn_bwd_padded(q, k, v, dout, B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D,
                                        Dv=Dv, seqlens_q=sq, seqlens_k=sk, window=w,
                                        scale=scale, mask=mask)
        for b in range(B):
            Qb = Q if sq is None else sq[b]
            Kb = K if sk is None else sk[b]
            # padded rows and keys get no gradient
            assert np.all(dq[b, Qb:] == 0.0) and np.all(dk[b, Kb:] == 0.0), (ci, b)
            assert np.all(dv[b, Kb:] == 0.0), (ci, b)
            if Qb == 0 or Kb == 0:
                assert np.all(dq[b] == 0.0) and np.all(dk[b] == 0.0) and np.all(dv[b] == 0.0)
                continue
            rq, rk, rv = autograd_reference(q[b, :Qb], k[b, :Kb], v[b, :Kb], dout[b, :Qb], Qb, Kb,
                                            Hq, Hkv, w, scale, mask)
            for name, got, ref in (("dq", dq[b, :Qb], rq), ("dk", dk[b, :Kb], rk),
                                   ("dv", dv[b, :Kb], rv)):
                assert np.allclose(got, ref, atol=1e-12, rtol=1e-10), (ci, b, name)


def pin_bwd_finite_differences(ol):
    """Central differences of the (separately pinned) forward oracle: the
    directional derivative of L = sum(O * dO) along a random direction of q,
    k or v equals <grad, direction>.  The step is a power of two so that the
    perturbed float32 inputs are exact."""
    B, Hq, Hkv, Q, K, D, Dv = 2, 4, 2, 6, 9, 8, 6
    sq, sk = [6, 4], [9, 6]
    for ci, (w, mask) in enumerate(((0, 0), (3, 0), (0, 1), (0, 2))):
        q, k, v, dout = _bwd_inputs(600 + ci, B, Hq, Hkv, Q, K, D, Dv)
        # inputs on a 2^-16 grid: the perturbed values stay exact in float32
        q, k, v = (np.round(t * 65536.0).astype(np.float32) / np.float32(65536.0) for t in (q, k, v))
        kw = dict(B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv, seqlens_q=sq, seqlens_k=sk,
                  window=w, scale=0.4, mask=mask)
        grads = ol.attn_bwd_padded(q, k, v, dout, **kw)

        def loss(q_, k_, v_):
            o, _ = ol.attn_padded(q_, k_, v_, **kw)
            return float((o * dout.astype(np.float64)).sum())

        g = np.random.default_rng(700 + ci)
        h = 2.0 ** -13
        for which, grad in zip(range(3), grads):
            args = [q, k, v]
            # direction of small integers, masked to the sequence's valid rows
            dirn = g.integers(-2, 3, size=args[which].shape).astype(np.float32)
            for b in range(B):
                dirn[b, (sq if which == 0 else sk)[b]:] = 0
            plus, minus = list(args), list(args)
            plus[which] = (args[which] + np.float32(h) * dirn).astype(np.float32)
            minus[which] = (args[which] - np.float32(h) * dirn).astype(np.float32)
            assert np.array_equal(plus[which].astype(np.float64) - args[which],
                                  h * dirn.astype(np.float64)), "perturbation not exact"
            fd = (loss(*plus) - loss(*minus)) / (2 * h)
            an = float((grad * dirn.astype(np.float64)).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (ci, which, fd, an)


def pin_bwd_invariants(ol):
    """Consequences of the softmax definition:
    * the scores of a row shift by the same q.c when every key moves by c,
      and softmax ignores a shift, so the keys' gradients sum to zero;
    * the probabilities of a row sum to one, so the values' gradients of a
      KV head sum to the sum of dO over the rows (with a key) of its query heads;
    * identical keys give every query a zero gradient;
    * a constant V makes O independent of the scores: dQ = dK = 0;
    * dO = 0 gives zero gradients everywhere."""
    B, Hq, Hkv, Q, K, D, Dv = 2, 6, 2, 7, 10, 8, 5
    sq, sk = [7, 5], [10, 6]
    for w, mask in ((0, 0), (4, 0), (0, 1), (0, 2)):
        q, k, v, dout = _bwd_inputs(800 + w + mask, B, Hq, Hkv, Q, K, D, Dv)
        kw = dict(B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv, seqlens_q=sq, seqlens_k=sk,
                  window=w, scale=0.35, mask=mask)
        dq, dk, dv = ol.attn_bwd_padded(q, k, v, dout, **kw)
        G = Hq // Hkv
        for b in range(B):
            Qb, Kb = sq[b], sk[b]
            has = mask_matrix(Qb, Kb, w, mask).any(axis=1)
            assert np.allclose(dk[b].sum(axis=0), 0.0, atol=1e-12), (w, mask, b)
            for kh in range(Hkv):
                want = dout[b, :Qb][has][:, kh * G:(kh + 1) * G].astype(np.float64).sum(axis=(0, 1))
                assert np.allclose(dv[b, :, kh].sum(axis=0), want, atol=1e-12), (w, mask, b, kh)
        k_same = np.broadcast_to(k[:, :1], k.shape).copy()
        dq2, _, _ = ol.attn_bwd_padded(q, k_same, v, dout, **kw)
        assert np.allclose(dq2, 0.0, atol=1e-12), ("identical keys", w, mask)
        v_const = np.broadcast_to(v[:, :1], v.shape).copy()
        dq3, dk3, _ = ol.attn_bwd_padded(q, k, v_const, dout, **kw)
        assert np.allclose(dq3, 0.0, atol=1e-12) and np.allclose(dk3, 0.0, atol=1e-12), \
            ("constant V", w, mask)
        z = ol.attn_bwd_padded(q, k, v, np.zeros_like(dout), **kw)
        assert all(np.all(t == 0.0) for t in z), ("dO = 0", w, mask)


def pin_bwd_sampled_matches_full(ol):
    """The sampled backward (rows of dQ, key blocks of dK / dV, for checks of
    large problems) gives the pinned full backward's values."""
    for ci, (B, Hq, Hkv, Q, K, D, Dv, w, sq, sk, mask) in enumerate(BWD_CASES):
        q, k, v, dout = _bwd_inputs(900 + ci, B, Hq, Hkv, Q, K, D, Dv)
        kw = dict(B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv, seqlens_q=sq, seqlens_k=sk,
                  window=w, scale=0.3, mask=mask)
        dq, dk, dv = ol.attn_bwd_padded(q, k, v, dout, **kw)
        rows = np.array([(b, qi, h) for b in range(B) for qi in range(Q) for h in range(Hq)],
                        np.int32)
        sdq, _, _ = ol.attn_bwd_sampled(q, k, v, dout, rows=rows, **kw)
        assert np.array_equal(sdq, dq.reshape(-1, D)), ci
        for b in range(B):
            for kh in range(Hkv):
                for k0, k1 in ((0, K), (K // 2, K), (1, 2)):
                    _, sdk, sdv = ol.attn_bwd_sampled(q, k, v, dout, key_block=(b, kh, k0, k1),
                                                      **kw)
                    assert np.allclose(sdk, dk[b, k0:k1, kh], rtol=1e-12, atol=1e-14), (ci, b)
                    assert np.allclose(sdv, dv[b, k0:k1, kh], rtol=1e-12, atol=1e-14), (ci, b)


# ---------------------------------------------------------------------------
# the arbitrary (boolean) mask extension

def sdpa_reference_allow(q, k, v, Qb, Kb, Hq, Hkv, window, scale, mask, allow):
    """fp64 torch SDPA for one sequence with a per-head boolean mask: the
    numpy-triangle mask of ``mask``/``window`` ANDed with ``allow`` [Hm,Qb,Kb]
    (Hm = 1 broadcasts over the heads).  Returns (o [Qb,Hq,Dv], lse [Qb,Hq],
    has [Qb,Hq])."""
    G = Hq // Hkv
    qt = torch.from_numpy(np.asarray(q, np.float64)).permute(1, 0, 2)       # [Hq,Qb,D]
    kt = torch.from_numpy(np.asarray(k, np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
    vt = torch.from_numpy(np.asarray(v, np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)
    m = mask_matrix(Qb, Kb, window, mask)[None] & np.broadcast_to(allow, (Hq, Qb, Kb))
    has = m.any(axis=2)                                                     # [Hq,Qb]
    mt = torch.from_numpy(np.ascontiguousarray(m))
    safe = mt.clone()
    safe[~torch.from_numpy(has)] = True
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.unsqueeze(0), kt.unsqueeze(0), vt.unsqueeze(0), attn_mask=safe.unsqueeze(0),
        scale=scale)[0]
    sc = torch.matmul(qt, kt.transpose(1, 2)) * scale
    sc = sc.masked_fill(~mt, -math.inf)
    lse = torch.logsumexp(sc, dim=-1)
    return o.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy(), has.T


ALLOW_CASES = [
    # B, Hq, Hkv, Q, K, D, Dv, window, mask, Hm, density, seqlens_q, seqlens_k
    (2, 4, 2, 10, 23, 8, 6, 0, 2, 1, 0.5, None, None),       # a pure arbitrary mask, shared
    (1, 6, 3, 12, 12, 5, 7, 0, 0, 6, 0.3, None, None),       # causal AND a per-head mask
    (2, 4, 1, 9, 31, 8, 8, 4, 0, 4, 0.7, [9, 5], [31, 12]),  # window, per-head, ragged
    (1, 4, 2, 14, 20, 6, 6, 3, 1, 1, 0.6, None, None),       # top-left causal + window
]


def pin_allow_sdpa(ol):
    for ci, (B, Hq, Hkv, Q, K, D, Dv, w, mode, Hm, dens, sq, sk) in enumerate(ALLOW_CASES):
        q, k, v = rng_inputs(300 + ci, B, Hq, Hkv, Q, K, D, Dv)
        allow = np.random.default_rng(400 + ci).random((B, Hm, Q, K)) < dens
        allow[:, :, 1, :] = False          # a row with no allowed key in every case
        scale = 1.0 / math.sqrt(D) * (1.0 + 0.3 * ci)
        o, lse = ol.attn_padded_allow(q, k, v, allow, B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv,
                                      seqlens_q=sq, seqlens_k=sk, window=w, scale=scale,
                                      mask=mode)
        for b in range(B):
            Qb = Q if sq is None else sq[b]
            Kb = K if sk is None else sk[b]
            assert np.all(o[b, Qb:] == 0.0) and np.all(lse[b, Qb:] == -math.inf), (ci, b)
            if Qb == 0:
                continue
            ro, rl, has = sdpa_reference_allow(q[b, :Qb], k[b, :Kb], v[b, :Kb], Qb, Kb, Hq, Hkv,
                                               w, scale, mode, allow[b, :, :Qb, :Kb])
            ob, lb = o[b, :Qb], lse[b, :Qb]
            assert has.any() and not has.all(), ("case mixes empty and non-empty rows", ci)
            assert np.allclose(ob[has], ro[has], atol=1e-12, rtol=1e-10), (ci, b)
            assert np.allclose(lb[has], rl[has], atol=1e-12, rtol=1e-12), (ci, b)
            assert np.all(ob[~has] == 0.0) and not np.any(np.signbit(ob[~has])), (ci, b)
            assert np.all(lb[~has] == -math.inf), (ci, b)


def pin_allow_invariants(ol):
    B, Hq, Hkv, Q, K, D, Dv = 2, 4, 2, 11, 17, 8, 5
    q, k, v = rng_inputs(31, B, Hq, Hkv, Q, K, D, Dv)
    kw = dict(B=B, Hq=Hq, Hkv=Hkv, Q=Q, K=K, D=D, Dv=Dv)
    G = Hq // Hkv
    # every key allowed: the plain masks, bit for bit
    for mode, w in ((0, 0), (0, 5), (1, 3), (2, 0)):
        ones = np.ones((B, 1, Q, K), bool)
        oa, la = ol.attn_padded_allow(q, k, v, ones, window=w, mask=mode, **kw)
        op, lp = ol.attn_padded(q, k, v, window=w, mask=mode, **kw)
        assert np.array_equal(oa, op) and np.array_equal(la, lp), ("all allowed", mode, w)
    # the bottom-right triangle as an arbitrary mask with no mask mode = the causal rule
    tri = np.broadcast_to(np.tril(np.ones((Q, K), bool), k=K - Q), (B, Hq, Q, K))
    oa, la = ol.attn_padded_allow(q, k, v, tri, mask=2, **kw)
    op, lp = ol.attn_padded(q, k, v, mask=0, **kw)
    assert np.array_equal(oa, op) and np.array_equal(la, lp), "triangle == causal"
    # nothing allowed: +0 and -inf on every row
    oz, lz = ol.attn_padded_allow(q, k, v, np.zeros((B, Hq, Q, K), bool), mask=2, **kw)
    assert np.all(oz == 0.0) and not np.any(np.signbit(oz)) and np.all(lz == -math.inf)
    # one allowed key per (row, head): its V row, and its score as the LSE
    g = np.random.default_rng(32)
    one = np.zeros((B, Hq, Q, K), bool)
    pick = g.integers(0, K, size=(B, Hq, Q))
    for b in range(B):
        for h in range(Hq):
            one[b, h, np.arange(Q), pick[b, h]] = True
    o1, l1 = ol.attn_padded_allow(q, k, v, one, mask=2, **kw)
    scale = 1.0 / math.sqrt(D)
    for b in range(B):
        for h in range(Hq):
            for i in range(Q):
                kk = pick[b, h, i]
                assert np.allclose(o1[b, i, h], v[b, kk, h // G], atol=1e-14), "one key"
                s = scale * float(np.dot(q[b, i, h].astype(np.float64), k[b, kk, h // G]))
                assert abs(l1[b, i, h] - s) < 1e-12, "one key lse"


ALL_PINS = [pin_golden, pin_sdpa, pin_invariants, pin_packed_matches_padded,
            pin_rows_match_full, pin_legal_pairs, pin_sdpa_masks, pin_bwd_autograd,
            pin_bwd_finite_differences, pin_bwd_invariants, pin_bwd_sampled_matches_full,
            pin_allow_sdpa, pin_allow_invariants]
