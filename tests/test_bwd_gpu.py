"""attn_bwd / attn_bwd_varlen against the oracle's fp64 backward.

The oracle recomputes O and LSE from its own definition; the library takes
the O and LSE its forward produced (as a caller would), so the bf16 / fp16
comparison also carries the forward's rounding of O.

Tolerances (the gradients are sums of many rounded products; the kernels
round P and dS to the storage type before the tensor-core products and the
results to the storage type at the end):
* fp32 storage: max |err| <= 1e-4 * max(1, max |ref|) per tensor;
* bf16 / fp16: max |err| <= 2e-2 * max(1, max |ref|) and
  ||err||_2 <= 1e-2 * ||ref||_2 per tensor;
* padded rows / keys, rows without a legal key and keys no row attends to:
  exactly zero.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tests.oracle_pins import mask_matrix
from causal_gqa_attention_online_gb300 import (AttnError, attn_bwd, attn_bwd_varlen, attn_fwd,
                                               attn_fwd_varlen, synth)

pytestmark = pytest.mark.gpu
NAN = float("nan")
BTOL = {"f32": (1e-4, None), "bf16": (2e-2, 1e-2), "f16": (2e-2, 1e-2)}


def gpu_bwd(inp, dout, algo="auto", mask=0):
    dev = torch.device("cuda")
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    sq = None if inp.seqlens_q is None else torch.from_numpy(inp.seqlens_q).to(dev)
    sk = None if inp.seqlens_k is None else torch.from_numpy(inp.seqlens_k).to(dev)
    o, lse = attn_fwd(q, k, v, seqlens_q=sq, seqlens_k=sk, window=inp.window, scale=inp.scale,
                      mask=parity.MASK_NAMES[mask])
    g = dout.to(dev)
    bufs = [torch.full((t.numel() + parity.GUARD,), NAN, dtype=t.dtype, device=dev) for t in (q, k, v)]
    dq, dk, dv = (b[:t.numel()].view(t.shape) for b, t in zip(bufs, (q, k, v)))
    attn_bwd(q, k, v, o, lse, g, dq, dk, dv, seqlens_q=sq, seqlens_k=sk, window=inp.window,
             scale=inp.scale, algo=algo, mask=parity.MASK_NAMES[mask])
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.isnan(b[-parity.GUARD:].float()).all(), "write past the end of a gradient"
    return tuple(t.float().cpu().numpy() for t in (dq, dk, dv))


def oracle_bwd(inp, dout, mask=0):
    return oracle.attn_bwd_padded(
        synth.exact_f32(inp.q), synth.exact_f32(inp.k), synth.exact_f32(inp.v),
        synth.exact_f32(dout), B=inp.B, Hq=inp.Hq, Hkv=inp.Hkv, Q=inp.Q, K=inp.K, D=inp.D,
        Dv=inp.Dv, seqlens_q=inp.seqlens_q, seqlens_k=inp.seqlens_k, window=inp.window,
        scale=inp.scale, mask=mask)


def structural_zeros(B, Q, K, seqlens_q, seqlens_k, window, mask):
    """[B,Q] rows and [B,K] keys that take part in no legal pair (padding,
    rows without a legal key, keys no row attends to)."""
    zq = np.ones((B, Q), bool)
    zk = np.ones((B, K), bool)
    for b in range(B):
        Qb = Q if seqlens_q is None else int(np.clip(seqlens_q[b], 0, Q))
        Kb = K if seqlens_k is None else int(np.clip(seqlens_k[b], 0, K))
        if Qb and Kb:
            m = mask_matrix(Qb, Kb, window if window < Kb else 0, mask)
            zq[b, :Qb] = ~m.any(axis=1)
            zk[b, :Kb] = ~m.any(axis=0)
    return zq, zk


def compare(dtype, got, ref, what, zeros=None):
    mx, l2 = BTOL[dtype]
    for i, (name, a, r) in enumerate(zip(("dq", "dk", "dv"), got, ref)):
        assert np.isfinite(a).all(), f"{what} {name}: non-finite values"
        if zeros is not None:
            z = zeros[0] if i == 0 else zeros[1]
            assert np.all(a[z] == 0.0) and np.all(r[z] == 0.0), \
                f"{what} {name}: non-zero gradient outside every legal pair"
        err = np.abs(a - r)
        scale = max(1.0, float(np.abs(r).max(initial=0.0)))
        assert err.max(initial=0.0) <= mx * scale, \
            f"{what} {name}: max err {err.max():.3e} > {mx * scale:.3e}"
        if l2 is not None and r.size:
            assert np.linalg.norm(a - r) <= l2 * max(np.linalg.norm(r), 1e-30), \
                f"{what} {name}: l2 err {np.linalg.norm(a - r):.3e} vs {np.linalg.norm(r):.3e}"


def compare_one(dtype, got, ref, what):
    """One tensor under the bar of compare()."""
    mx, l2 = BTOL[dtype]
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - ref)
    scale = max(1.0, float(np.abs(ref).max(initial=0.0)))
    assert err.max(initial=0.0) <= mx * scale, f"{what}: max err {err.max():.3e}"
    if l2 is not None and ref.size:
        assert np.linalg.norm(got - ref) <= l2 * max(np.linalg.norm(ref), 1e-30), \
            f"{what}: l2 err {np.linalg.norm(got - ref):.3e} vs {np.linalg.norm(ref):.3e}"


CASES = [
    # dtype, algo, B, Hq, Hkv, Q, K, D, Dv, window, mask, ragged
    ("bf16", "mma", 2, 8, 2, 200, 200, 128, 128, 0, 0, True),
    ("bf16", "mma", 1, 8, 2, 130, 330, 128, 128, 0, 0, False),
    ("f16", "mma", 2, 4, 2, 150, 300, 64, 64, 70, 0, True),
    ("bf16", "mma", 2, 4, 1, 97, 180, 80, 48, 0, 0, True),
    ("bf16", "mma", 1, 6, 6, 120, 120, 64, 128, 0, 1, False),
    ("bf16", "mma", 2, 8, 4, 70, 90, 128, 64, 0, 2, True),
    ("bf16", "mma", 3, 32, 8, 1, 700, 128, 128, 0, 0, True),
    ("bf16", "generic", 2, 8, 2, 100, 140, 128, 128, 0, 0, True),
    ("bf16", "generic", 1, 4, 2, 60, 75, 256, 256, 20, 0, False),
    ("f16", "generic", 1, 4, 2, 50, 70, 40, 24, 0, 1, False),
    ("f32", "auto", 2, 4, 2, 64, 128, 64, 64, 0, 0, True),
    ("f32", "auto", 1, 8, 2, 33, 90, 80, 96, 9, 0, False),
    ("f32", "generic", 2, 6, 3, 40, 40, 32, 16, 0, 2, True),
    ("bf16", "mma", 1, 16, 2, 90, 140, 128, 128, 0, 0, True),    # G = 8
    ("f16", "mma", 1, 32, 2, 40, 70, 64, 64, 30, 0, False),      # G = 16, window
    ("bf16", "mma", 2, 8, 2, 300, 300, 128, 128, 0, 0, False),   # several row tiles of a key tile
    # tcgen05 dQ and dK/dV (mma.sync dK/dV where Hq / Hkv does not divide 128)
    ("bf16", "tcgen05", 2, 8, 2, 200, 200, 128, 128, 0, 0, True),
    ("bf16", "tcgen05", 1, 8, 2, 130, 330, 128, 128, 0, 0, False),
    ("f16", "tcgen05", 2, 4, 2, 150, 300, 64, 64, 70, 0, True),
    ("bf16", "tcgen05", 2, 4, 1, 97, 180, 80, 112, 0, 0, True),
    ("bf16", "tcgen05", 1, 6, 6, 120, 120, 64, 128, 0, 1, False),
    ("bf16", "tcgen05", 2, 8, 4, 70, 90, 128, 64, 0, 2, True),
    ("bf16", "tcgen05", 3, 32, 8, 1, 700, 128, 128, 0, 0, True),
    ("f16", "tcgen05", 1, 32, 2, 40, 70, 64, 64, 30, 0, False),
    ("bf16", "tcgen05", 1, 4, 2, 300, 40, 128, 128, 0, 0, False),  # Q > K: rows without keys
    ("bf16", "tcgen05", 1, 6, 2, 90, 150, 128, 128, 0, 0, True),   # G = 3: mma.sync dK/dV
    ("bf16", "tcgen05", 1, 16, 1, 70, 300, 128, 128, 50, 0, True),  # G = 16, window
    ("f16", "tcgen05", 2, 8, 8, 260, 260, 96, 80, 0, 1, True),     # MHA, padded widths
    ("bf16", "tcgen05", 1, 64, 2, 50, 120, 64, 64, 0, 0, True),    # G = 32: 4 positions a row tile
    ("bf16", "tcgen05", 1, 64, 1, 33, 90, 128, 128, 0, 0, True),   # G = 64
    ("f16", "tcgen05", 1, 128, 1, 21, 60, 64, 64, 0, 1, False),    # G = 128: one position a tile
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}-" + "x".join(map(str, c[2:])))
def test_bwd_parity(case):
    dtype, algo, B, Hq, Hkv, Q, K, D, Dv, window, mask, ragged = case
    sq = sk = None
    if ragged:
        g = np.random.default_rng(B * 31 + Q)
        sk = g.integers(0, K + 1, size=B).astype(np.int32)
        sq = np.minimum(g.integers(0, Q + 1, size=B), sk).astype(np.int32) if Q > 1 else None
        sk[0] = K
        if sq is not None:
            sq[0] = Q
            if B > 1:
                sq[1] = 0
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=71 + Q, seqlens_q=sq,
                            seqlens_k=sk, window=window, pad_value=NAN)
    dout = synth.make_dout(inp, seed=72 + K, pad_value=NAN)
    got = gpu_bwd(inp, dout, algo, mask)
    ref = oracle_bwd(inp, dout, mask)
    compare(dtype, got, ref, f"bwd {case}",
            structural_zeros(B, Q, K, sq, sk, window, mask))


@pytest.mark.parametrize("algo", ["mma", "tcgen05"])
def test_bwd_negative_scale(algo):
    inp = synth.make_padded(1, 8, 2, 100, 150, 128, 128, "bf16", seed=85, scale=-0.15)
    dout = synth.make_dout(inp, seed=86)
    compare("bf16", gpu_bwd(inp, dout, algo), oracle_bwd(inp, dout), f"negative scale {algo}")


def test_bwd_deterministic_and_algos_agree():
    inp = synth.make_padded(2, 8, 2, 190, 260, 128, 128, "bf16", seed=81)
    dout = synth.make_dout(inp, seed=82)
    a = gpu_bwd(inp, dout, "mma")
    b = gpu_bwd(inp, dout, "mma")
    for x, y in zip(a, b):
        assert np.array_equal(x, y), "two runs differ"
    c = gpu_bwd(inp, dout, "generic")
    t1 = gpu_bwd(inp, dout, "tcgen05")
    t2 = gpu_bwd(inp, dout, "tcgen05")
    for x, y in zip(t1, t2):
        assert np.array_equal(x, y), "two tcgen05 runs differ"
    ref = oracle_bwd(inp, dout)
    compare("bf16", c, ref, "generic")
    compare("bf16", a, ref, "mma")
    compare("bf16", t1, ref, "tcgen05")


@pytest.mark.parametrize("window", [0, 45])
def test_bwd_varlen_matches_padded(window):
    sq = np.array([0, 130, 64, 1, 200], np.int32)
    sk = np.array([50, 200, 64, 300, 200], np.int32)
    pk = synth.make_packed(sq, sk, 8, 2, 128, 128, "bf16", seed=91, window=window)
    dev = torch.device("cuda")
    q, k, v = pk.q.to(dev), pk.k.to(dev), pk.v.to(dev)
    cq = torch.from_numpy(pk.cu_seqlens_q).to(dev)
    ck = torch.from_numpy(pk.cu_seqlens_k).to(dev)
    o, lse = attn_fwd_varlen(q, k, v, cq, ck, pk.Q, pk.K, window=window)
    dout = synth.make_dout(pk, seed=92).to(dev)
    dq, dk, dv = attn_bwd_varlen(q, k, v, o, lse, dout, cq, ck, pk.Q, pk.K, window=window)
    torch.cuda.synchronize()
    # the same problem in the padded layout, through the oracle
    B, Qm, Km = pk.B, pk.Q, pk.K

    def pad(x, cu, cap):
        out = np.zeros((B, cap) + x.shape[1:], np.float32)
        for b in range(B):
            out[b, :cu[b + 1] - cu[b]] = x[cu[b]:cu[b + 1]]
        return out

    cqn, ckn = pk.cu_seqlens_q, pk.cu_seqlens_k
    ref = oracle.attn_bwd_padded(pad(synth.exact_f32(pk.q), cqn, Qm), pad(synth.exact_f32(pk.k), ckn, Km),
                                 pad(synth.exact_f32(pk.v), ckn, Km),
                                 pad(dout.float().cpu().numpy(), cqn, Qm), B=B, Hq=8, Hkv=2, Q=Qm,
                                 K=Km, D=128, Dv=128, seqlens_q=sq, seqlens_k=sk, scale=pk.scale,
                                 window=window)
    got = (pad(dq.float().cpu().numpy(), cqn, Qm), pad(dk.float().cpu().numpy(), ckn, Km),
           pad(dv.float().cpu().numpy(), ckn, Km))
    compare("bf16", got, ref, "varlen")


def test_bwd_rejects_tensor_kernels_on_fp32_and_bad_algo():
    inp = synth.make_padded(1, 2, 1, 8, 8, 64, 64, "f32", seed=93)
    dout = synth.make_dout(inp, seed=94)
    with pytest.raises(AttnError) as ei:
        gpu_bwd(inp, dout, "mma")
    assert ei.value.status == 2
    with pytest.raises(AttnError) as ei:
        gpu_bwd(inp, dout, "tcgen05")
    assert ei.value.status == 2
    with pytest.raises(AttnError) as ei:
        gpu_bwd(inp, dout, "decode")
    assert ei.value.status == 1


def test_bwd_misaligned_gradients_rejected():
    """Gradient buffers 8 bytes past a 16-byte boundary are refused before any
    launch (the kernels store 16 bytes at a time), for every kernel choice,
    and the buffers are left untouched."""
    inp = synth.make_padded(1, 8, 2, 150, 200, 128, 128, "bf16", seed=95)
    dout = synth.make_dout(inp, seed=96)
    dev = torch.device("cuda")
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    o, lse = attn_fwd(q, k, v, scale=inp.scale)
    g = dout.to(dev)

    def shifted(t):
        buf = torch.full((t.numel() + 4,), NAN, dtype=t.dtype, device=dev)
        return buf[4:].view(t.shape)  # 4 bf16 elements = 8 bytes in

    dq, dk, dv = shifted(q), shifted(k), shifted(v)
    assert dq.data_ptr() % 16 == 8
    for algo in ("auto", "tcgen05", "mma", "generic"):
        with pytest.raises(AttnError) as ei:
            attn_bwd(q, k, v, o, lse, g, dq, dk, dv, scale=inp.scale, algo=algo)
        assert ei.value.status == 1, algo
    torch.cuda.synchronize()
    assert all(torch.isnan(t.float()).all() for t in (dq, dk, dv))


def test_bwd_no_query_rows_zeroes_key_gradients():
    dev = torch.device("cuda")
    q = torch.zeros((2, 0, 4, 64), dtype=torch.bfloat16, device=dev)
    k = torch.randn((2, 16, 2, 64), device=dev).bfloat16()
    v = torch.randn((2, 16, 2, 64), device=dev).bfloat16()
    o = torch.zeros((2, 0, 4, 64), dtype=torch.bfloat16, device=dev)
    lse = torch.zeros((2, 0, 4), dtype=torch.float32, device=dev)
    dk = torch.full_like(k, NAN)
    dv = torch.full_like(v, NAN)
    attn_bwd(q, k, v, o, lse, o, None, dk, dv)
    torch.cuda.synchronize()
    assert bool((dk == 0).all()) and bool((dv == 0).all())


def test_bwd_full_size_sampled():
    """attn_bwd on the benchmark's launch (bf16 causal B=4 Hq=32 Hkv=8
    Q=K=4096 D=Dv=128, dO ~ N(0,1)): dQ of sampled rows and dK / dV of the
    last 64 keys of two (sequence, KV head) pairs against the oracle, and
    over every key the sum the definition fixes (a KV head's value gradients
    sum to its rows' dO)."""
    inp = synth.prefill_bf16_b4_h32x8_s4096_d128()
    dout = synth.make_dout(inp, seed=4321)
    dev = torch.device("cuda")
    q, k, v, g = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), dout.to(dev)
    o, lse = attn_fwd(q, k, v)
    dq, dk, dv = attn_bwd(q, k, v, o, lse, g)
    torch.cuda.synchronize()
    B, Hq, Hkv, S, D = inp.B, inp.Hq, inp.Hkv, inp.Q, inp.D
    G = Hq // Hkv
    kw = dict(B=B, Hq=Hq, Hkv=Hkv, Q=S, K=S, D=D, Dv=D, scale=inp.scale)
    qf, kf, vf, gf = (synth.exact_f32(t) for t in (inp.q, inp.k, inp.v, dout))
    rng = np.random.default_rng(5)
    rows = np.stack([rng.integers(0, B, 1200), rng.integers(0, S, 1200),
                     rng.integers(0, Hq, 1200)], axis=1).astype(np.int32)
    rows = np.concatenate([rows, [[0, 0, 0], [B - 1, S - 1, Hq - 1], [1, S - 1, 5]]]).astype(np.int32)
    ref_q, _, _ = oracle.attn_bwd_sampled(qf, kf, vf, gf, rows=rows, **kw)
    got_q = dq.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]]
    compare_one("bf16", got_q, ref_q, "full-size dq rows")
    dkc, dvc = dk.float().cpu().numpy(), dv.float().cpu().numpy()
    for b, kh in ((0, 0), (B - 1, Hkv - 1)):
        _, ref_k, ref_v = oracle.attn_bwd_sampled(qf, kf, vf, gf, key_block=(b, kh, S - 64, S), **kw)
        compare_one("bf16", dkc[b, S - 64:, kh], ref_k, f"full-size dk keys b={b} kh={kh}")
        compare_one("bf16", dvc[b, S - 64:, kh], ref_v, f"full-size dv keys b={b} kh={kh}")
    # every (sequence, KV head): the value gradients sum to the dO of the
    # group's rows (each row's probabilities sum to one).  Rounding P to bf16
    # moves a row's sum by at most u = 2^-8 of its |dO|, rounding dV by u of
    # each |dV|: the bound is twice that.
    u = 2.0 ** -8
    sum_dv = dv.double().sum(dim=1)                                  # [B, Hkv, Dv]
    gg = g.double().view(B, S, Hkv, G, D)
    want_dv = gg.sum(dim=(1, 3))
    bound = 2 * u * (dv.double().abs().sum(dim=1) + gg.abs().sum(dim=(1, 3))) + 1e-3
    assert bool(((sum_dv - want_dv).abs() <= bound).all()), "value gradients do not sum to dO"


def test_sdpa_example_shape_forward_and_backward():
    """The SDPA usage example of "Accelerating PyTorch on AMD GPUs with FlyDSL"
    (q, k, v of shape (4, 16, 4096, 128) bf16, is_causal=True, then the
    backward), as a synthetic shape: MHA (G = 1), so the dK/dV kernel's row
    tiles hold 128 positions of one head.  Forward: every row against the
    oracle; backward: sampled dQ rows and the last 64 keys of two heads."""
    inp = synth.make_padded(4, 16, 16, 4096, 4096, 128, 128, "bf16", seed=1166)
    parity.check(inp, "auto", "SDPA example forward")
    dout = synth.make_dout(inp, seed=1167)
    dev = torch.device("cuda")
    q, k, v, g = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev), dout.to(dev)
    o, lse = attn_fwd(q, k, v)
    dq, dk, dv = attn_bwd(q, k, v, o, lse, g)
    torch.cuda.synchronize()
    B, H, S, D = 4, 16, 4096, 128
    kw = dict(B=B, Hq=H, Hkv=H, Q=S, K=S, D=D, Dv=D, scale=inp.scale)
    qf, kf, vf, gf = (synth.exact_f32(t) for t in (inp.q, inp.k, inp.v, dout))
    rng = np.random.default_rng(1168)
    rows = np.stack([rng.integers(0, B, 600), rng.integers(0, S, 600),
                     rng.integers(0, H, 600)], axis=1).astype(np.int32)
    ref_q, _, _ = oracle.attn_bwd_sampled(qf, kf, vf, gf, rows=rows, **kw)
    compare_one("bf16", dq.float().cpu().numpy()[rows[:, 0], rows[:, 1], rows[:, 2]], ref_q,
                "SDPA example dq rows")
    dkc, dvc = dk.float().cpu().numpy(), dv.float().cpu().numpy()
    for b, kh in ((0, 3), (B - 1, H - 1)):
        _, ref_k, ref_v = oracle.attn_bwd_sampled(qf, kf, vf, gf, key_block=(b, kh, S - 64, S), **kw)
        compare_one("bf16", dkc[b, S - 64:, kh], ref_k, f"SDPA example dk b={b} h={kh}")
        compare_one("bf16", dvc[b, S - 64:, kh], ref_v, f"SDPA example dv b={b} h={kh}")


@pytest.mark.parametrize("Hq,Hkv,launches", [(8, 2, 2), (6, 2, 3)])
def test_bwd_tcgen05_launch_sequence(Hq, Hkv, launches):
    """The tcgen05 backward's launches: with the tcgen05 dK/dV kernel (G =
    Hq / Hkv divides 128) two, the dQ kernel -- which computes each of its
    rows' Dq = rowsum(dO * O) from the O tile it stages and writes it -- then
    the dK/dV kernel as its programmatic dependent; with the mma.sync dK/dV
    kernel (G = 3) three, the Dq launch first.  Gradients against the oracle
    in both cases, padded rows with NaN."""
    from causal_gqa_attention_online_gb300 import binding
    g = np.random.default_rng(Hq)
    sq = g.integers(1, 261, size=2).astype(np.int32)
    sk = np.maximum(sq, g.integers(1, 301, size=2)).astype(np.int32)
    inp = synth.make_padded(2, Hq, Hkv, 260, 300, 128, 128, "bf16", seed=81, seqlens_q=sq,
                            seqlens_k=sk, pad_value=NAN)
    dout = synth.make_dout(inp, seed=82, pad_value=NAN)
    dev = torch.device("cuda")
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    tsq, tsk = torch.from_numpy(sq).to(dev), torch.from_numpy(sk).to(dev)
    o, lse = attn_fwd(q, k, v, seqlens_q=tsq, seqlens_k=tsk, scale=inp.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    torch.cuda.synchronize()
    n0 = binding.kernel_launches()
    attn_bwd(q, k, v, o, lse, dout.to(dev), dq, dk, dv, seqlens_q=tsq, seqlens_k=tsk,
             scale=inp.scale, algo="tcgen05")
    torch.cuda.synchronize()
    assert binding.kernel_launches() - n0 == launches
    got = tuple(t.float().cpu().numpy() for t in (dq, dk, dv))
    ref = oracle_bwd(inp, dout)
    compare("bf16", got, ref, f"launch sequence Hq={Hq} Hkv={Hkv}",
            structural_zeros(2, 260, 300, sq, sk, 0, 0))
