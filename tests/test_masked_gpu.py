"""GPU parity of the arbitrary (boolean) mask, attn_fwd_masked, against the
fp64 oracle's masked definition (oracle_attn_padded_allow) on the same seeded
inputs, element by element.

"Attention execution mapping" (LuisaCompute), section 7: an arbitrary mask is
a semantic extension that needs an independent oracle.  The mask is ANDed
with the mask mode and the window; rows left without a legal key are +0 /
-inf, compared bit-exactly.  Cases: random element masks and random
block-sparse masks (128-key blocks) shared by every head or one per head, all
allowed, nothing allowed, ragged sequences with NaN padding, windows, both
causal modes, fp32 on the CUDA-core kernel, bf16 / fp16 on the tcgen05 kernel,
and a key block that no row may attend to holding NaN: the tcgen05 kernel
skips such dead tiles without loading them, so the NaN never reaches O.
"""
import math

import numpy as np
import pytest
import torch

import causal_gqa_attention_online_gb300 as attn
import oracle
from causal_gqa_attention_online_gb300 import build_ext, synth
from tests import parity

pytestmark = pytest.mark.gpu

NAN = float("nan")
MODES = {"causal": 0, "causal_top_left": 1, "none": 2}


@pytest.fixture(scope="module", autouse=True)
def built():
    build_ext.build()


def block_mask(g, B, Hm, Q, K, qblock, density):
    """A mask of (qblock x 128)-blocks, each allowed with the given density."""
    nq, nk = (Q + qblock - 1) // qblock, (K + 127) // 128
    blocks = g.random((B, Hm, nq, nk)) < density
    m = np.repeat(np.repeat(blocks, qblock, axis=2), 128, axis=3)
    return m[:, :, :Q, :K]


def run_masked(inp, allow, algo, mode, dev="cuda"):
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    words = attn.pack_mask(torch.from_numpy(allow)).to(dev)
    sq = None if inp.seqlens_q is None else torch.from_numpy(inp.seqlens_q).to(dev)
    sk = None if inp.seqlens_k is None else torch.from_numpy(inp.seqlens_k).to(dev)
    obuf = torch.full((inp.B * inp.Q * inp.Hq * inp.Dv + 256,), NAN, dtype=q.dtype, device=dev)
    lbuf = torch.full((inp.B * inp.Q * inp.Hq + 256,), NAN, dtype=torch.float32, device=dev)
    o = obuf[:-256].view(inp.B, inp.Q, inp.Hq, inp.Dv)
    lse = lbuf[:-256].view(inp.B, inp.Q, inp.Hq)
    attn.attn_fwd_masked(q, k, v, words, o, lse, seqlens_q=sq, seqlens_k=sk, window=inp.window,
                         scale=inp.scale, algo=algo, mask=mode)
    torch.cuda.synchronize()
    assert torch.isnan(obuf[-256:].float()).all() and torch.isnan(lbuf[-256:]).all()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def check(inp, allow, algo, mode="none", what=""):
    o, lse = run_masked(inp, allow, algo, mode)
    ro, rl = oracle.attn_padded_allow(
        synth.exact_f32(inp.q), synth.exact_f32(inp.k), synth.exact_f32(inp.v), allow,
        B=inp.B, Hq=inp.Hq, Hkv=inp.Hkv, Q=inp.Q, K=inp.K, D=inp.D, Dv=inp.Dv,
        seqlens_q=inp.seqlens_q, seqlens_k=inp.seqlens_k, window=inp.window, scale=inp.scale,
        mask=MODES[mode])
    return parity.compare(inp.dtype, o, lse, ro, rl, what or f"{algo} {mode}")


CASES = [
    # algo, dtype, B, Hq, Hkv, Q, K, D, Dv, mode, window, heads, kind, density
    ("generic", "f32", 2, 4, 2, 70, 150, 64, 48, "none", 0, "shared", "elem", 0.4),
    ("generic", "f32", 1, 8, 2, 90, 90, 32, 32, "causal", 20, "per_head", "elem", 0.6),
    ("generic", "bf16", 2, 4, 1, 33, 200, 64, 64, "causal_top_left", 0, "shared", "block", 0.5),
    ("tcgen05", "bf16", 2, 8, 2, 300, 500, 128, 128, "none", 0, "shared", "block", 0.5),
    ("tcgen05", "bf16", 2, 8, 2, 300, 500, 128, 128, "causal", 0, "per_head", "elem", 0.3),
    ("tcgen05", "f16", 1, 8, 2, 257, 700, 64, 64, "causal", 200, "shared", "block", 0.6),
    ("tcgen05", "bf16", 1, 16, 4, 400, 400, 128, 96, "causal_top_left", 0, "per_head", "block", 0.4),
    ("tcgen05", "bf16", 3, 8, 8, 130, 260, 96, 80, "none", 0, "per_head", "elem", 0.05),
    ("tcgen05", "bf16", 2, 32, 8, 1, 1500, 128, 128, "none", 0, "shared", "block", 0.5),  # decode rows
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_masked_parity(case):
    algo, dtype, B, Hq, Hkv, Q, K, D, Dv, mode, w, heads, kind, dens = case
    g = np.random.default_rng(B * 131 + Q + K)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    sq = g.integers(0, Q + 1, size=B).astype(np.int32)
    sq[0] = Q
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=77, seqlens_q=sq,
                            seqlens_k=sk, window=w, pad_value=NAN)
    Hm = 1 if heads == "shared" else Hq
    if kind == "elem":
        allow = g.random((B, Hm, Q, K)) < dens
    else:
        allow = block_mask(g, B, Hm, Q, K, 64, dens)
    allow[:, :, min(2, Q - 1), :] = False  # a row left without a legal key
    check(inp, allow, algo, mode, f"{case}")


@pytest.mark.parametrize("algo,dtype", [("tcgen05", "bf16"), ("generic", "f32")])
def test_masked_all_and_nothing(algo, dtype):
    inp = synth.make_padded(2, 8, 2, 200, 333, 128, 128, dtype, seed=78)
    ones = np.ones((2, 1, 200, 333), bool)
    check(inp, ones, algo, "causal", "all allowed, causal")
    check(inp, ones, algo, "none", "all allowed, no mask")
    o, lse = run_masked(inp, np.zeros((2, 8, 200, 333), bool), algo, "none")
    assert np.all(o == 0.0) and not np.any(np.signbit(o)) and np.all(lse == -math.inf)


def test_masked_dead_tiles_are_not_loaded():
    """Keys [256, 384) are allowed to no row of any head: on the tcgen05
    kernel that 128-key tile is dead for every work unit and is skipped, so NaN
    in those K / V rows never reaches O (an element-wise masked product would
    turn 0 * NaN into NaN)."""
    B, Hq, Hkv, Q, K = 2, 8, 2, 300, 600
    inp = synth.make_padded(B, Hq, Hkv, Q, K, 128, 128, "bf16", seed=79)
    inp.k[:, 256:384] = NAN
    inp.v[:, 256:384] = NAN
    g = np.random.default_rng(80)
    allow = g.random((B, 1, Q, K)) < 0.5
    allow[:, :, :, 256:384] = False
    check(inp, allow, "tcgen05", "none", "dead tile with NaN")


def test_masked_full_size_block_sparse():
    """bf16 B=2 Hq=16 Hkv=4 Q=K=2048 D=128, causal AND a per-head block-sparse
    mask (64 x 128 blocks at density 0.5): every row against the oracle."""
    B, Hq, Hkv, S = 2, 16, 4, 2048
    inp = synth.make_padded(B, Hq, Hkv, S, S, 128, 128, "bf16", seed=81)
    allow = block_mask(np.random.default_rng(82), B, Hq, S, S, 64, 0.5)
    check(inp, allow, "auto", "causal", "block-sparse 2048")
