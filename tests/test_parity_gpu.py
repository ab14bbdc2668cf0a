"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs, element by element (tolerances in tests/parity.py).

Shapes: the named synthetic workloads, the held-out matrix of the
LuisaCompute attention-mapping page (section 7: Q/K tails, small Q with a
bottom-right offset, MQA/MHA/batch, long KV), reduction lengths
0/1/7/16/31/32/33/65 around tile edges (same page, section 21.4), windows,
Q > K, all-empty and K = 0 problems, and the packed layout with empty
sequences (Laya fast backends, numerical verification)."""
import math

import numpy as np
import pytest
import torch

from causal_gqa_attention_online_gb300 import AttnError, attn_fwd, attn_lse_combine, build_ext, synth
from tests import parity

pytestmark = pytest.mark.gpu

NAN = float("nan")


@pytest.fixture(scope="module", autouse=True)
def built():
    build_ext.build()


HELD_OUT = [
    # B, Hq, Hkv, Q, K, D, Dv
    (1, 4, 2, 65, 131, 64, 64),
    (1, 8, 2, 256, 1024, 64, 64),
    (1, 8, 2, 3, 67, 80, 96),
    (1, 4, 2, 65, 65, 64, 64),
    (2, 8, 1, 1, 2053, 80, 96),
    (1, 8, 8, 1, 2048, 64, 64),
    (1, 16, 4, 1, 8193, 128, 128),
    (1, 8, 2, 1, 32768, 64, 96),
    (1, 8, 2, 1, 2048, 64, 64),
    (1, 16, 4, 1, 4096, 128, 128),
]


def test_named_fp32_prefill():
    parity.check(synth.prefill_f32_b1_h4x2_q64_k128_d64(), "auto", "fp32 prefill 1,4,2,64,128")


def test_named_fp32_decode():
    parity.check(synth.decode_f32_b1_h8x2_k2053_d80x96(), "auto", "fp32 decode 1,8,2,1,2053")


@pytest.mark.parametrize("shape", HELD_OUT, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_generic_held_out(shape, dtype):
    B, Hq, Hkv, Q, K, D, Dv = shape
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=11)
    parity.check(inp, "generic", f"generic {dtype} {shape}")


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_generic_reduction_lengths(dtype):
    # lengths around the 32-key tile: 0/1/7/16/31/32/33/65; NaN in padded rows
    sk = np.array([0, 1, 7, 16, 31, 32, 33, 65], np.int32)
    sq = np.array([5, 1, 7, 3, 31, 32, 33, 65], np.int32)
    inp = synth.make_padded(8, 4, 2, 65, 65, 64, 48, dtype, seed=3, seqlens_q=sq, seqlens_k=sk,
                            pad_value=NAN)
    parity.check(inp, "generic", f"lengths {dtype}")


@pytest.mark.parametrize("window", [1, 7, 64, 199])
def test_generic_window(window):
    inp = synth.make_padded(2, 6, 2, 200, 200, 32, 32, "f32", seed=5, window=window)
    parity.check(inp, "generic", f"window {window}")


def test_generic_q_longer_than_k():
    # rows q < Qb - Kb have no legal key: +0 / -inf
    inp = synth.make_padded(2, 4, 2, 40, 10, 16, 16, "f32", seed=6)
    parity.check(inp, "generic", "Q > K")


def test_generic_all_empty_and_k_zero():
    inp = synth.make_padded(3, 4, 1, 9, 12, 16, 16, "bf16", seed=7,
                            seqlens_k=np.zeros(3, np.int32), pad_value=NAN)
    parity.check(inp, "generic", "all empty")
    inp = synth.make_padded(1, 4, 2, 5, 0, 16, 16, "f32", seed=8)
    parity.check(inp, "auto", "K = 0")


def test_generic_varlen_packed():
    sk = np.array([0, 5, 33, 130, 1, 64, 0, 300], np.int32)
    sq = np.minimum(sk, np.array([0, 5, 7, 64, 1, 64, 0, 100]))
    for dtype, w in (("f32", 0), ("bf16", 40), ("f16", 0)):
        inp = synth.make_packed(sq, sk, 8, 2, 64, 64, dtype, seed=9, window=w)
        parity.check(inp, "generic", f"varlen {dtype} w={w}")


def test_generic_split_kv_long_decode_with_lengths():
    # few units and long keys: the key axis is split and merged
    sk = np.array([0, 1, 511, 512, 513, 4000], np.int32)
    inp = synth.make_padded(6, 8, 2, 1, 4096, 64, 64, "bf16", seed=10, seqlens_k=sk,
                            pad_value=NAN)
    parity.check(inp, "generic", "split-KV lengths")


def test_lse_combine_entry_point():
    # two partials of a decode row: keys [0, c) (seqlens_k = c) and [c, Kb)
    # (window = Kb - c); their merge must equal the full row.
    B, Hq, Hkv, K, D, Dv = 2, 8, 2, 700, 64, 64
    inp = synth.make_padded(B, Hq, Hkv, 1, K, D, Dv, "f32", seed=12)
    c = 300
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    o1, l1 = attn_fwd(q, k, v, seqlens_k=torch.full((B,), c, dtype=torch.int32, device="cuda"),
                      algo="generic")
    o2, l2 = attn_fwd(q, k, v, window=K - c, algo="generic")
    parts_o = torch.stack([o1.reshape(-1, Dv), o2.reshape(-1, Dv)]).contiguous()
    parts_l = torch.stack([l1.reshape(-1), l2.reshape(-1)]).contiguous()
    o, lse = attn_lse_combine(parts_o, parts_l, dtype=torch.float32)
    ro, rl = parity.run_oracle(inp)
    parity.compare("f32", o.cpu().numpy(), lse.cpu().numpy(), ro.reshape(-1, Dv),
                   rl.reshape(-1), "combine")
    # all partials empty -> +0 / -inf
    e_o = torch.zeros((3, 4, 16), device="cuda")
    e_l = torch.full((3, 4), -math.inf, device="cuda")
    o, lse = attn_lse_combine(e_o, e_l, dtype=torch.bfloat16)
    assert torch.all(o.float() == 0) and not torch.any(torch.signbit(o.float()))
    assert torch.all(lse == -math.inf)


def test_unsupported_algo_reports():
    inp = synth.make_padded(1, 4, 2, 8, 8, 16, 16, "f32", seed=1)
    with pytest.raises(AttnError) as ei:
        attn_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), algo="tcgen05")
    assert ei.value.status == 2


# ---------------------------------------------------------------------------
# split-KV tensor-core decode

DECODE_SHAPES = [
    # B, Hq, Hkv, Q, K, D, Dv
    (8, 32, 8, 1, 1024, 128, 128),
    (3, 16, 2, 1, 700, 64, 64),      # G = 8
    (2, 16, 1, 1, 333, 128, 64),     # MQA, G = 16 (two n-tiles)
    (2, 8, 8, 1, 257, 64, 128),      # MHA
    (2, 8, 2, 2, 300, 128, 128),     # two query rows per sequence (causal offset)
    (1, 16, 4, 4, 129, 128, 128),    # Q*G = 16
    (1, 8, 2, 1, 32768, 64, 64),     # long KV: many splits
    (1, 16, 4, 1, 8193, 128, 128),
    # head dim 256 (one block an SM)
    (4, 16, 4, 1, 1000, 256, 256),
    (2, 16, 1, 1, 700, 256, 256),    # G = 16: two n-tiles
    # many (sequence, KV head) units, as in batched serving
    (40, 16, 1, 1, 333, 128, 64),
    (20, 8, 2, 2, 300, 128, 128),
    (10, 16, 4, 4, 129, 64, 128),
    (48, 16, 2, 1, 700, 64, 64),
    (38, 8, 1, 1, 5000, 128, 128),
]


@pytest.mark.parametrize("shape", DECODE_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_decode_shapes(shape, dtype):
    B, Hq, Hkv, Q, K, D, Dv = shape
    g = np.random.default_rng(B * 131 + K)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=21, seqlens_k=sk, pad_value=NAN)
    parity.check(inp, "decode", f"decode {dtype} {shape}")


@pytest.mark.parametrize("window", [1, 100, 1000])
def test_decode_window(window):
    sk = np.array([0, 5, 999, 1000, 2500], np.int32)
    inp = synth.make_padded(5, 32, 8, 1, 2500, 128, 128, "bf16", seed=22, seqlens_k=sk,
                            window=window, pad_value=NAN)
    parity.check(inp, "decode", f"decode window {window}")


def test_decode_reduction_lengths():
    sk = np.array([0, 1, 7, 16, 31, 32, 33, 63, 64, 65, 127, 128, 129, 511, 512, 513], np.int32)
    inp = synth.make_padded(16, 8, 2, 1, 600, 128, 128, "bf16", seed=23, seqlens_k=sk,
                            pad_value=NAN)
    parity.check(inp, "decode", "decode lengths")


def test_decode_padded_query_rows():
    # Q capacity 2 with Qb = 1 or 0: padded rows must be +0 / -inf
    inp = synth.make_padded(3, 8, 2, 2, 200, 64, 64, "bf16", seed=24, seqlens_q=[1, 0, 2],
                            seqlens_k=[200, 50, 0], pad_value=NAN)
    parity.check(inp, "decode", "decode padded rows")


def test_decode_varlen_packed():
    sk = np.array([0, 1, 300, 4097, 64], np.int32)
    sq = np.array([0, 1, 1, 1, 1], np.int32)
    inp = synth.make_packed(sq, sk, 32, 8, 128, 128, "bf16", seed=25)
    parity.check(inp, "decode", "decode packed")


def test_decode_full_size_batched():
    """bf16 batched decode B=64 Hq=32 Hkv=8 D=Dv=128, key lengths uniform on
    [0, 8192], KV padded to 8192 (NaN in the padding): every row checked."""
    inp = synth.decode_bf16_b64_h32x8_k8192_d128(pad_value=NAN)
    o, lse = parity.run_gpu(inp, "auto")
    rows = np.array([(b, 0, h) for b in range(inp.B) for h in range(inp.Hq)], np.int32)
    parity.check_sampled_padded(inp, o, lse, rows, "decode full size")


# ---------------------------------------------------------------------------
# tcgen05 / TMEM prefill

TC_SHAPES = [
    # B, Hq, Hkv, Q, K, D, Dv
    (1, 4, 2, 64, 128, 64, 64),       # the fp32 prefill shape, in bf16
    (1, 4, 2, 65, 131, 64, 64),       # Q/K tails
    (1, 8, 2, 256, 1024, 64, 64),
    (2, 8, 2, 300, 300, 128, 128),
    (1, 4, 1, 129, 129, 128, 64),     # MQA, G = 4
    (1, 2, 2, 200, 200, 64, 128),     # MHA: one head per row block
    (2, 32, 8, 512, 512, 128, 128),   # G = 4 as in the 4096^2 workload
    (1, 16, 2, 100, 357, 128, 128),   # G = 8
    (1, 32, 2, 70, 70, 64, 64),       # G = 16
    (1, 6, 2, 90, 150, 128, 128),     # G = 3: three subgroups of one head
    (1, 8, 2, 3, 67, 128, 128),       # short query chunk, bottom-right offset
    (1, 4, 2, 300, 40, 64, 64),       # Q > K: leading rows without keys
    # head dims between the tile widths: zero-filled tile columns
    (1, 8, 2, 200, 260, 80, 80),
    (1, 8, 2, 130, 130, 96, 96),
    (2, 8, 4, 100, 300, 112, 64),     # G = 2
    (1, 4, 2, 150, 150, 64, 96),
    (1, 4, 1, 77, 200, 96, 128),
]


@pytest.mark.parametrize("shape", TC_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tcgen05_shapes(shape, dtype):
    B, Hq, Hkv, Q, K, D, Dv = shape
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=31)
    parity.check(inp, "tcgen05", f"tcgen05 {dtype} {shape}")


@pytest.mark.parametrize("window", [1, 50, 128, 129, 1000])
def test_tcgen05_window(window):
    inp = synth.make_padded(2, 8, 2, 400, 700, 128, 128, "bf16", seed=32, window=window)
    parity.check(inp, "tcgen05", f"tcgen05 window {window}")


def test_tcgen05_lengths_nan_padding():
    sq = np.array([0, 1, 7, 16, 31, 32, 33, 65, 200, 130], np.int32)
    sk = np.array([0, 1, 7, 16, 31, 32, 33, 65, 250, 129], np.int32)
    inp = synth.make_padded(10, 8, 2, 200, 250, 128, 128, "bf16", seed=33, seqlens_q=sq,
                            seqlens_k=sk, pad_value=NAN)
    parity.check(inp, "tcgen05", "tcgen05 lengths")


def test_tcgen05_all_empty():
    inp = synth.make_padded(2, 8, 2, 64, 64, 128, 128, "bf16", seed=34,
                            seqlens_k=np.zeros(2, np.int32), pad_value=NAN)
    parity.check(inp, "tcgen05", "tcgen05 all empty")


def test_tcgen05_negative_scale():
    inp = synth.make_padded(1, 4, 2, 130, 130, 64, 64, "bf16", seed=35, scale=-0.2)
    parity.check(inp, "tcgen05", "tcgen05 negative scale")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("dims", [(128, 128), (96, 80)], ids=lambda d: f"d{d[0]}x{d[1]}")
def test_tcgen05_varlen_packed(dtype, dims):
    sk = np.array([0, 5, 33, 130, 1, 640, 0, 300, 1000], np.int32)
    sq = np.minimum(sk, np.array([0, 5, 7, 64, 1, 512, 0, 100, 512]))
    for w in (0, 100):
        inp = synth.make_packed(sq, sk, 16, 4, dims[0], dims[1], dtype, seed=36, window=w)
        parity.check(inp, "tcgen05", f"tcgen05 varlen {dtype} {dims} w={w}")


def test_tcgen05_full_size_prefill_every_row():
    """bf16 causal prefill B=4 Hq=32 Hkv=8 Q=K=4096 D=Dv=128, the benchmark's
    launch and seed: all 524,288 output rows against the fp64 oracle (about
    0.55 TFLOP of fp64 work, seconds on the host's cores)."""
    inp = synth.prefill_bf16_b4_h32x8_s4096_d128(seed=1234)
    parity.check(inp, "auto", "prefill full size, every row")


def test_tcgen05_full_size_prefill_second_seed_sampled():
    """The same launch on a second seed: sampled rows against the oracle, and
    row 0 of every (sequence, head), which sees exactly key 0, equals V[0]."""
    inp = synth.prefill_bf16_b4_h32x8_s4096_d128(seed=4321)
    o, lse = parity.run_gpu(inp, "auto")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    rows = parity.sample_rows(inp, 3000, seed=4)
    parity.check_sampled_padded(inp, o, lse, rows, "prefill full size, seed 4321")
    v0 = synth.exact_f32(inp.v[:, 0])            # [B, Hkv, Dv]
    G = inp.Hq // inp.Hkv
    want = np.repeat(v0, G, axis=1)             # [B, Hq, Dv]
    assert np.max(np.abs(o[:, 0] - want)) <= 2e-2


def test_tcgen05_full_size_varlen():
    """bf16 varlen chunked prefill: 16 packed sequences, key lengths U[0,4096]
    incl. empty, queries = last min(512, Kb) tokens, Hq=16 Hkv=4, window 1024:
    every row against the oracle."""
    inp = synth.varlen_bf16_16seq_h16x4_k4096_q512_w1024()
    parity.check(inp, "auto", "varlen full size")


# ---------------------------------------------------------------------------
# the two masks beyond the pages' bottom-right rule: top-left causal, none

MASK_SHAPES = [
    # algo, dtype, B, Hq, Hkv, Q, K, D, Dv, window
    ("generic", "f32", 2, 4, 2, 70, 150, 64, 48, 0),
    ("generic", "f32", 1, 8, 2, 130, 60, 32, 32, 9),    # Q > K
    ("tcgen05", "bf16", 2, 8, 2, 300, 500, 128, 128, 0),
    ("tcgen05", "f16", 1, 8, 2, 500, 300, 64, 64, 0),   # Q > K
    ("tcgen05", "bf16", 1, 8, 4, 257, 400, 128, 64, 100),
    ("decode", "bf16", 8, 32, 8, 1, 1500, 128, 128, 0),
    ("decode", "bf16", 4, 16, 4, 4, 900, 64, 64, 0),    # Q*G = 16
]


@pytest.mark.parametrize("mask", [1, 2], ids=["top_left", "none"])
@pytest.mark.parametrize("case", MASK_SHAPES, ids=lambda c: f"{c[0]}-{c[1]}-" + "x".join(map(str, c[2:])))
def test_masks(case, mask):
    algo, dtype, B, Hq, Hkv, Q, K, D, Dv, window = case
    if mask == 2:
        window = 0
    g = np.random.default_rng(B * 31 + K + mask)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=51, seqlens_k=sk,
                            window=window, pad_value=NAN)
    parity.check(inp, algo, f"mask {mask} {case}", mask=mask)


@pytest.mark.parametrize("mask", [1, 2], ids=["top_left", "none"])
def test_masks_varlen_packed(mask):
    sk = np.array([0, 5, 33, 130, 1, 640, 0, 300, 1000], np.int32)
    sq = np.minimum(sk + 20, np.array([0, 5, 7, 64, 1, 512, 0, 100, 512]) + 20)
    inp = synth.make_packed(sq, sk, 16, 4, 128, 128, "bf16", seed=52)
    for algo in ("tcgen05", "generic"):
        parity.check(inp, algo, f"mask {mask} varlen {algo}", mask=mask)


def test_mask_none_rejects_window():
    inp = synth.make_padded(1, 4, 2, 8, 8, 64, 64, "bf16", seed=53)
    with pytest.raises(AttnError) as ei:
        attn_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), window=3, mask="none")
    assert ei.value.status == 1


# mma.sync forward: head widths above the tcgen05 kernel's (up to 256), and
# the narrower widths it also takes when chosen explicitly
MMA_SHAPES = [
    # B, Hq, Hkv, Q, K, D, Dv
    (2, 8, 2, 200, 200, 256, 256),
    (1, 8, 2, 130, 330, 256, 256),    # Q < K: bottom-right offset
    (1, 4, 2, 300, 40, 256, 256),     # Q > K: leading rows without keys
    (1, 16, 2, 100, 357, 192, 160),   # G = 8, padded tile columns
    (1, 4, 4, 77, 200, 136, 256),     # MHA, D just above 128
    (2, 6, 2, 90, 150, 256, 64),
    (1, 8, 2, 3, 67, 256, 256),       # short query chunk
    (2, 8, 2, 150, 150, 128, 128),
    (1, 4, 1, 65, 131, 64, 64),
    (1, 8, 4, 1, 700, 256, 256),      # one query row
    # wide heads: warp pairs split the width
    (1, 8, 2, 130, 200, 512, 512),
    (2, 4, 2, 90, 150, 320, 512),
    (1, 4, 1, 70, 70, 512, 64),
    (1, 8, 2, 100, 300, 128, 512),
    (1, 6, 2, 40, 100, 264, 200),
]


@pytest.mark.parametrize("shape", MMA_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_mma_forward_shapes(shape, dtype):
    B, Hq, Hkv, Q, K, D, Dv = shape
    g = np.random.default_rng(Q + K)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=37, seqlens_k=sk, pad_value=NAN)
    parity.check(inp, "mma", f"mma {dtype} {shape}")


@pytest.mark.parametrize("window", [1, 50, 129])
@pytest.mark.parametrize("mask", [0, 1, 2])
@pytest.mark.parametrize("width", [256, 512])
def test_mma_forward_window_and_masks(window, mask, width):
    if mask == 2:
        window = 0
    inp = synth.make_padded(2, 8, 2, 180, 260, width, width, "bf16", seed=38, window=window)
    parity.check(inp, "mma", f"mma window {window} mask {mask} width {width}", mask=mask)


def test_mma_forward_varlen_packed_and_auto_choice():
    sk = np.array([0, 5, 33, 130, 1, 640, 0, 300], np.int32)
    sq = np.minimum(sk, np.array([0, 5, 7, 64, 1, 512, 0, 100]))
    for w in (0, 100):
        inp = synth.make_packed(sq, sk, 16, 4, 256, 256, "bf16", seed=39, window=w)
        parity.check(inp, "auto", f"auto (tcgen05 wide) varlen w={w}")


def test_mma_forward_rejects_fp32_and_wide_heads():
    inp = synth.make_padded(1, 2, 1, 8, 8, 64, 64, "f32", seed=40)
    with pytest.raises(AttnError) as ei:
        parity.run_gpu(inp, "mma")
    assert ei.value.status == 2
    inp = synth.make_padded(1, 2, 1, 8, 8, 256, 250, "bf16", seed=40)
    with pytest.raises(AttnError) as ei:
        parity.run_gpu(inp, "mma")
    assert ei.value.status == 2


# head widths above 256 (up to 512): the CUDA-core kernel (every dtype) and
# the mma.sync kernel (bf16 / fp16, the automatic choice)
@pytest.mark.parametrize("dtype,dims", [("f32", (512, 512)), ("bf16", (320, 512)),
                                        ("f16", (512, 264))])
def test_wide_heads_cuda_cores(dtype, dims):
    D, Dv = dims
    sk = np.array([90, 0, 33], np.int32)
    inp = synth.make_padded(3, 4, 2, 70, 90, D, Dv, dtype, seed=41, seqlens_k=sk, pad_value=NAN)
    parity.check(inp, "generic", f"wide heads {dtype} {dims}")
    inp = synth.make_padded(1, 8, 2, 1, 3000, D, Dv, dtype, seed=42, window=700)
    parity.check(inp, "generic", f"wide heads decode {dtype} {dims}")
    if dtype != "f32":
        parity.check(inp, "auto", f"wide heads decode, auto (mma) {dtype} {dims}")


def test_wide_heads_rejected_above_512_and_by_tensor_kernels():
    inp = synth.make_padded(1, 2, 1, 8, 8, 520, 64, "bf16", seed=43)
    with pytest.raises(AttnError) as ei:
        parity.run_gpu(inp, "auto")
    assert ei.value.status == 1
    # tcgen05 takes widths that are multiples of 16 up to 512; the decode
    # kernel D = Dv in {64, 128, 256}
    for shape, algo in (((504, 504), "tcgen05"), ((512, 512), "decode")):
        inp = synth.make_padded(1, 2, 1, 8, 8, *shape, "bf16", seed=43)
        with pytest.raises(AttnError) as ei:
            parity.run_gpu(inp, algo)
        assert ei.value.status == 2
