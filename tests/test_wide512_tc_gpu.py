"""GPU parity of the tcgen05 prefill for head widths above 256 (up to 512):
the output columns in halves of 256, each half of a Q tile a work unit of
its own that recomputes the scores, K streamed through the shared-memory ring
two 64-column chunks a slot and V 64 keys a slot -- against the fp64 oracle on
the same seeded inputs (tolerances in tests/parity.py).

Cases: square, Q < K and Q > K problems, D just above 256 (five K chunks),
D below 256 with Dv above, a second output half narrower than 256 (64, 144
columns) and one half only (Dv <= 256), a single query row, GQA packing
G = 1..8, windows, the three mask modes, ragged sequences with NaN padding
(V rows past the last key zeroed in the last 64-key slot), the packed layout
with empty sequences, scores that grow by more than 2^8 from tile to tile
(the O rescale), fp16, and the benchmark's D = 512 launch on every row."""
import numpy as np
import pytest

from causal_gqa_attention_online_gb300 import build_ext, synth
from tests import parity

pytestmark = pytest.mark.gpu

NAN = float("nan")


@pytest.fixture(scope="module", autouse=True)
def built():
    build_ext.build()


SHAPES = [
    # B, Hq, Hkv, Q, K, D, Dv
    (2, 8, 2, 200, 200, 512, 512),
    (1, 8, 2, 130, 330, 512, 512),    # Q < K: bottom-right offset
    (1, 4, 2, 300, 40, 512, 512),     # Q > K: leading rows without keys
    (1, 16, 2, 100, 357, 448, 320),   # G = 8, second half 64 columns wide
    (1, 4, 4, 77, 200, 272, 512),     # MHA, D just above 256
    (2, 6, 2, 90, 150, 512, 64),      # one output half, narrow
    (1, 8, 2, 100, 300, 128, 512),    # narrow D, wide Dv
    (1, 8, 2, 200, 300, 512, 400),    # second half 144 columns wide
    (1, 8, 2, 3, 67, 512, 512),       # short query chunk
    (1, 8, 4, 1, 700, 512, 512),      # one query row
    (3, 16, 4, 513, 1100, 512, 512),  # many tiles a unit, ragged last tile
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_wide512_tc_shapes(shape, dtype):
    B, Hq, Hkv, Q, K, D, Dv = shape
    g = np.random.default_rng(Q + K + D + Dv)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    sq = g.integers(0, Q + 1, size=B).astype(np.int32)
    sq[0] = Q
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=57, seqlens_q=sq, seqlens_k=sk,
                            pad_value=NAN)
    parity.check(inp, "tcgen05", f"wide512 tc {dtype} {shape}")


@pytest.mark.parametrize("window", [1, 50, 129, 300])
@pytest.mark.parametrize("mask", [0, 1, 2])
def test_wide512_tc_window_and_masks(window, mask):
    if mask == 2:
        window = 0
    inp = synth.make_padded(2, 8, 2, 380, 460, 512, 512, "bf16", seed=58, window=window)
    parity.check(inp, "tcgen05", f"wide512 tc window {window} mask {mask}", mask=mask)


def test_wide512_tc_varlen_packed():
    sk = np.array([0, 5, 33, 130, 1, 640, 0, 300], np.int32)
    sq = np.minimum(sk, np.array([0, 5, 7, 64, 1, 512, 0, 100]))
    for w in (0, 100):
        inp = synth.make_packed(sq, sk, 16, 4, 512, 512, "bf16", seed=59, window=w)
        parity.check(inp, "auto", f"wide512 tc varlen w={w}")


def test_wide512_tc_growing_scores_rescale_o():
    """Scores rise by 10 (natural units) per 128-key tile, so the running max
    grows by more than 2^8 at every tile and both output halves rescale O
    (after the previous tile's PV)."""
    import torch
    B, Hq, Hkv, Q, K, D = 1, 4, 2, 128, 1024, 512
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, D, "bf16", seed=60, scale=1.0)
    q = torch.zeros_like(inp.q)
    q[..., :16] = 1.0
    k = torch.zeros_like(inp.k)
    steps = (torch.arange(K) // 128).to(torch.float32) * (10.0 / 16)
    k[0, :, :, :16] = steps[:, None, None].to(k.dtype)
    inp.q.copy_(q)
    inp.k.copy_(k)
    parity.check(inp, "tcgen05", "wide512 tc growing scores")


def test_wide512_tc_full_size_every_row():
    """bf16 causal prefill B=1 Hq=16 Hkv=4 Q=K=4096 D=Dv=512 (the benchmark's
    512-wide launch): every row against the oracle."""
    inp = synth.make_padded(1, 16, 4, 4096, 4096, 512, 512, "bf16", seed=778)
    parity.check(inp, "auto", "wide512 tc 4096^2 D=512")
