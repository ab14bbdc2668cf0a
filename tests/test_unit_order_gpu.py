"""GPU parity of the tcgen05 prefill's longest-first unit order on larger
ragged problems.

A work unit is 128 rows of one (sequence, query block, KV head, head subgroup).
On a ragged problem a one-block order launch ahead of the prefill sorts the
units by KV tile count, most first (a counting sort), and the persistent CTAs
take them in alternating rounds from that order.  Cases with many classes of
equal tile count, many rounds a CTA (up to ~70 on 152 SMs), in the packed and
the padded layouts, every output row against the fp64 oracle: a unit lost or
taken twice leaves NaN canaries or wrong rows behind.  Two launches a call
(the order, then the prefill)."""
import numpy as np
import pytest

from causal_gqa_attention_online_gb300 import binding, build_ext, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build_ext.build()


def _check(inp, what):
    n0 = binding.kernel_launches()
    o, lse = parity.run_gpu(inp, "tcgen05")
    got = binding.kernel_launches() - n0
    ro, rl = parity.run_oracle(inp)
    parity.compare(inp.dtype, o, lse, ro, rl, what)
    assert got == 2, f"{what}: {got} launches, expected the order and the prefill"


@pytest.mark.parametrize("B", [200, 210])
def test_packed_many_sequences(B):
    """G = 4 packs 4 heads x 32 positions a tile (64 query positions a unit);
    query chunks up to 320 of keys up to 640: 1000 and 1050 units."""
    g = np.random.default_rng(B)
    sk = g.integers(0, 641, size=B).astype(np.int32)
    sk[0] = 640
    sq = np.minimum(sk, g.integers(0, 321, size=B)).astype(np.int32)
    sq[0] = 320
    inp = synth.make_packed(sq, sk, 4, 1, 64, 64, "bf16", seed=61, window=0)
    _check(inp, f"packed {B} sequences")


@pytest.mark.parametrize("Hkv", [16, 32])
def test_padded_many_rounds(Hkv):
    """G = 2 packs 2 heads x 64 positions a tile (128 positions a unit);
    80 sequences, Q = K = 512 ragged, Hkv units a (sequence, query block):
    5120 and 10240 units, 34 and 68 rounds a CTA on 152 SMs."""
    B, Q, K = 80, 512, 512
    g = np.random.default_rng(Hkv)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    sq = np.minimum(sk, g.integers(0, Q + 1, size=B)).astype(np.int32)
    sq[0] = Q
    inp = synth.make_padded(B, 2 * Hkv, Hkv, Q, K, 64, 64, "bf16", seed=62, seqlens_q=sq,
                            seqlens_k=sk, pad_value=float("nan"))
    _check(inp, f"padded Hkv={Hkv}")


def test_packed_window_one_unit_per_sequence():
    """Short chunks (one query block a sequence), a window, fp16, G = 8 (8
    heads x 16 positions a tile): many units of equal tile count."""
    g = np.random.default_rng(63)
    sk = g.integers(0, 900, size=300).astype(np.int32)
    sq = np.minimum(sk, g.integers(0, 33, size=300)).astype(np.int32)
    inp = synth.make_packed(sq, sk, 16, 2, 128, 128, "f16", seed=64, window=200)
    _check(inp, "packed 300 sequences, window 200")
