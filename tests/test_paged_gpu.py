"""attn_fwd_paged: keys and values in pages addressed by a block table.  A
paged problem is laid out from a padded one (pages shuffled, unused pages and
the tail of the last page of each sequence NaN), so the oracle's answer is the
padded problem's; where the kernels walk the same tiles, the result is also
bit-identical to attn_fwd on the padded layout."""
import numpy as np
import pytest
import torch

from tests import parity
from causal_gqa_attention_online_gb300 import attn_fwd, attn_fwd_paged, synth

pytestmark = pytest.mark.gpu
NAN = float("nan")


def paginate(inp, page, seed, spare=3):
    """Pools [P, page, Hkv, D|Dv] and a block table [B, max_pages] holding the
    padded problem's K / V: page j of sequence b is a random physical page."""
    B, K = inp.B, inp.K
    max_pages = (K + page - 1) // page
    P = B * max_pages + spare
    g = np.random.default_rng(seed)
    perm = g.permutation(P)[: B * max_pages].reshape(B, max_pages).astype(np.int32)
    kp = torch.full((P, page, inp.Hkv, inp.D), NAN, dtype=inp.k.dtype)
    vp = torch.full((P, page, inp.Hkv, inp.Dv), NAN, dtype=inp.v.dtype)
    kb = np.full(B, K) if inp.seqlens_k is None else np.clip(inp.seqlens_k, 0, K)
    for b in range(B):
        for j in range(max_pages):
            lo, hi = j * page, min((j + 1) * page, int(kb[b]))
            if hi > lo:
                kp[perm[b, j], : hi - lo] = inp.k[b, lo:hi]
                vp[perm[b, j], : hi - lo] = inp.v[b, lo:hi]
    return kp, vp, torch.from_numpy(perm), kb.astype(np.int32)


def run_paged(inp, page, algo, mask=0, seed=0):
    dev = torch.device("cuda")
    kp, vp, table, kb = paginate(inp, page, seed)
    o = torch.full((inp.B, inp.Q, inp.Hq, inp.Dv), NAN, dtype=inp.q.dtype, device=dev)
    lse = torch.full((inp.B, inp.Q, inp.Hq), NAN, dtype=torch.float32, device=dev)
    sq = None if inp.seqlens_q is None else torch.from_numpy(inp.seqlens_q).to(dev)
    attn_fwd_paged(inp.q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), torch.from_numpy(kb).to(dev),
                   o, lse, seqlens_q=sq, window=inp.window, scale=inp.scale, algo=algo,
                   mask=parity.MASK_NAMES[mask])
    torch.cuda.synchronize()
    return o, lse


CASES = [
    # algo, dtype, B, Hq, Hkv, Q, K, D, Dv, page, window, mask
    ("decode", "bf16", 8, 32, 8, 1, 1000, 128, 128, 16, 0, 0),
    ("decode", "f16", 6, 16, 2, 1, 700, 64, 64, 64, 0, 0),
    ("decode", "bf16", 4, 16, 4, 4, 900, 128, 128, 32, 100, 0),
    ("tcgen05", "bf16", 2, 8, 2, 300, 300, 128, 128, 128, 0, 0),
    ("tcgen05", "bf16", 2, 8, 2, 200, 700, 128, 128, 256, 150, 0),
    ("tcgen05", "f16", 1, 8, 4, 260, 400, 64, 64, 128, 0, 1),
    ("mma", "bf16", 2, 8, 2, 120, 300, 256, 256, 16, 0, 0),
    ("mma", "f16", 1, 4, 2, 70, 200, 512, 512, 64, 40, 0),
    ("generic", "f32", 2, 4, 2, 50, 90, 64, 48, 32, 0, 0),
    ("generic", "f32", 2, 4, 2, 50, 90, 32, 32, 8, 11, 0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}-" + "x".join(map(str, c[2:])))
def test_paged_parity(case):
    algo, dtype, B, Hq, Hkv, Q, K, D, Dv, page, window, mask = case
    g = np.random.default_rng(B * 7 + K)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=61, seqlens_k=sk, window=window,
                            pad_value=NAN)
    o, lse = run_paged(inp, page, algo, mask, seed=B + K)
    ro, rl = parity.run_oracle(inp, mask=mask)
    parity.compare(dtype, o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, f"paged {case}")
    if window == 0:
        # same tiles as the padded layout: the same bits
        dev = torch.device("cuda")
        po, pl = attn_fwd(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev),
                          seqlens_k=torch.from_numpy(sk).to(dev), scale=inp.scale, algo=algo,
                          mask=parity.MASK_NAMES[mask])
        torch.cuda.synchronize()
        assert torch.equal(parity._bits(o), parity._bits(po))
        assert torch.equal(parity._bits(lse), parity._bits(pl))


def test_paged_prefill_rejects_small_pages_on_tcgen05():
    from causal_gqa_attention_online_gb300 import AttnError
    inp = synth.make_padded(1, 4, 2, 130, 130, 64, 64, "bf16", seed=62)
    with pytest.raises(AttnError) as ei:
        run_paged(inp, 64, "tcgen05")
    assert ei.value.status == 2
