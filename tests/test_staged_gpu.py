"""attn_fwd_staged: attention on host tensors, copies overlapped with the
attention of other groups of sequences.  Parity against the oracle, and the
prefill result bit-identical to attn_fwd on the same inputs (a group's
launch computes exactly what the whole batch's launch computes for it)."""
import numpy as np
import pytest
import torch

from tests import parity
from causal_gqa_attention_online_gb300 import attn_fwd, attn_fwd_staged, synth

pytestmark = pytest.mark.gpu
NAN = float("nan")


def _staged(inp, chunks, fill=NAN):
    dev = torch.device("cuda")
    hq, hk, hv = inp.q.pin_memory(), inp.k.pin_memory(), inp.v.pin_memory()
    # device staging buffers start as NaN: rows the call does not copy in must
    # never be read
    q = torch.full(inp.q.shape, fill, dtype=inp.q.dtype, device=dev)
    k = torch.full(inp.k.shape, fill, dtype=inp.k.dtype, device=dev)
    v = torch.full(inp.v.shape, fill, dtype=inp.v.dtype, device=dev)
    o = torch.full((inp.B, inp.Q, inp.Hq, inp.Dv), fill, dtype=inp.q.dtype, device=dev)
    lse = torch.full((inp.B, inp.Q, inp.Hq), fill, dtype=torch.float32, device=dev)
    sq = None if inp.seqlens_q is None else torch.from_numpy(inp.seqlens_q)
    sk = None if inp.seqlens_k is None else torch.from_numpy(inp.seqlens_k)
    ho, hl, bin_, bout = attn_fwd_staged(hq, hk, hv, q, k, v, o, lse, seqlens_q=sq, seqlens_k=sk,
                                         window=inp.window, scale=inp.scale, chunks=chunks)
    torch.cuda.current_stream().synchronize()
    return ho, hl, bin_, bout


def _expected_bytes(inp):
    es = inp.q.element_size()
    qb = np.full(inp.B, inp.Q) if inp.seqlens_q is None else np.clip(inp.seqlens_q, 0, inp.Q)
    kb = np.full(inp.B, inp.K) if inp.seqlens_k is None else np.clip(inp.seqlens_k, 0, inp.K)
    bin_ = int(qb.sum()) * inp.Hq * inp.D * es + int(kb.sum()) * inp.Hkv * (inp.D + inp.Dv) * es
    bout = inp.B * inp.Q * inp.Hq * (inp.Dv * es + 4)
    return bin_, bout


@pytest.mark.parametrize("chunks", [1, 3, 0, 100])
def test_staged_prefill_matches_attn_fwd_bitwise(chunks):
    sk = np.array([200, 0, 57, 200, 131], np.int32)
    inp = synth.make_padded(5, 8, 2, 200, 200, 128, 128, "bf16", seed=41, seqlens_k=sk,
                            seqlens_q=sk, pad_value=NAN)
    ho, hl, bin_, bout = _staged(inp, chunks)
    dev = torch.device("cuda")
    ro, rl = attn_fwd(inp.q.to(dev), inp.k.to(dev), inp.v.to(dev),
                      seqlens_q=torch.from_numpy(sk).to(dev), seqlens_k=torch.from_numpy(sk).to(dev),
                      window=inp.window, scale=inp.scale)
    torch.cuda.synchronize()
    assert torch.equal(parity._bits(ho), parity._bits(ro.cpu()))
    assert torch.equal(parity._bits(hl), parity._bits(rl.cpu()))
    ro_, rl_ = parity.run_oracle(inp)
    parity.compare("bf16", ho.float().numpy(), hl.numpy(), ro_, rl_, f"staged prefill {chunks}")
    assert (bin_, bout) == _expected_bytes(inp)


def test_staged_decode_ragged_keys():
    g = np.random.default_rng(5)
    sk = g.integers(0, 3000, size=24).astype(np.int32)
    sk[0], sk[1] = 3000, 0
    inp = synth.make_padded(24, 32, 8, 1, 3000, 128, 128, "bf16", seed=42, seqlens_k=sk,
                            pad_value=NAN)
    ho, hl, bin_, bout = _staged(inp, 4)
    ro, rl = parity.run_oracle(inp)
    parity.compare("bf16", ho.float().numpy(), hl.numpy(), ro, rl, "staged decode")
    assert (bin_, bout) == _expected_bytes(inp)


def test_staged_fp32_window():
    inp = synth.make_padded(3, 4, 2, 70, 90, 64, 48, "f32", seed=43, window=17)
    ho, hl, _, _ = _staged(inp, 2)
    ro, rl = parity.run_oracle(inp)
    parity.compare("f32", ho.numpy(), hl.numpy(), ro, rl, "staged fp32")
