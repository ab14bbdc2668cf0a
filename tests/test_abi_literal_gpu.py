"""The two primary C symbols themselves, attn_fwd (padded layout) and
attn_fwd_varlen (packed layout), called through ctypes with raw device
pointers exactly as a C caller would -- not through the binding's *_ex route --
and compared with the fp64 oracle on the same seeded inputs."""
import ctypes

import numpy as np
import pytest
import torch

import causal_gqa_attention_online_gb300 as attn
from causal_gqa_attention_online_gb300 import build_ext, synth
from tests import parity

pytestmark = pytest.mark.gpu

NAN = float("nan")
DT = {"f32": attn.ATTN_F32, "f16": attn.ATTN_F16, "bf16": attn.ATTN_BF16}


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return attn.load_library()


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("case", [
    # dtype, B, Hq, Hkv, Q, K, D, Dv, window
    ("bf16", 3, 8, 2, 200, 333, 128, 128, 0),     # tcgen05 prefill
    ("f16", 2, 16, 4, 1, 3000, 128, 128, 500),    # split-KV decode
    ("f32", 1, 4, 2, 64, 128, 64, 64, 0),         # CUDA-core kernel
], ids=lambda c: "-".join(map(str, c)))
def test_attn_fwd_symbol(lib, case):
    dtype, B, Hq, Hkv, Q, K, D, Dv, window = case
    g = np.random.default_rng(B + K)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    sq = np.minimum(g.integers(0, Q + 1, size=B), Q).astype(np.int32)
    sq[0] = Q
    inp = synth.make_padded(B, Hq, Hkv, Q, K, D, Dv, dtype, seed=61, seqlens_q=sq, seqlens_k=sk,
                            window=window, pad_value=NAN)
    dev = torch.device("cuda")
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    dsq, dsk = torch.from_numpy(sq).to(dev), torch.from_numpy(sk).to(dev)
    o = torch.full((B, Q, Hq, Dv), NAN, dtype=q.dtype, device=dev)
    lse = torch.full((B, Q, Hq), NAN, dtype=torch.float32, device=dev)
    rc = lib.attn_fwd(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), B,
                      Hq, Hkv, Q, K, D, Dv, _vp(dsq), _vp(dsk), window, ctypes.c_float(inp.scale),
                      DT[dtype], _stream())
    assert rc == 0, lib.attn_last_error().decode()
    torch.cuda.synchronize()
    ro, rl = parity.run_oracle(inp)
    parity.compare(dtype, o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl, "attn_fwd symbol")


def test_attn_fwd_varlen_symbol(lib):
    sk = np.array([0, 5, 700, 1500, 64, 0, 1024], np.int32)
    sq = np.minimum(sk, 512).astype(np.int32)
    inp = synth.make_packed(sq, sk, 16, 4, 128, 128, "bf16", seed=62, window=300)
    dev = torch.device("cuda")
    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    cq = torch.from_numpy(inp.cu_seqlens_q).to(dev)
    ck = torch.from_numpy(inp.cu_seqlens_k).to(dev)
    Tq, Tk = int(inp.cu_seqlens_q[-1]), int(inp.cu_seqlens_k[-1])
    o = torch.full((Tq, 16, 128), NAN, dtype=q.dtype, device=dev)
    lse = torch.full((Tq, 16), NAN, dtype=torch.float32, device=dev)
    rc = lib.attn_fwd_varlen(_vp(q), _vp(k), _vp(v), _vp(o), _vp(lse), len(sk), 16, 4, Tq, Tk,
                             int(sq.max()), int(sk.max()), 128, 128, _vp(cq), _vp(ck), 300,
                             ctypes.c_float(inp.scale), attn.ATTN_BF16, _stream())
    assert rc == 0, lib.attn_last_error().decode()
    torch.cuda.synchronize()
    ro, rl = parity.run_oracle(inp)
    parity.compare("bf16", o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl,
                   "attn_fwd_varlen symbol")
