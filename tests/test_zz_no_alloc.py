"""attn_fwd_decode_noalloc: the split-KV decode for callers that may not
allocate device memory while attention runs (a process whose device memory is
owned by another runtime's allocator or held under a hard cap, or a
latency-critical decode loop).  Its partial results live in the library's
fixed device array instead of coming from an allocator.

Calls go through the C ABI, several in a row on different problems, and each
result is checked twice within the tolerances of the other parity tests:
against the fp64 CPU oracle on the same inputs, and against attn_fwd (the
allocating entry point).  Between two checked calls a larger problem fills the
array with unrelated partials, so a result that read stale scratch would show.
The checked calls must not change the device's free memory.  The cases cover
bf16 and fp16, a sliding window, empty and full sequences, NaN in the padding,
and a short problem that needs no scratch at all (one split).  The file is
collected last and needs nothing from the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import causal_gqa_attention_online_gb300 as attn
from causal_gqa_attention_online_gb300 import build_ext, synth
from tests import parity

pytestmark = pytest.mark.gpu

DT = {"bf16": attn.ATTN_BF16, "f16": attn.ATTN_F16}


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return attn.load_library()


def _problem(seed, B, K, dtype="bf16", window=0):
    g = np.random.default_rng(seed)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    sk[1] = 0
    return synth.make_padded(B, 32, 8, 1, K, 128, 128, dtype, seed=seed, seqlens_k=sk,
                             window=window, pad_value=float("nan"))


class Staged:
    """Device copies of a problem, NaN-filled outputs, and attn_fwd's result."""

    def __init__(self, inp):
        dev = torch.device("cuda")
        self.inp = inp
        self.q, self.k, self.v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
        self.sk = torch.from_numpy(inp.seqlens_k).to(dev)
        self.ref_o, self.ref_lse = attn.attn_fwd(self.q, self.k, self.v, seqlens_k=self.sk,
                                                 window=inp.window, scale=inp.scale)
        self.o = torch.full_like(self.ref_o, float("nan"))
        self.lse = torch.full_like(self.ref_lse, float("nan"))


def _call_noalloc(lib, s: Staged):
    vp = ctypes.c_void_p
    inp = s.inp
    rc = lib.attn_fwd_decode_noalloc(
        vp(s.q.data_ptr()), vp(s.k.data_ptr()), vp(s.v.data_ptr()), vp(s.o.data_ptr()),
        vp(s.lse.data_ptr()), inp.B, inp.Hq, inp.Hkv, inp.Q, inp.K, inp.D, inp.Dv, None,
        vp(s.sk.data_ptr()), inp.window, inp.scale, DT[inp.dtype],
        vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.attn_last_error().decode()


def _check(s: Staged, what):
    o = s.o.float().cpu().numpy()
    lse = s.lse.cpu().numpy()
    ro, rl = parity.run_oracle(s.inp)
    parity.compare(s.inp.dtype, o, lse, ro, rl, f"{what}: noalloc vs oracle")
    parity.compare(s.inp.dtype, o, lse, s.ref_o.float().cpu().numpy(),
                   s.ref_lse.cpu().numpy().astype(np.float64), f"{what}: noalloc vs attn_fwd")


def test_noalloc_matches_oracle_and_allocating_entry_point(lib):
    first = Staged(_problem(71, 16, 4096))
    filler = Staged(_problem(75, 64, 8192))        # more partials than the checked calls
    second = Staged(_problem(72, 24, 3000, "f16", window=700))
    single = Staged(_problem(73, 4, 100))          # one split: no scratch at all
    torch.cuda.synchronize()

    # the first call on the device looks up the array's address
    _call_noalloc(lib, first)
    torch.cuda.synchronize()
    _call_noalloc(lib, filler)                     # leaves unrelated partials behind
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    _call_noalloc(lib, second)
    _call_noalloc(lib, single)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "a call changed free device memory"

    _check(first, "bf16 B=16 K=4096")
    _check(second, "fp16 B=24 K=3000 window 700")
    _check(single, "bf16 B=4 K=100 (one split)")
    _check(filler, "bf16 B=64 K=8192")


def test_noalloc_rejects_problems_beyond_the_array(lib):
    # 512 sequences x 32 heads x 8 splits of fp32 partials (68 MB) exceed 32 MiB
    B, K = 512, 8192
    dev = torch.device("cuda")
    q = torch.zeros((B, 1, 32, 128), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((1, 16), dtype=torch.bfloat16, device=dev)  # never read: rejected first
    o = torch.empty_like(q)
    vp = ctypes.c_void_p
    rc = lib.attn_fwd_decode_noalloc(vp(q.data_ptr()), vp(kv.data_ptr()), vp(kv.data_ptr()),
                                     vp(o.data_ptr()), None, B, 32, 8, 1, K, 128, 128, None, None,
                                     0, 0.088, attn.ATTN_BF16, None)
    assert rc == 2
    assert "bytes of split-KV scratch" in lib.attn_last_error().decode()
