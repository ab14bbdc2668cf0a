"""attn_fwd_decode_noalloc: the split-KV decode for callers that may not
allocate device memory while attention runs (a process whose device memory is
owned by another runtime's allocator or held under a hard cap, or a
latency-critical decode loop).  Its partial results live in the library's
fixed device array instead of coming from an allocator.

The test calls the entry point through the C ABI twice in a row, on two
different problems, and checks each result against attn_fwd (the allocating
entry point) within the tolerances of the other parity tests; the second call
must not change the device's free memory.  It sits in a file of its own that
pytest collects last and needs nothing from the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import causal_gqa_attention_online_gb300 as attn
from causal_gqa_attention_online_gb300 import build_ext, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return attn.load_library()


def _problem(seed, B, K):
    g = np.random.default_rng(seed)
    sk = g.integers(0, K + 1, size=B).astype(np.int32)
    sk[0] = K
    sk[1] = 0
    return synth.make_padded(B, 32, 8, 1, K, 128, 128, "bf16", seed=seed, seqlens_k=sk,
                             pad_value=float("nan"))


def _call_noalloc(lib, q, k, v, o, lse, sk, inp):
    vp = ctypes.c_void_p
    rc = lib.attn_fwd_decode_noalloc(
        vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()),
        vp(lse.data_ptr()), inp.B, inp.Hq, inp.Hkv, inp.Q, inp.K, inp.D, inp.Dv, None,
        vp(sk.data_ptr()), inp.window, inp.scale, attn.ATTN_BF16,
        vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.attn_last_error().decode()


def test_noalloc_matches_allocating_entry_point_twice(lib):
    problems = [_problem(71, 16, 4096), _problem(72, 24, 3000)]
    dev = torch.device("cuda")
    staged, refs = [], []
    for inp in problems:
        q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
        sk = torch.from_numpy(inp.seqlens_k).to(dev)
        ro, rl = attn.attn_fwd(q, k, v, seqlens_k=sk, window=inp.window, scale=inp.scale)
        o = torch.full_like(ro, float("nan"))
        lse = torch.full_like(rl, float("nan"))
        staged.append((q, k, v, o, lse, sk))
        refs.append((ro, rl))
    torch.cuda.synchronize()

    # first call (looks up the array's address), then a second, different one
    _call_noalloc(lib, *staged[0], problems[0])
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    _call_noalloc(lib, *staged[1], problems[1])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before, "the call changed free device memory"

    for inp, (q, k, v, o, lse, sk), (ro, rl) in zip(problems, staged, refs):
        parity.compare("bf16", o.float().cpu().numpy(), lse.cpu().numpy(),
                       ro.float().cpu().numpy(), rl.cpu().numpy().astype(np.float64),
                       "noalloc vs attn_fwd")


def test_noalloc_rejects_problems_beyond_the_array(lib):
    # 512 sequences x 32 heads x 16 splits of fp32 partials exceed 32 MiB
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
