"""Bounded waits: a tcgen05 launch whose mbarrier waits run out reports
ATTN_ERR_TIMEOUT through the device status word and unwinds cleanly, so the
next launch on the same GPU is correct.

"Attention execution mapping" (LuisaCompute), section 21.9, records a
submission that stalled in a copy-only step; that is the reason every wait of
these kernels has a time limit and a failure is kept as an error status
instead of a hang.  Here the limit is shortened (attn_set_wait_limit, a
kernel argument, no rebuild) far below the time a unit of work takes, so that
a consumer-side wait -- the epilogue's wait for a finished O tile, the softmax
warps' wait for S -- gives up while the launch is otherwise correct.  Nothing
here faults: the unwinding blocks wait (with their own 2 s bound) for the
copies and tensor-core operations they issued before freeing tensor memory.
"""
import numpy as np
import pytest
import torch

import causal_gqa_attention_online_gb300 as attn
from causal_gqa_attention_online_gb300 import build_ext, synth
from tests import parity

pytestmark = pytest.mark.gpu

ATTN_ERR_TIMEOUT = 4
PREFILL_CODES = set(range(0x101, 0x107))  # the prefill kernel's timeout details
BWD_TC_CODE = 0x301


@pytest.fixture(scope="module", autouse=True)
def built():
    build_ext.build()
    yield
    attn.set_wait_limit(0)


def _clear_status():
    torch.cuda.synchronize()
    attn.device_status()


def test_prefill_wait_runs_out_then_next_launch_is_correct():
    # one KV group of long units: the epilogue's first wait lasts a whole unit
    inp = synth.make_padded(1, 8, 2, 4096, 4096, 128, 128, "bf16", seed=91)
    _clear_status()
    prev = attn.set_wait_limit(1)  # 1 ns: any wait that is not over at once gives up
    try:
        q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
        attn.attn_fwd(q, k, v, algo="tcgen05")
        st, detail = attn.device_status()
    finally:
        attn.set_wait_limit(prev)
    assert st == ATTN_ERR_TIMEOUT, (st, hex(detail))
    assert detail in PREFILL_CODES, hex(detail)
    # the default limit again: the same launch is correct and reports nothing
    small = synth.make_padded(2, 8, 2, 300, 400, 128, 128, "bf16", seed=92)
    parity.check(small, "tcgen05", "after a timeout")
    o, lse = parity.run_gpu(inp, "tcgen05")
    rows = parity.sample_rows(inp, 400, seed=5)
    parity.check_sampled_padded(inp, o, lse, rows, "after a timeout, same problem")
    assert attn.device_status() == (0, 0)


def test_backward_wait_runs_out_then_next_launch_is_correct():
    inp = synth.make_padded(1, 8, 2, 2048, 2048, 128, 128, "bf16", seed=93)
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    o, lse = attn.attn_fwd(q, k, v)
    g = synth.make_dout(inp, seed=94).cuda()
    ref = attn.attn_bwd(q, k, v, o, lse, g, algo="tcgen05")
    _clear_status()
    prev = attn.set_wait_limit(1)
    try:
        attn.attn_bwd(q, k, v, o, lse, g, algo="tcgen05")
        st, detail = attn.device_status()
    finally:
        attn.set_wait_limit(prev)
    assert st == ATTN_ERR_TIMEOUT, (st, hex(detail))
    assert detail == BWD_TC_CODE, hex(detail)
    again = attn.attn_bwd(q, k, v, o, lse, g, algo="tcgen05")
    torch.cuda.synchronize()
    assert attn.device_status() == (0, 0)
    for a, b in zip(again, ref):  # deterministic kernels: the same bits
        assert torch.equal(a, b)

