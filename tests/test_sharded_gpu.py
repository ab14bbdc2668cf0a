"""The sharded decode on the GPU: two ranks, both on cuda:0, each holding half
of every sequence's keys, exchange their partials through gloo (host memory)
and merge them with the library's combine kernel; the result is compared with
the fp64 oracle on the whole problem.  The two ranks' kernels never wait on
each other: the only exchange is the host-side all-gather between launches.

"Attention execution mapping" (LuisaCompute), section 5: split-KV needs a legal
merge of the (max, sum, acc) state -- here across GPUs instead of within one.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

from causal_gqa_attention_online_gb300 import build_ext

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, dtype, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist

    from causal_gqa_attention_online_gb300 import sharded, synth
    from tests import parity
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    B, Hq, Hkv, K, D = 4, 32, 8, 3000, 128
    seqlens = np.array([3000, 1234, 0, 1537], np.int32)
    inp = synth.make_padded(B, Hq, Hkv, 1, K, D, D, dtype, seed=93, seqlens_k=seqlens,
                            pad_value=float("nan"))
    shard = 1536  # rank 1 holds keys [1536, 3000): a shorter shard
    k_lo = rank * shard
    q = inp.q.cuda()
    ks = inp.k[:, k_lo:k_lo + shard].contiguous().cuda()
    vs = inp.v[:, k_lo:k_lo + shard].contiguous().cuda()
    o, lse = sharded.attn_decode_sharded_keys(q, ks, vs, torch.from_numpy(seqlens), k_lo,
                                              scale=inp.scale)
    torch.cuda.synchronize()
    ro, rl = parity.run_oracle(inp)
    eo, el = parity.compare(inp.dtype, o.float().cpu().numpy(), lse.cpu().numpy(), ro, rl,
                            f"sharded decode rank {rank}")
    out[rank] = (eo, el)
    dist.destroy_process_group()


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_sharded_decode_two_ranks_on_one_gpu(dtype):
    build_ext.build()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, dtype, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(600)
        assert p.exitcode == 0
    assert sorted(out.keys()) == [0, 1]
