"""Multi-process host paths on CPU: two gloo ranks.

The benchmark: each rank runs its own replica of the workload (weak scaling,
no data-path collective); the only cross-rank operations are the barrier and
the max of the per-rank step times.  Under torchrun the reference arm runs on
rank 0 alone, and the other ranks exit 0 without work.

The sharded decode (one long context's keys split across ranks): the shard
lengths, the all-gather of the partials and their LSE merge, with the
partials taken from the oracle on each rank's shard."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, lr = bench.dist_setup()
    assert (w, r, lr) == (world, rank, rank)
    bench.barrier(w)
    # rank r measured (r + 1) ms: every rank must report the slowest
    out[rank] = bench.max_over_ranks(float(rank + 1), w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.0, 1: 2.0}


def test_reference_arm_under_torchrun_rank0_only(tmp_path):
    pytest.importorskip("numpy")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--ref-seconds", "0.4"]
    env = dict(os.environ, PYTHONPATH=ROOT, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=tmp_path)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def _shard_rank(rank, world, port, out):
    """One rank of the sharded decode's host path: its shard's key lengths,
    its partial (here from the oracle, standing in for the GPU kernel), the
    all-gather over gloo, and the merge, checked against the whole problem."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import math

    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from causal_gqa_attention_online_gb300 import sharded, synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    B, Hq, Hkv, K, D = 3, 8, 2, 700, 16
    seqlens = np.array([700, 333, 0], np.int32)
    inp = synth.make_padded(B, Hq, Hkv, 1, K, D, D, "f32", seed=91, seqlens_k=seqlens)
    shard = (K + world - 1) // world
    k_lo = rank * shard
    local = sharded.shard_key_lengths(torch.from_numpy(seqlens), k_lo, shard).numpy()
    kk = synth.exact_f32(inp.k)[:, k_lo:k_lo + shard]
    vv = synth.exact_f32(inp.v)[:, k_lo:k_lo + shard]
    o, lse = oracle.attn_padded(synth.exact_f32(inp.q), kk, vv, B=B, Hq=Hq, Hkv=Hkv, Q=1,
                                K=kk.shape[1], D=D, Dv=D, seqlens_k=local, scale=inp.scale)
    o_all, lse_all = sharded.gather_partials(torch.from_numpy(o.reshape(B * Hq, D)),
                                             torch.from_numpy(lse.reshape(B * Hq)))
    o_all, lse_all = o_all.numpy(), lse_all.numpy()
    mx = lse_all.max(axis=0)
    fin = np.isfinite(mx)
    w = np.where(fin, np.exp(lse_all - np.where(fin, mx, 0.0)), 0.0)
    merged = np.einsum("sr,srd->rd", w, o_all) / np.where(fin, w.sum(axis=0), 1.0)[:, None]
    ro, rl = oracle.attn_padded(synth.exact_f32(inp.q), synth.exact_f32(inp.k),
                                synth.exact_f32(inp.v), B=B, Hq=Hq, Hkv=Hkv, Q=1, K=K, D=D, Dv=D,
                                seqlens_k=seqlens, scale=inp.scale)
    ro, rl = ro.reshape(B * Hq, D), rl.reshape(B * Hq)
    ok = np.allclose(merged[fin], ro[fin], atol=1e-12) and np.array_equal(fin, np.isfinite(rl))
    ok = ok and np.allclose(mx[fin] + np.log(w.sum(axis=0)[fin]), rl[fin], atol=1e-12)
    ok = ok and bool(np.all(~fin[2 * Hq:])) and math.isinf(rl[-1])
    out[rank] = bool(ok)
    dist.destroy_process_group()


def test_sharded_decode_host_path_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_shard_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    assert dict(out) == {0: True, 1: True}
