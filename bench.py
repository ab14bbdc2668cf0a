"""Benchmark of the causal GQA attention forward on one GB300 (or N, one
process per GPU under torchrun: weak scaling, each rank runs its own copy of
the workload, no data-path collective).

Headline workload (value): bf16 causal prefill B=4 Hq=32 Hkv=8 Q=K=4096
D=Dv=128, TFLOP/s counted over legal (query, key) pairs only:
FLOP = B * Hq * pairs * (2*D + 2*Dv).
Second workload (the "decode" object): bf16 batched decode B=64 Hq=32 Hkv=8
Q=1 D=Dv=128, key lengths uniform on [0, 8192] (0 included), KV padded to
8192, KV GB/s counted over valid key rows: bytes = sum_b Kb * Hkv * (D+Dv) * 2.

The "wide_heads" list: bf16 causal prefill with D = Dv = 256 (B=2 Hq=16
Hkv=4 Q=K=4096) and 512 (B=1), TFLOP/s over legal pairs as above.
Third workload (the "backward" object): attn_bwd on the prefill workload for
a seeded N(0,1) dO, FLOP = B * Hq * pairs * (6*D + 4*Dv) (the five products
S, dP, dV, dK, dQ).

Timing: W warm-up steps, then K timed steps; before every step a 512 MiB
buffer is written to flush L2, and each step is bracketed by CUDA events on
the launching stream (device time of the attention call only); a barrier and
a device synchronize bracket the timed region; the max over ranks is taken.
The e2e figures time the public staged entry point (attn_fwd_staged) on
pinned host tensors: every step copies the inputs' valid rows in, runs the
attention and copies O / LSE back, the copies of one group of sequences
overlapping the attention of another.

``--impl reference`` times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal GQA attention TFLOP/s (prefill) and KV GB/s (decode) on 1 GB300"
PREFILL = dict(B=4, Hq=32, Hkv=8, Q=4096, K=4096, D=128, Dv=128)
DECODE = dict(B=64, Hq=32, Hkv=8, Q=1, K=8192, D=128, Dv=128)
PREFILL_NAME = "bf16 causal prefill B=4 Hq=32 Hkv=8 Q=K=4096 D=Dv=128"
DECODE_NAME = ("bf16 batched decode B=64 Hq=32 Hkv=8 Q=1 D=Dv=128, key lengths U[0,8192], "
               "KV padded to 8192")
FLUSH_BYTES = 512 << 20


def prefill_flop() -> int:
    P = PREFILL
    return P["B"] * P["Hq"] * legal_pairs(P["Q"], P["K"]) * (2 * P["D"] + 2 * P["Dv"])


def prefill_config(world: int) -> dict:
    """The headline workload's config object (the same for both arms)."""
    P = PREFILL
    return {"workload": PREFILL_NAME, "B": P["B"], "Hq": P["Hq"], "Hkv": P["Hkv"],
            "seq_len": P["Q"], "D": P["D"], "Dv": P["Dv"], "global_batch": P["B"] * world,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "512 MiB buffer written before every timed step",
            "flop_per_step": prefill_flop()}


def legal_pairs(Qb: int, Kb: int, window: int = 0) -> int:
    """Legal (query, key) pairs of one sequence and head (closed form)."""
    total = 0
    if Qb <= 0 or Kb <= 0:
        return 0
    # row q sees keys [lo, hi) with hi = min(q + Kb - Qb + 1, Kb), lo = max(0, hi' - window)
    for q in range(Qb):
        diag = q + Kb - Qb
        hi = min(diag + 1, Kb)
        lo = max(0, diag - window + 1) if window > 0 else 0
        total += max(0, hi - lo)
    return total


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples every 20 ms, each stamped with the
    host time it arrived; summary() keeps the samples inside the timed windows
    recorded with mark() (or, if a window is shorter than the sampling
    interval, the samples within 50 ms of it)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.windows = []
        self.thread = None

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line))

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._reader, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.2)
        return self

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def __exit__(self, *exc):
        time.sleep(0.1)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def pick(margin):
            return [(t, l) for t, l in self.lines
                    if any(a - margin <= t <= b + margin for a, b in self.windows)]

        chosen, where = pick(0.0), "inside the timed region"
        if not chosen:
            chosen, where = pick(0.05), "within 50 ms of the timed region"
        sm, smax, reasons = [], None, set()
        for _, line in chosen:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "samples_from": where}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_steps(fn, steps, warmup, flush, stream, clk=None):
    """Per-step device time (ms) of fn() with an L2 flush before each step.
    The host-side window of the timed steps is recorded on ``clk``."""
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    t0 = time.time()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.mark(t0, time.time())
    return [a.elapsed_time(b) for a, b in evs]


def measure_prefill(args, world, rank, dev, stream, flush, attn, synth):
    P = PREFILL
    pin = synth.prefill_bf16_b4_h32x8_s4096_d128(seed=1234 + rank)
    q, k, v = pin.q.to(dev), pin.k.to(dev), pin.v.to(dev)
    o = torch.empty((P["B"], P["Q"], P["Hq"], P["Dv"]), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((P["B"], P["Q"], P["Hq"]), dtype=torch.float32, device=dev)
    flop = P["B"] * P["Hq"] * legal_pairs(P["Q"], P["K"]) * (2 * P["D"] + 2 * P["Dv"])

    def prefill():
        attn.attn_fwd(q, k, v, o, lse, stream=stream)

    prefill()
    torch.cuda.synchronize()
    n0 = attn.kernel_launches()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        times = time_steps(prefill, args.steps, args.warmup, flush, stream, clk)
    torch.cuda.synchronize()
    barrier(world)
    launches = (attn.kernel_launches() - n0) // (args.steps + args.warmup)
    ms = max_over_ranks(sum(times) / len(times), world)

    # e2e: pinned host inputs copied in, O / LSE copied back, every step, by
    # the library's staged entry point (copies of one group of sequences
    # overlap the attention of another)
    hq, hk, hv = pin.q.pin_memory(), pin.k.pin_memory(), pin.v.pin_memory()
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    moved = [0, 0]

    def prefill_e2e():
        _, _, moved[0], moved[1] = attn.attn_fwd_staged(hq, hk, hv, q, k, v, o, lse, ho, hl,
                                                        stream=stream)

    e2e_times = time_steps(prefill_e2e, max(3, args.steps // 2), 3, flush, stream)
    e2e_ms = max_over_ranks(sum(e2e_times) / len(e2e_times), world)
    return dict(pin=pin, flop=flop, ms=ms, launches=launches, clocks=clk.summary(),
                e2e_ms=e2e_ms, h2d=moved[0], d2h=moved[1])


def measure_decode(args, world, rank, dev, stream, flush, attn, synth):
    Dd = DECODE
    din = synth.decode_bf16_b64_h32x8_k8192_d128(seed=1234 + rank)
    dq, dk, dv = din.q.to(dev), din.k.to(dev), din.v.to(dev)
    dsk = torch.from_numpy(din.seqlens_k).to(dev)
    do = torch.empty((Dd["B"], 1, Dd["Hq"], Dd["Dv"]), dtype=torch.bfloat16, device=dev)
    dl = torch.empty((Dd["B"], 1, Dd["Hq"]), dtype=torch.float32, device=dev)
    kv_bytes = int(din.seqlens_k.astype(np.int64).sum()) * Dd["Hkv"] * (Dd["D"] + Dd["Dv"]) * 2

    def decode():
        attn.attn_fwd(dq, dk, dv, do, dl, seqlens_k=dsk, stream=stream)

    decode()
    torch.cuda.synchronize()
    n1 = attn.kernel_launches()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        times = time_steps(decode, args.steps, args.warmup, flush, stream, clk)
    barrier(world)
    launches = (attn.kernel_launches() - n1) // (args.steps + args.warmup)
    ms = max_over_ranks(sum(times) / len(times), world)
    hdq, hdk, hdv = din.q.pin_memory(), din.k.pin_memory(), din.v.pin_memory()
    hsk = torch.from_numpy(din.seqlens_k).pin_memory()
    hdo = torch.empty(do.shape, dtype=do.dtype).pin_memory()
    hdl = torch.empty(dl.shape, dtype=dl.dtype).pin_memory()
    moved = [0, 0]

    def decode_e2e():
        # key lengths in, then the valid K/V rows of each group of sequences
        # (the padding past Kb is never read), attention, O / LSE out
        with torch.cuda.stream(stream):
            dsk.copy_(hsk, non_blocking=True)
        _, _, moved[0], moved[1] = attn.attn_fwd_staged(hdq, hdk, hdv, dq, dk, dv, do, dl, hdo, hdl,
                                                        seqlens_k=hsk, seqlens_k_dev=dsk,
                                                        stream=stream)

    e2e_times = time_steps(decode_e2e, max(3, args.steps // 2), 3, flush, stream)
    e2e_ms = max_over_ranks(sum(e2e_times) / len(e2e_times), world)

    # the same decode with the K / V cache in shuffled 64-row pages (attn_fwd_paged)
    page = 64
    npg = Dd["K"] // page
    perm = torch.randperm(Dd["B"] * npg, generator=torch.Generator().manual_seed(99 + rank))
    table = perm.view(Dd["B"], npg).to(torch.int32).to(dev)
    kpool = torch.empty((Dd["B"] * npg, page, Dd["Hkv"], Dd["D"]), dtype=dk.dtype, device=dev)
    vpool = torch.empty((Dd["B"] * npg, page, Dd["Hkv"], Dd["Dv"]), dtype=dv.dtype, device=dev)
    kpool[perm.to(dev)] = dk.view(Dd["B"] * npg, page, Dd["Hkv"], Dd["D"])
    vpool[perm.to(dev)] = dv.view(Dd["B"] * npg, page, Dd["Hkv"], Dd["Dv"])

    def decode_paged():
        attn.attn_fwd_paged(dq, kpool, vpool, table, dsk, do, dl, stream=stream)

    paged_times = time_steps(decode_paged, max(3, args.steps // 2), 3, flush, stream)
    paged_ms = max_over_ranks(sum(paged_times) / len(paged_times), world)
    del kpool, vpool
    return dict(kv_bytes=kv_bytes, ms=ms, launches=launches, clocks=clk.summary(),
                e2e_ms=e2e_ms, h2d=moved[0] + dsk.numel() * 4, d2h=moved[1],
                paged_ms=paged_ms, page=page, inp=din,
                flop=int(din.seqlens_k.astype(np.int64).sum()) * Dd["Hq"] * 2 * (
                    Dd["D"] + Dd["Dv"]))


def measure_backward(args, world, rank, dev, stream, flush, attn, synth, pin):
    """attn_bwd on the prefill workload with a seeded N(0,1) dO: one step is
    the two launches (dQ with rowsum(dO*O), then dK/dV), O and LSE from
    attn_fwd."""
    P = PREFILL
    q, k, v = pin.q.to(dev), pin.k.to(dev), pin.v.to(dev)
    o, lse = attn.attn_fwd(q, k, v, stream=stream)
    g = synth.make_dout(pin, seed=4321 + rank).to(dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    # five products over the legal pairs: S, dP, dV, dK, dQ
    flop = P["B"] * P["Hq"] * legal_pairs(P["Q"], P["K"]) * (6 * P["D"] + 4 * P["Dv"])

    def bwd():
        attn.attn_bwd(q, k, v, o, lse, g, dq, dk, dv, stream=stream)

    bwd()
    torch.cuda.synchronize()
    n0 = attn.kernel_launches()
    steps = max(3, args.steps // 4)
    times = time_steps(bwd, steps, 3, flush, stream)
    launches = (attn.kernel_launches() - n0) // (steps + 3)
    ms = max_over_ranks(sum(times) / len(times), world)
    return dict(flop=flop, ms=ms, launches=launches, steps=steps)


def measure_small_configs(args, world, rank, dev, stream, flush, attn, synth):
    """The other named workloads, each through attn_fwd / attn_fwd_varlen as
    a caller runs it: fp32 prefill B=1 Hq=4 Hkv=2 Q=64 K=128 D=Dv=64, fp32
    decode B=1 Hq=8 Hkv=2 Q=1 K=2053 D=80 Dv=96, and the bf16 varlen chunked
    prefill (16 packed sequences, Hq=16 Hkv=4, window 1024).  Returns
    [(name, inputs, FLOP, KV bytes, ms)]."""
    out = []
    named = [("fp32 prefill B=1 Hq=4 Hkv=2 Q=64 K=128 D=Dv=64",
              synth.prefill_f32_b1_h4x2_q64_k128_d64(seed=1234 + rank)),
             ("fp32 decode B=1 Hq=8 Hkv=2 Q=1 K=2053 D=80 Dv=96",
              synth.decode_f32_b1_h8x2_k2053_d80x96(seed=1234 + rank)),
             ("bf16 varlen chunked prefill: 16 packed sequences, Kb U[0,4096] incl. empty, "
              "Qb = min(512, Kb), Hq=16 Hkv=4 D=Dv=128, window 1024",
              synth.varlen_bf16_16seq_h16x4_k4096_q512_w1024(seed=1234 + rank))]
    for name, inp in named:
        q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
        es = inp.q.element_size()
        if inp.layout == "padded":
            Qb = np.full(inp.B, inp.Q) if inp.seqlens_q is None else inp.seqlens_q
            Kb = np.full(inp.B, inp.K) if inp.seqlens_k is None else inp.seqlens_k

            def run():
                attn.attn_fwd(q, k, v, scale=inp.scale, window=inp.window, stream=stream)
        else:
            cq = torch.from_numpy(inp.cu_seqlens_q).to(dev)
            ck = torch.from_numpy(inp.cu_seqlens_k).to(dev)
            Qb = np.diff(inp.cu_seqlens_q)
            Kb = np.diff(inp.cu_seqlens_k)

            def run():
                attn.attn_fwd_varlen(q, k, v, cq, ck, inp.Q, inp.K, scale=inp.scale,
                                     window=inp.window, stream=stream)
        pairs = sum(legal_pairs(int(a), int(b), inp.window) for a, b in zip(Qb, Kb))
        flop = pairs * inp.Hq * (2 * inp.D + 2 * inp.Dv)
        kv = int(np.sum(Kb)) * inp.Hkv * (inp.D + inp.Dv) * es
        times = time_steps(run, 20, 3, flush, stream)
        out.append((name, inp, flop, kv, max_over_ranks(statistics.median(times), world)))
    return out


MASKED = dict(B=4, Hq=32, Hkv=8, Q=4096, K=4096, D=128, Dv=128, qblock=64, density=0.5)
MASKED_NAME = ("bf16 causal prefill B=4 Hq=32 Hkv=8 Q=K=4096 D=Dv=128 AND a block-sparse mask "
               "shared by the heads (64 x 128 blocks, each allowed with probability 0.5)")


def measure_masked(args, world, rank, dev, stream, flush, attn, synth, pin):
    """attn_fwd_masked on the prefill workload with a seeded block-sparse mask:
    TFLOP/s over the legal pairs (causal AND the mask), FLOP = pairs x (2D + 2Dv)."""
    M = MASKED
    q, k, v = pin.q.to(dev), pin.k.to(dev), pin.v.to(dev)
    g = np.random.default_rng(555 + rank)
    nq, nk = M["Q"] // M["qblock"], M["K"] // 128
    blocks = g.random((M["B"], 1, nq, nk)) < M["density"]
    allow = np.repeat(np.repeat(blocks, M["qblock"], axis=2), 128, axis=3)
    causal = np.tril(np.ones((M["Q"], M["K"]), bool), k=M["K"] - M["Q"])
    pairs = int(np.logical_and(allow[:, 0], causal[None]).sum()) * M["Hq"]
    flop = pairs * (2 * M["D"] + 2 * M["Dv"])
    words = attn.pack_mask(torch.from_numpy(allow)).to(dev)
    o = torch.empty((M["B"], M["Q"], M["Hq"], M["Dv"]), dtype=q.dtype, device=dev)
    lse = torch.empty((M["B"], M["Q"], M["Hq"]), dtype=torch.float32, device=dev)

    def run():
        attn.attn_fwd_masked(q, k, v, words, o, lse, mask="causal", stream=stream)

    run()
    torch.cuda.synchronize()
    n0 = attn.kernel_launches()
    steps = max(3, args.steps // 4)
    times = time_steps(run, steps, 3, flush, stream)
    launches = (attn.kernel_launches() - n0) // (steps + 3)
    ms = max_over_ranks(sum(times) / len(times), world)
    return dict(flop=flop, ms=ms, steps=steps, launches=launches,
                density=float(blocks.mean()))


WIDE = [dict(B=2, Hq=16, Hkv=4, Q=4096, K=4096, D=256, Dv=256),
        dict(B=1, Hq=16, Hkv=4, Q=4096, K=4096, D=512, Dv=512)]


def measure_wide(args, world, rank, dev, stream, flush, attn, synth):
    """bf16 causal prefill with head widths 256 (the tcgen05 wide-head kernel)
    and 512 (the tcgen05 kernel with the output columns in halves), as
    attn_fwd chooses them."""
    out = []
    for W in WIDE:
        inp = synth.make_padded(W["B"], W["Hq"], W["Hkv"], W["Q"], W["K"], W["D"], W["Dv"],
                                "bf16", seed=777 + rank)
        q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
        o, lse = attn.attn_fwd(q, k, v, stream=stream)
        flop = W["B"] * W["Hq"] * legal_pairs(W["Q"], W["K"]) * (2 * W["D"] + 2 * W["Dv"])

        def fwd():
            attn.attn_fwd(q, k, v, o, lse, stream=stream)

        steps = max(3, args.steps // 4)
        times = time_steps(fwd, steps, 3, flush, stream)
        ms = max_over_ranks(sum(times) / len(times), world)
        out.append((W, flop, ms, steps))
        del q, k, v, o, lse
    return out


def run_gpu(args, world, rank, local):
    import causal_gqa_attention_online_gb300 as attn
    from causal_gqa_attention_online_gb300 import build_ext, synth

    build_ext.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    hbm_peak, tf_peak, peak_src = measured_peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    traffic = load_traffic()
    P = PREFILL
    result = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
              "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
              "data": "synthetic: N(0,1) seeded (PCG64), bf16 round-to-nearest"}
    pin = None
    dec_in = None
    if args.only in ("all", "prefill"):
        r = measure_prefill(args, world, rank, dev, stream, flush, attn, synth)
        pin = r["pin"]
        tf = r["flop"] / (r["ms"] * 1e-3) / 1e12
        result.update({
            "value": round(world * tf, 3), "unit": "TFLOP/s", "ms_per_step": round(r["ms"], 5),
            "config": prefill_config(world),
            "roofline": {"bound": "tensor", "achieved": round(tf, 3), "peak": tf_peak,
                         "unit": "TFLOP/s", "frac": round(tf / tf_peak, 4),
                         "traffic": traffic.get("prefill"),
                         "peak_source": f"{peak_src} bf16 dense (cuBLAS burst)"},
            "e2e": {"value": round(world * r["flop"] / (r["e2e_ms"] * 1e-3) / 1e12, 3),
                    "unit": "TFLOP/s", "ms_per_step": round(r["e2e_ms"], 4),
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": int(r["launches"] * args.steps),
            "clocks": r["clocks"],
        })
    if args.only in ("all", "backward"):
        if pin is None:
            pin = synth.prefill_bf16_b4_h32x8_s4096_d128(seed=1234 + rank)
        bw = measure_backward(args, world, rank, dev, stream, flush, attn, synth, pin)
        tfb = bw["flop"] / (bw["ms"] * 1e-3) / 1e12
        bwd = {"workload": PREFILL_NAME + ", backward (dQ, dK, dV) for N(0,1) dO",
               "value": round(world * tfb, 3), "unit": "TFLOP/s",
               "ms_per_step": round(bw["ms"], 5), "steps": bw["steps"],
               "flop_per_step": bw["flop"], "gpu_launches": int(bw["launches"] * bw["steps"]),
               "kernels": "tcgen05 dQ (computing rowsum(dO*O)), then tcgen05 dK/dV as its "
                          "programmatic dependent (TMEM accumulators, TMA-fed)",
               "roofline": {"bound": "tensor", "achieved": round(tfb, 3), "peak": tf_peak,
                            "unit": "TFLOP/s", "frac": round(tfb / tf_peak, 4),
                            "traffic": traffic.get("backward"),
                            "peak_source": f"{peak_src} bf16 dense (cuBLAS burst)"}}
        if args.only == "backward":
            result.update({"value": bwd["value"], "unit": "TFLOP/s",
                           "ms_per_step": bwd["ms_per_step"],
                           "config": {"workload": bwd["workload"]}, "roofline": bwd["roofline"],
                           "gpu_launches": bwd["gpu_launches"]})
        else:
            result["backward"] = bwd
    if args.only in ("all", "masked"):
        if pin is None:
            pin = synth.prefill_bf16_b4_h32x8_s4096_d128(seed=1234 + rank)
        mk = measure_masked(args, world, rank, dev, stream, flush, attn, synth, pin)
        tfm = mk["flop"] / (mk["ms"] * 1e-3) / 1e12
        result["masked"] = {
            "workload": MASKED_NAME, "value": round(world * tfm, 3), "unit": "TFLOP/s",
            "ms_per_step": round(mk["ms"], 5), "steps": mk["steps"], "flop_per_step": mk["flop"],
            "block_density": round(mk["density"], 4), "gpu_launches": int(mk["launches"] * mk["steps"]),
            "kernels": "mask_summary_kernel + unit_order_kernel + prefill_tc_kernel (dead tiles skipped)",
            "roofline": {"bound": "tensor", "achieved": round(tfm, 3), "peak": tf_peak,
                         "unit": "TFLOP/s", "frac": round(tfm / tf_peak, 4),
                         "traffic": traffic.get("masked"),
                         "peak_source": f"{peak_src} bf16 dense (cuBLAS burst)"}}
        if args.only == "masked":
            result.update({"value": result["masked"]["value"], "unit": "TFLOP/s",
                           "ms_per_step": result["masked"]["ms_per_step"],
                           "config": {"workload": MASKED_NAME},
                           "roofline": result["masked"]["roofline"]})
    small = None
    if args.only in ("all", "configs"):
        small = measure_small_configs(args, world, rank, dev, stream, flush, attn, synth)
        result["configs"] = []
        for name, inp, flop, kv, ms in small:
            entry = {"workload": name, "ms_per_step": round(ms, 5),
                     "us_per_step": round(ms * 1e3, 2),
                     "TFLOP/s": round(world * flop / (ms * 1e-3) / 1e12, 4),
                     "KV GB/s": round(world * kv / (ms * 1e-3) / 1e9, 2), "flop_per_step": flop,
                     "kv_bytes_per_step": kv,
                     "timing": ("median of 20 steps, L2 flushed before each; CUDA events on "
                                "the launching stream around one call")}
            if inp.dtype != "f32":
                tfv = flop / (ms * 1e-3) / 1e12
                entry["kernel"] = "prefill_tc_kernel (tcgen05, packed layout)"
                entry["roofline"] = {
                    "bound": "tensor", "achieved": round(tfv, 3), "peak": tf_peak,
                    "unit": "TFLOP/s", "frac": round(tfv / tf_peak, 4),
                    "traffic": traffic.get("varlen"),
                    "peak_source": f"{peak_src} bf16 dense (cuBLAS burst)"}
            else:
                entry["bound"] = "latency (a few MFLOP: launch and one wave of small blocks)"
            result["configs"].append(entry)
        if args.only == "configs":
            c0 = result["configs"][0]
            result.update({"value": c0["TFLOP/s"], "unit": "TFLOP/s",
                           "ms_per_step": c0["ms_per_step"], "config": {"workload": c0["workload"]}})
    if args.only in ("all", "wide"):
        wide = []
        for W, flop, ms, steps in measure_wide(args, world, rank, dev, stream, flush, attn,
                                               synth):
            tfw = flop / (ms * 1e-3) / 1e12
            wide.append({
                "workload": (f"bf16 causal prefill B={W['B']} Hq={W['Hq']} Hkv={W['Hkv']} "
                             f"Q=K={W['Q']} D=Dv={W['D']}"),
                "value": round(world * tfw, 3), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
                "steps": steps, "flop_per_step": flop,
                "kernel": ("prefill_wide512_tc_kernel (tcgen05, output columns in halves of "
                           "256, K / V streamed in 16 KB chunks)" if W["D"] > 256
                           else "prefill_wide_tc_kernel (tcgen05, one Q tile, S double-buffered)"),
                "roofline": {"bound": "tensor", "achieved": round(tfw, 3), "peak": tf_peak,
                             "unit": "TFLOP/s", "frac": round(tfw / tf_peak, 4),
                             "traffic": traffic.get(f"wide{W['D']}"),
                             "peak_source": f"{peak_src} bf16 dense (cuBLAS burst)"}})
        result["wide_heads"] = wide
        if args.only == "wide":
            result.update({"value": wide[0]["value"], "unit": "TFLOP/s",
                           "ms_per_step": wide[0]["ms_per_step"],
                           "config": {"workload": wide[0]["workload"]},
                           "roofline": wide[0]["roofline"]})
    if args.only in ("all", "decode"):
        d = measure_decode(args, world, rank, dev, stream, flush, attn, synth)
        dec_in = (DECODE_NAME, d["inp"], d["flop"], d["kv_bytes"])
        gbs = d["kv_bytes"] / (d["ms"] * 1e-3) / 1e9
        dec = {
            "workload": DECODE_NAME, "metric": "KV GB/s", "value": round(world * gbs, 2),
            "unit": "GB/s", "ms_per_step": round(d["ms"], 5), "kv_bytes_per_step": d["kv_bytes"],
            "gpu_launches": int(d["launches"] * args.steps), "clocks": d["clocks"],
            "roofline": {"bound": "hbm", "achieved": round(gbs, 2), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                         "traffic": traffic.get("decode"),
                         "peak_source": f"{peak_src} HBM copy"},
            "e2e": {"value": round(world * d["kv_bytes"] / (d["e2e_ms"] * 1e-3) / 1e9, 2),
                    "unit": "GB/s", "ms_per_step": round(d["e2e_ms"], 4),
                    "h2d_bytes_per_step": d["h2d"], "d2h_bytes_per_step": d["d2h"]},
            "paged": {"page_size": d["page"], "layout": "K/V in shuffled pages (attn_fwd_paged)",
                      "value": round(world * d["kv_bytes"] / (d["paged_ms"] * 1e-3) / 1e9, 2),
                      "unit": "GB/s", "ms_per_step": round(d["paged_ms"], 5)},
        }
        if args.only == "decode":
            result.update({"value": dec["value"], "unit": "GB/s", "ms_per_step": dec["ms_per_step"],
                           "config": {"workload": DECODE_NAME}, "roofline": dec["roofline"],
                           "e2e": dec["e2e"], "gpu_launches": dec["gpu_launches"],
                           "clocks": dec["clocks"], "paged": dec["paged"]})
        else:
            result["decode"] = dec
    return result, (pin, small, dec_in)


KERNEL_SOURCES = {
    "prefill": "causal_gqa_attention_online_gb300/csrc/kernel_prefill_tc.cu",
    "varlen": "causal_gqa_attention_online_gb300/csrc/kernel_prefill_tc.cu",
    "masked": "causal_gqa_attention_online_gb300/csrc/kernel_prefill_tc.cu",
    "decode": "causal_gqa_attention_online_gb300/csrc/kernel_decode.cu",
    "backward": ("causal_gqa_attention_online_gb300/csrc/kernel_bwd.cu",
                 "causal_gqa_attention_online_gb300/csrc/kernel_bwd_tc.cu"),
    "wide256": ("causal_gqa_attention_online_gb300/csrc/kernel_prefill_wide_tc.cu",
                "causal_gqa_attention_online_gb300/csrc/wide_common.cuh"),
    "wide512": ("causal_gqa_attention_online_gb300/csrc/kernel_prefill_wide512_tc.cu",
                "causal_gqa_attention_online_gb300/csrc/wide_common.cuh"),
}


def source_sha(rel) -> str:
    """sha256[:16] of a kernel source file (or of several, concatenated)."""
    import hashlib
    h = hashlib.sha256()
    for r in ((rel,) if isinstance(rel, str) else rel):
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic():
    """Per-launch DRAM bytes (read + write) from the committed ncu summary
    profiles/traffic.json, kept only while the kernel source is unchanged
    since the capture (its sha256 prefix is stored beside the figure)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        d = json.load(f)
    out = {}
    for name, rel in KERNEL_SOURCES.items():
        e = d.get(name)
        if e and e.get("source_sha") == source_sha(rel):
            out[name] = e.get("bytes_per_launch")
    return out


def oracle_inputs(inp):
    """The prefill workload's inputs as the exact float32 values the oracle takes."""
    from causal_gqa_attention_online_gb300 import synth
    return synth.exact_f32(inp.q), synth.exact_f32(inp.k), synth.exact_f32(inp.v)


def oracle_sample_rate(qkv, rows_budget_s=12.0, nthreads=0, seed=0):
    """Time the CPU oracle on random query rows of the prefill workload (its
    inputs ``qkv`` from oracle_inputs) until about ``rows_budget_s`` seconds of
    work; returns (TFLOP/s, rows, secs, threads)."""
    import oracle

    q32, k32, v32 = qkv
    g = np.random.default_rng(seed)
    P = PREFILL
    total_flop, total_s, nrows = 0, 0.0, 0
    batch = 2048 if rows_budget_s >= 1.0 else 64
    while total_s < rows_budget_s:
        rows = np.stack([g.integers(0, P["B"], batch), g.integers(0, P["Q"], batch),
                         g.integers(0, P["Hq"], batch)], axis=1).astype(np.int32)
        t0 = time.perf_counter()
        oracle.attn_padded_rows(q32, k32, v32, rows, B=P["B"], Hq=P["Hq"], Hkv=P["Hkv"],
                                Q=P["Q"], K=P["K"], D=P["D"], Dv=P["Dv"], nthreads=nthreads)
        total_s += time.perf_counter() - t0
        # row q of a Q=K problem sees q+1 keys
        total_flop += int((rows[:, 1].astype(np.int64) + 1).sum()) * (2 * P["D"] + 2 * P["Dv"])
        nrows += batch
    threads = nthreads if nthreads > 0 else oracle.max_threads()
    return total_flop / total_s / 1e12, nrows, total_s, threads


def oracle_small_configs(workloads):
    """The oracle in full on the other named workloads (the two fp32 ones, the
    bf16 varlen chunked prefill and the bf16 batched decode): median wall time
    of a few runs on every host core, and on one thread for the fp32 ones;
    each with the throughput in the workload's own unit."""
    import oracle
    cores = oracle.max_threads()  # before any call sets a thread count
    out = []
    for name, inp, flop, kv in workloads:
        q32, k32, v32 = (synth_exact(t) for t in (inp.q, inp.k, inp.v))
        row = {"workload": name, "cores": cores}
        runs = (("all_cores", cores), ("1_thread", 1)) if inp.dtype == "f32" else (
            ("all_cores", cores),)
        for label, nt in runs:
            ts = []
            for _ in range(5 if inp.dtype == "f32" else 3):
                t0 = time.perf_counter()
                if inp.layout == "padded":
                    oracle.attn_padded(q32, k32, v32, B=inp.B, Hq=inp.Hq, Hkv=inp.Hkv, Q=inp.Q,
                                       K=inp.K, D=inp.D, Dv=inp.Dv, seqlens_q=inp.seqlens_q,
                                       seqlens_k=inp.seqlens_k, window=inp.window,
                                       scale=inp.scale, nthreads=nt)
                else:
                    oracle.attn_packed(q32, k32, v32, B=inp.B, Hq=inp.Hq, Hkv=inp.Hkv, D=inp.D,
                                       Dv=inp.Dv, cu_seqlens_q=inp.cu_seqlens_q,
                                       cu_seqlens_k=inp.cu_seqlens_k, window=inp.window,
                                       scale=inp.scale, nthreads=nt)
                ts.append(time.perf_counter() - t0)
            sec = statistics.median(ts)
            row[f"us_{label}"] = round(sec * 1e6, 1)
            row[f"TFLOP/s_{label}"] = round(flop / sec / 1e12, 5)
            row[f"KV GB/s_{label}"] = round(kv / sec / 1e9, 3)
        out.append(row)
    return out


def synth_exact(t):
    return t.detach().to("cpu").float().numpy()


def run_reference(args, world, rank):
    """The reference arm: the fp64 CPU oracle on every host core, on the
    headline workload's inputs.  Each step is a bounded sample of the
    workload (random (b, q, h) output rows, about ``ref_seconds / (steps +
    warmup)`` seconds of oracle work) whose wall time is measured: ms_per_step
    is that measured time, value the sampled rows' legal-pair FLOP over it."""
    from causal_gqa_attention_online_gb300 import synth
    if rank != 0:
        return None
    qkv = oracle_inputs(synth.prefill_bf16_b4_h32x8_s4096_d128(seed=1234))
    per_step_s = max(0.05, args.ref_seconds / max(1, args.steps + args.warmup))
    step_s, step_flop, step_rows = [], [], []
    threads = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        r, nrows, secs, threads = oracle_sample_rate(qkv, per_step_s, seed=i)
        wall = time.perf_counter() - t0
        if i >= args.warmup:
            step_s.append(wall)
            step_flop.append(r * 1e12 * secs)
            step_rows.append(nrows)
    value = sum(step_flop) / sum(step_s) / 1e12
    ms = sum(step_s) / len(step_s) * 1e3
    sample = (f"{int(statistics.mean(step_rows))} random (b, q, h) output rows of the prefill "
              f"workload per step (batches of 2048 rows, ~{per_step_s:.1f} s of oracle work); "
              f"value = their legal-pair FLOP / measured wall time")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": prefill_config(world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: total seconds of oracle work over all steps")
    ap.add_argument("--only", default="all",
                    choices=["all", "prefill", "decode", "backward", "wide", "configs", "masked"],
                    help="profiling aid: run one workload (the JSON line then lacks the other)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res))
        return
    res, (pin, small, dec_in) = run_gpu(args, world, rank, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline and pin is not None:
            r, nrows, secs, threads = oracle_sample_rate(oracle_inputs(pin), 12.0)
            res["cpu_baseline"] = {
                "value": r, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "sample": f"{nrows} random (b, q, h) rows of the prefill workload, {secs:.1f} s"}
            more = [(name, inp, flop, kv) for name, inp, flop, kv, _ in (small or [])]
            if dec_in is not None:
                more.append(dec_in)
            if more:
                res["cpu_baseline"]["configs"] = oracle_small_configs(more)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
