"""Benchmark: effective attended TFLOP/s of the block-sparse attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one vsa_fwd (or jenga_fwd) call over the whole workload: every query block's
LUT/bitmap walk, selected K/V fetch, QK^T, masked online softmax, PV and the epilogue.
Metric = 4 * D * attended_pairs / step time, where attended_pairs counts the (query, key)
pairs the definition attends (keys masked by variable_block_sizes excluded, padding work
of the union-pair tiles not counted).

Reported on one JSON line:
  value      device-timed throughput, inputs resident in HBM, L2 flushed before each step
             (CUDA events on the launch stream around the kernel only; mean over the K
             steps), summed over ranks
  timing     the median of the same flushed steps, and the median of >= 20 back-to-back
             launches with L2 warm (no flush between them)
  e2e        the same metric through vsa_fwd_from_host: pinned host buffers, host->device
             copies of every input, the kernel and device->host copies of out and lse
  roofline   the forward kernel against the measured dense bf16 tensor peak
  cpu_baseline  the fp64 oracle on the host cores on a bounded sample of the workload
  clocks     nvidia-smi samples taken during the timed loop
--impl reference times the oracle itself (the only other place this file runs it).
Multi-GPU (torchrun): every rank runs an independent replica of the workload (weak
scaling, no collective on the data path); time = max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "vsa_long_video"  # the largest single-GPU workload


def attended_pairs(w) -> int:
    """Attended (query, key) pairs of a workload: per query block, the distinct in-range
    selected key blocks (counts clamped to [0, max_kv]) times their valid key counts,
    times the block's query rows."""
    if w.kind == "jenga":
        return int(w.bitmap.astype(bool).sum()) * w.block * w.block * w.B * w.H
    nb = w.nbk
    vbs = np.clip(w.vbs.astype(np.int64), 0, w.block)
    n = np.clip(w.q2k_num.astype(np.int64), 0, w.max_kv)
    total = 0
    idx = w.q2k_idx.reshape(-1, w.max_kv).astype(np.int64)
    n = n.reshape(-1)
    valid_slot = np.arange(w.max_kv)[None, :] < n[:, None]
    in_range = (idx >= 0) & (idx < nb)
    ok = valid_slot & in_range
    rows = np.repeat(np.arange(idx.shape[0]), w.max_kv)[ok.ravel()]
    blocks = idx.ravel()[ok.ravel()]
    uniq = np.unique(rows * nb + blocks)
    total = int(vbs[uniq % nb].sum()) * w.block
    return total


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}, "fallback"


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) while the timed loop runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, dist, device=None) -> float:
    """Largest value of ``x`` over all ranks (x itself without a process group); the
    tensor lives on ``device`` (CUDA for NCCL, CPU for gloo)."""
    if dist is None or not dist.is_initialized():
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample(w, budget_s: float, seed: int = 0):
    """Time the oracle on whole query blocks, head-major order from a seeded shuffle,
    adding blocks until about ``budget_s`` seconds of CPU work; returns
    (pairs, seconds, n_blocks, threads)."""
    from oracle import oracle as orc
    from block_sparse_attention_vsa_gb300 import workloads
    qb, kb, vb = workloads.bits(w.q), workloads.bits(w.k), workloads.bits(w.v)
    h = orc.load()
    threads = orc.num_threads(h)
    allsel = orc.all_qblocks(w.B, w.H, w.nbq)
    rng = np.random.default_rng(seed)
    order = allsel[rng.permutation(len(allsel))]
    if w.kind == "vsa":
        mask = orc.lut_to_blockmask(w.q2k_idx, w.q2k_num, w.nbk, h=h)
    else:
        mask = w.bitmap
    vbs = w.vbs if w.kind == "vsa" else None

    def pairs_of(sel):
        tot = 0
        for (b, hh, q) in sel:
            row = mask[q] if mask.ndim == 2 else mask[b, hh, q]
            vv = np.full(w.nbk, w.block) if vbs is None else np.clip(vbs, 0, w.block)
            tot += int(vv[row != 0].sum()) * w.block
        return tot

    n = max(1, threads)
    spent, pairs, used = 0.0, 0, 0
    while used < len(order) and spent < budget_s:
        sel = order[used:used + n]
        t0 = time.perf_counter()
        orc.masked_attention(qb, kb, vb, mask, w.block, w.scale, vbs=vbs, sel=sel, h=h)
        spent += time.perf_counter() - t0
        pairs += pairs_of(sel)
        used += len(sel)
        n = min(len(order) - used, n * 2)
    return pairs, spent, used, threads


def oracle_bwd_sample(w, budget_s: float):
    """Time the oracle backward on the first query blocks of the first heads (all of their
    keys), doubling the slice until about ``budget_s`` seconds.  The oracle runs its key/value
    heads in parallel, so the sample takes as many heads as it has threads (at most H);
    returns (pairs, seconds, n_blocks per head, threads used, heads)."""
    import torch
    from oracle import oracle as orc
    from block_sparse_attention_vsa_gb300 import workloads
    h = orc.load()
    nh = max(1, min(orc.num_threads(h), w.Hkv, w.H))
    kb = workloads.bits(w.k[:1, :nh])
    vb = workloads.bits(w.v[:1, :nh])
    g = torch.Generator().manual_seed(1)
    n, spent, pairs, used = 1, 0.0, 0, 0
    vv = np.clip(w.vbs, 0, w.block)
    while n <= w.nbq:
        rows = n * w.block
        qb = workloads.bits(w.q[:1, :nh, :rows])
        dob = workloads.bits(torch.randn((1, nh, rows, w.D), generator=g).to(torch.bfloat16))
        idx = np.ascontiguousarray(w.q2k_idx[:1, :nh, :n])
        num = np.ascontiguousarray(w.q2k_num[:1, :nh, :n])
        t0 = time.perf_counter()
        orc.vsa_backward(qb, kb, vb, dob, idx, num, w.vbs, w.block, w.scale, h=h)
        spent = time.perf_counter() - t0
        mask = orc.lut_to_blockmask(idx, num, w.nbk, h=h)[0]
        pairs = int(sum(int(vv[r != 0].sum()) for hm in mask for r in hm)) * w.block
        used = n
        if spent >= budget_s / 2 or n == w.nbq:
            break
        n = min(w.nbq, n * 2)
    return pairs, spent, used, nh, nh


def run_reference(args, w, pairs_total, flop_per_pair):
    """The oracle on the host cores: each step is a bounded sample of the workload."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, per_step / 4, seed=1)
    tot_p, tot_t, tot_blocks, threads = 0, 0.0, 0, 1
    for s in range(args.steps):
        p, t, nblk, threads = oracle_sample(w, per_step, seed=100 + s)
        tot_p, tot_t, tot_blocks = tot_p + p, tot_t + t, tot_blocks + nblk
    value = tot_p * flop_per_pair / tot_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, pairs_total),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{tot_blocks} query blocks of {w.name} over {args.steps} steps"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "effective attended TFLOP/s (4*d*pairs) and % of GB300 bf16 TC peak"
METRIC_BWD = "backward: effective attended TFLOP/s (10*d*pairs) and % of GB300 bf16 TC peak"


def config_of(w, pairs):
    c = {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D, "block": w.block,
         "attended_pairs": pairs, "l2": "flushed (256 MiB write) before every timed step"}
    if w.Sk != w.S or w.Hkv != w.H:
        c.update({"Hkv": w.Hkv, "Sk": w.Sk})
    if w.extra.get("num_splits"):
        c["num_splits"] = w.extra["num_splits"]
    if w.kind == "vsa":
        c["max_kv"] = w.max_kv
    else:
        c["bitmap"] = list(w.bitmap.shape)
    return c


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--pass", dest="pass_", default="fwd", choices=["fwd", "bwd"],
                    help="bwd times vsa_bwd (dq, dk, dv) on the workload instead")
    ap.add_argument("--heads", type=int, default=0,
                    help="time only the first N heads of the workload (a smaller case of the "
                         "same per-head structure, for profiler captures)")
    args = ap.parse_args()

    import torch
    from block_sparse_attention_vsa_gb300 import workloads

    ws, rank, local = dist_env()
    w = workloads.make(args.workload, seed=0)
    if args.heads:
        w = workloads.first_heads(w, args.heads)
    pairs = attended_pairs(w)
    bwd = args.pass_ == "bwd"
    if bwd and w.kind != "vsa":
        raise SystemExit("--pass bwd needs a LUT (vsa_*) workload")
    # forward: QK^T and PV (2d each); backward: S recomputed, dP, dV, dK, dQ (2d each)
    flop_per_pair = (10 if bwd else 4) * w.D

    if args.impl == "reference":
        if ws > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        run_reference(args, w, pairs, flop_per_pair)
        if ws > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    import __graft_entry__
    __graft_entry__.build()
    from block_sparse_attention_vsa_gb300 import binding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()

    q, k, v = (t.to(dev) for t in (w.q, w.k, w.v))
    if w.kind == "vsa":
        idx = torch.from_numpy(w.q2k_idx).to(dev)
        num = torch.from_numpy(w.q2k_num).to(dev)
        vbs = torch.from_numpy(w.vbs).to(dev)
    else:
        bm = torch.from_numpy(w.bitmap).to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    wsbuf = binding.new_workspace(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    split = w.kind == "vsa" and (w.Sk != w.S or w.Hkv != w.H)  # the split-KV route
    if split:
        n_split = binding.default_splits(w.B, w.H, w.S, w.block,
                                         torch.cuda.get_device_properties(dev).multi_processor_count)
        w.extra["num_splits"] = n_split
        wsbuf = binding.new_split_workspace(w.B, w.H, w.S, w.block, n_split, dev)

    if bwd:
        out, lse = binding.vsa_fwd_gqa(q, k, v, idx, num, vbs, block=w.block, scale=w.scale)
        gen = torch.Generator().manual_seed(1)
        dout = torch.randn(w.q.shape, generator=gen).to(torch.bfloat16).to(dev)
        bws = torch.empty(binding.load().vsa_bwd_workspace_bytes(w.B, w.H, w.S, w.Sk, w.block),
                          dtype=torch.uint8, device=dev)

    def step():
        if bwd:
            binding.vsa_bwd(q, k, v, out, dout, lse, idx, num, vbs, block=w.block,
                            scale=w.scale, workspace=bws, stream=stream)
        elif split:
            binding.vsa_fwd_split(q, k, v, idx, num, vbs, block=w.block, scale=w.scale,
                                  num_splits=n_split, out=out, lse=lse, workspace=wsbuf,
                                  stream=stream)
        elif w.kind == "vsa":
            binding.vsa_fwd(q, k, v, idx, num, vbs, block=w.block, scale=w.scale, out=out,
                            lse=lse, workspace=wsbuf, stream=stream)
        else:
            binding.jenga_fwd(q, k, v, bm, w.block, w.block, scale=w.scale, out=out, lse=lse,
                              workspace=wsbuf, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    code, detail = binding.vsa_device_status()
    if code != binding.VSA_OK:
        raise RuntimeError(f"device status {code} detail {detail:#x} after warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    n_warm = max(20, args.steps)
    wstarts = [torch.cuda.Event(enable_timing=True) for _ in range(n_warm)]
    wends = [torch.cuda.Event(enable_timing=True) for _ in range(n_warm)]
    launches = 0
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
            launches += binding.vsa_last_launch_count()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        # warm L2: back-to-back launches, outside the K timed steps (the sampler keeps
        # running so the clock record covers both loops)
        for i in range(n_warm):
            wstarts[i].record(stream)
            step()
            wends[i].record(stream)
        torch.cuda.synchronize()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    wtimes = [s.elapsed_time(e) for s, e in zip(wstarts, wends)]
    ms = max_over_ranks(sum(times) / len(times), dist, dev)
    ms_med = max_over_ranks(statistics.median(times), dist, dev)
    ms_warm = max_over_ranks(statistics.median(wtimes), dist, dev)
    code, detail = binding.vsa_device_status()
    if code != binding.VSA_OK:
        raise RuntimeError(f"device status {code} detail {detail:#x} after timing")
    value = ws * pairs * flop_per_pair / (ms * 1e-3) / 1e12

    # ---- end to end through the host-buffer entry point (VSA workloads)
    e2e = None
    if bwd:
        pass  # the host-buffer leg belongs to the forward line
    elif split and args.e2e_steps > 0:
        # host buffers through the Python binding: copies in, split forward, copies out
        h = dict(q=w.q.pin_memory(), k=w.k.pin_memory(), v=w.v.pin_memory(),
                 idx=torch.from_numpy(w.q2k_idx).pin_memory(),
                 num=torch.from_numpy(w.q2k_num).pin_memory(),
                 vbs=torch.from_numpy(w.vbs).pin_memory())
        d = dict(q=q, k=k, v=v, idx=idx, num=num, vbs=vbs)
        h_out = torch.empty_like(w.q).pin_memory()
        h_lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in h.values())
        d2h = h_out.numel() * 2 + h_lse.numel() * 4

        def e2e_step():
            for key in d:
                d[key].copy_(h[key], non_blocking=True)
            step()
            h_out.copy_(out, non_blocking=True)
            h_lse.copy_(lse, non_blocking=True)
            stream.synchronize()

        for _ in range(2):
            e2e_step()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            e2e_step()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) / args.e2e_steps * 1e3, dist, dev)
        e2e = {"value": ws * pairs * flop_per_pair / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    elif w.kind == "vsa" and args.e2e_steps > 0:
        h = dict(q=w.q.pin_memory(), k=w.k.pin_memory(), v=w.v.pin_memory(),
                 idx=torch.from_numpy(w.q2k_idx).pin_memory(),
                 num=torch.from_numpy(w.q2k_num).pin_memory(),
                 vbs=torch.from_numpy(w.vbs).pin_memory())
        h_out = torch.empty_like(w.q).pin_memory()
        h_lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32).pin_memory()
        bufs = dict(q=q, k=k, v=v, idx=idx, num=num, vbs=vbs, out=out, lse=lse)
        h2d = sum(t.numel() * t.element_size() for t in h.values())
        d2h = h_out.numel() * 2 + h_lse.numel() * 4
        for _ in range(2):
            binding.vsa_fwd_from_host(h["q"], h["k"], h["v"], h["idx"], h["num"], h["vbs"],
                                      w.block, w.scale, h_out, h_lse, bufs, workspace=wsbuf,
                                      stream=stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            binding.vsa_fwd_from_host(h["q"], h["k"], h["v"], h["idx"], h["num"], h["vbs"],
                                      w.block, w.scale, h_out, h_lse, bufs, workspace=wsbuf,
                                      stream=stream)
            stream.synchronize()
        e2e_ms = max_over_ranks((time.perf_counter() - t0) / args.e2e_steps * 1e3, dist, dev)
        e2e = {"value": ws * pairs * flop_per_pair / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])
    achieved = pairs * flop_per_pair / (ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": TRAFFIC.get(w.name),
                "peak_source": f"{peak_src} dense bf16 (burst)",
                "kernel": f"bsa_bwd_kernel<{w.block}> (whole vsa_bwd call timed)" if bwd
                          else "bsa_fwd_kernel"}
    if bwd:
        roofline["traffic"] = TRAFFIC_BWD.get(w.name)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and bwd:
        p, t, nblk, threads, nh = oracle_bwd_sample(w, 15.0)
        cpu = {"value": p * flop_per_pair / t / 1e12, "unit": "TFLOP/s", "cores": threads,
               "kind": "oracle",
               "sample": f"backward of query blocks 0..{nblk - 1} of heads 0..{nh - 1} of "
                         f"{w.name} against all their keys ({p} attended pairs, {t:.1f} s)"}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and not bwd:
        p, t, nblk, threads = oracle_sample(w, 15.0)
        whole = nblk == w.B * w.H * w.nbq
        cpu = {"value": p * flop_per_pair / t / 1e12, "unit": "TFLOP/s", "cores": threads,
               "kind": "oracle",
               "sample": f"{nblk} of {w.B * w.H * w.nbq} query blocks of {w.name} "
                         f"({p} attended pairs, {t:.1f} s)"
                         + ("" if whole else "; extrapolated per attended pair")}

    if rank == 0:
        line = {
            "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, shapes of the workload)",
            "config": config_of(w, pairs), "e2e": e2e, "gpu_launches": launches,
            "roofline": roofline, "cpu_baseline": cpu, "clocks": clk.summary(),
            "pct_of_peak": 100.0 * achieved / peak,
            "timing": {
                "flushed_median_ms": ms_med,
                "flushed_median_value": ws * pairs * flop_per_pair / (ms_med * 1e-3) / 1e12,
                "warm_l2_median_ms": ms_warm,
                "warm_l2_median_value": ws * pairs * flop_per_pair / (ms_warm * 1e-3) / 1e12,
                "warm_l2_launches": n_warm, "unit": "TFLOP/s"},
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# DRAM bytes (read + write) per launch of the forward kernel, from an ncu capture of the
# same kernel build on the same workload; absent = not measured for the current kernel.
TRAFFIC = {"vsa_long_video": 2454.0e6,  # captured on 4 of 24 heads, scaled by 6
           "jenga": 384.6e6, "vsa_mid": 182.7e6, "vsa_blk128": 1610.7e6}
# the same for the backward kernel (bsa_bwd_kernel<64> or <128>)
TRAFFIC_BWD = {"vsa_mid": 456.6e6,
               "vsa_blk128": 3916.4e6,  # captured on 8 of 24 heads, scaled by 3
               "vsa_long_video": 13593.1e6}  # captured on 4 of 24 heads, scaled by 6


if __name__ == "__main__":
    main()
