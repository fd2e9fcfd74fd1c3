#!/usr/bin/env python
"""Benchmark of the cross-model attention-map reuse hot path on one GB300.

Workload (default, the largest configuration): 16 packed sequences with
lengths ~ U[1024, 8192] (81,514 tokens), one 40-layer, 40-head sender
(d = 128, bf16, B = 64, p = 0.95) whose state is compressed once and consumed
by two receivers: (a) 36 layers, 32 query / 8 KV heads, recomputing its first
4 layers and reusing layers 5..36 through m(j) = round(j * 40 / 36), and
(b) 26 layers, 24 query / 8 KV heads, r = 3, m(j) = round(j * 40 / 26).

One step = the whole hot path over that batch, streamed per sender layer
(40 sender layers of kept tiles would not fit any device): for each sender
layer, compress it (statistics, top-p, BSR pack), run the fused retrieval
of every receiver layer of both receivers that maps to it, release it.
Inputs are seeded synthetic tensors (no model weights or datasets) drawn on
the device and resident in HBM before the timed region; every per-layer BSR
(~16 GB) and every layer's Q/K (1.7 GB) is far larger than L2.

Printed JSON (one line, rank 0):
  value       retrieval GB/s: algorithmic bytes of the step's retrieval
              launches / their summed device time (CUDA events per launch)
  compressor  tokens/s of the compressor and its Q.K^T tensor fraction
  roofline    the dominant kernel (largest device time in the step) against
              MEASURED_PEAKS.json; `rooflines` has all three hot kernels
  e2e         the same metrics through the public API with host buffers:
              every step's host->device copies of Q/K/V/W and device->host
              copies of every O inside the timed region
  workloads   the 32-layer N = 16384 workload and the N = 32768, B = 128
              density sweep (p = 0.80/0.90/0.95/0.99), measured in this run
  residency   a compressed layer fetched back from host memory while other
              layers are compressed and retrieved (copy hidden or not)
  cpu_baseline  the fp64 oracle on a bounded sample, host cores

`--impl reference` times the oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from cross_model_attention_gb300 import synth, workloads  # noqa: E402
from cross_model_attention_gb300.accounting import (  # noqa: E402
    candidate_blocks, pack_bytes, qk_flops, retrieval_bytes, union_blocks)

METRIC = "retrieval GB/s & % HBM roofline; compressor tokens/s & % tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DEFAULT_WORKLOAD = 4


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return json.load(fh), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def traffic_for(kernel: str, alg_bytes: float, max_blocks: int = 0):
    """DRAM bytes of one launch from the committed ncu summary, if it was
    taken on the current source of that kernel, else None.  The capture is
    of a smaller launch; its traffic is scaled by the ratio of algorithmic
    bytes (the traffic of these kernels grows in proportion to the tiles
    they move).  The statistics step runs the two-CTAs-per-SM kernel when no
    row has more than 128 candidate blocks (`max_blocks`), the one-CTA kernel
    otherwise."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    stats_src = "mf_stats2_tc.cu" if max_blocks <= 128 else "mf_stats_tc.cu"
    src = {"stats": stats_src, "pack": "mf_pack_tc.cu", "retrieve": "mf_retrieve_team.cu"}[kernel]
    with open(os.path.join(ROOT, "cross_model_attention_gb300", "csrc", src), "rb") as fh:
        sha = hashlib.sha256(fh.read()).hexdigest()[:16]
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == sha:
            return float(parts[2]) * alg_bytes / float(parts[3])
    return None


def host_budget_bytes() -> int:
    """A share of the host memory this process may still use (the smaller of
    MemAvailable and the cgroup's remaining limit), at most 24 GiB, for pinned
    buffers."""
    avail = None
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                avail = int(line.split()[1]) * 1024
    except OSError:
        pass
    try:
        lim = open("/sys/fs/cgroup/memory.max").read().strip()
        cur = int(open("/sys/fs/cgroup/memory.current").read().strip())
        if lim != "max":
            cg = int(lim) - cur
            avail = cg if avail is None else min(avail, cg)
    except (OSError, ValueError):
        pass
    return int(min(24 << 30, 0.35 * (avail if avail is not None else 16 << 30)))


def link_bandwidth(nbytes: int = 256 << 20, reps: int = 4):
    """Host<->device copy bandwidth (GB/s) of one pinned buffer: the host
    link is shared with other jobs on the machine and varies from run to
    run, so it is taken around every end-to-end repetition."""
    import torch
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    out = {}
    for name, f in (("h2d", lambda: dev.copy_(host, non_blocking=True)),
                    ("d2h", lambda: host.copy_(dev, non_blocking=True))):
        f()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            f()
        e1.record(s)
        torch.cuda.synchronize()
        out[name] = round(reps * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9, 1)
    return out


# -------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int = 0):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ CPU leg ----

def host_layer(w, layer: int):
    """One sender layer's Q/K and the first reuse layer's V and W of the
    first receiver, drawn on the host (numpy), as fp64 arrays."""
    x = synth.sender_qk(w, layer)
    rcv = w.receivers[0]
    j = rcv.layer_map(w.sender_layers)[0][0]
    return x["q64"], x["k64"], synth.receiver_v(w, rcv, j)["v64"], \
        synth.head_map_weights(w, rcv, j).astype(np.float64)


def oracle_sample(w, q64, k64, v64, W, budget_rows: int, heads: int, seed: int = 0):
    """Time the oracle on a bounded sample of the workload: the compressor on
    `heads` heads of one sender layer, and the retrieval of `budget_rows`
    block-rows of one reuse layer of the first receiver (all sender heads,
    every receiver head).  Returns per-unit throughputs."""
    from oracle import mapflow_oracle as orc
    rcv = w.receivers[0]
    p = w.p[0]
    t0 = time.perf_counter()
    bsr = orc.compress(q64[:, :heads], k64[:, :heads], w.cu_seqlens, w.B, p, True,
                       keep_tiles=False)
    t_comp = time.perf_counter() - t0
    grid = bsr.grid
    rng = np.random.default_rng(seed)
    rows = sorted(int(x) for x in rng.choice(grid.R, size=min(budget_rows, grid.R), replace=False))
    kept = {}  # the oracle's own selection on the sampled rows (untimed)
    for h in range(w.sender_heads):
        for rb in rows:
            kept[(h, rb)] = orc.select_topp(orc.block_row_reference(q64, k64, grid, h, rb)["mass"], p)
    t0 = time.perf_counter()
    nbytes = 0.0
    for rb in rows:
        orc.retrieve_block_row(q64, k64, grid, lambda h, r: kept[(h, r)], W, v64, rcv.kv_heads, rb)
        nk = sum(len(kept[(h, rb)]) for h in range(w.sender_heads))
        nrow = min(w.B, int(grid.lens[grid.rb_seq[rb]]) - int(grid.rb_local[rb]) * w.B)
        nbytes += nk * (2 * w.B * w.B + 4) + 2 * nrow * (rcv.heads + rcv.kv_heads) * w.d
    t_ret = time.perf_counter() - t0
    return {
        "retrieval_gbs": nbytes / t_ret / 1e9,
        "compressor_tokens_per_s": w.T * heads / w.sender_heads / t_comp,
        "seconds": t_comp + t_ret,
        "sample": (f"oracle compressor on {heads}/{w.sender_heads} heads of one sender layer "
                   f"(T={w.T}); oracle retrieval of {len(rows)}/{grid.R} block-rows of one reuse "
                   f"layer of receiver {rcv.name} (all {w.sender_heads} sender heads, {rcv.heads} "
                   f"receiver heads)"),
    }


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    w = workloads.get(args.workload)
    q64, k64, v64, W = host_layer(w, 1)
    for i in range(args.warmup):
        oracle_sample(w, q64, k64, v64, W, budget_rows=args.ref_rows, heads=1, seed=100 + i)
    vals, comps = [], []
    t0 = time.perf_counter()
    for i in range(args.steps):
        r = oracle_sample(w, q64, k64, v64, W, budget_rows=args.ref_rows, heads=1, seed=i)
        vals.append(r["retrieval_gbs"])
        comps.append(r["compressor_tokens_per_s"])
        sample = r["sample"]
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    cores = os.cpu_count()
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(w, world),
        "compressor": {"tokens_per_s": statistics.median(comps)},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def job_times(local_times, world: int, device):
    """Per-quantity maximum over the ranks: the slowest replica sets the job
    time (each rank runs the whole workload on its own GPU; no data path
    between ranks)."""
    import torch
    t = torch.tensor(list(local_times), dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(units_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job throughput of `world` replicas that each processed
    `units_per_rank` in the job time `seconds` (weak scaling)."""
    return units_per_rank * world / seconds


def config_dict(w, world):
    rc = [{"name": r.name, "layers": r.layers, "heads": r.heads, "kv_heads": r.kv_heads,
           "recompute_r": r.recompute, "reuse_layers": r.layers - r.recompute}
          for r in w.receivers]
    return {"workload": f"workload {w.index}: {w.name}", "sequences": len(w.seqlens),
            "tokens": w.T, "sender_layers": w.sender_layers, "sender_heads": w.sender_heads,
            "sender_kv_heads": w.sender_kv_heads, "receivers": rc, "d": w.d, "B": w.B,
            "p": w.p[0], "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "streaming": "per sender layer: compress, retrieve every receiver layer mapped "
                         "to it, release",
            "l2": "inputs larger than L2 (each layer's Q/K and kept tiles are GBs)"}


# ------------------------------------------------------------ GPU leg ----

class DeviceWorkload:
    """Every input of one workload resident on the device: Q/K of each sender
    layer, V, W and an output buffer of each reuse layer of each receiver."""

    def __init__(self, w, dev, layers=None):
        import torch
        self.w = w
        self.layers = list(range(1, w.sender_layers + 1)) if layers is None else list(layers)
        self.q, self.k = {}, {}
        for l in self.layers:
            self.q[l], self.k[l] = synth.sender_qk_device(w, l, dev)
        self.reuse = [(ri, j, m) for ri, rcv in enumerate(w.receivers)
                      for j, m in rcv.layer_map(w.sender_layers) if m in self.q]
        self.by_layer = {l: [(ri, j) for ri, j, m in self.reuse if m == l] for l in self.layers}
        self.v, self.W, self.o = {}, {}, {}
        for ri, j, m in self.reuse:
            rcv = w.receivers[ri]
            self.v[ri, j] = synth.receiver_v_device(w, rcv, j, dev)[None]
            self.W[ri, j] = torch.from_numpy(synth.head_map_weights(w, rcv, j))[None].to(dev)
            self.o[ri, j] = torch.empty((1, w.T, rcv.heads, w.d), dtype=self.v[ri, j].dtype,
                                        device=dev)
        torch.cuda.synchronize()


def streamed_step(bsr, D, p, waits=None):
    """One step, streamed per sender layer through two BSR slots."""
    for l in D.layers:
        slot = l % 2
        if waits is not None:
            waits("qk", l)
        bsr.compress(slot, D.q[l], D.k[l], p)
        for key in D.by_layer[l]:
            if waits is not None:
                waits("v", key)
            bsr.retrieve(D.W[key], D.v[key], D.o[key], [slot])
            if waits is not None:
                waits("o", key)
        bsr.release_layer(slot)


def structure_pass(bsr, D, p):
    """Untimed pass that records each sender layer's kept tiles (nnz) and the
    union of kept blocks over heads (for the retrieval's tensor work)."""
    w = D.w
    R = sum((L + w.B - 1) // w.B for L in w.seqlens)
    nnz, U = {}, {}
    for l in D.layers:
        slot = l % 2
        bsr.compress(slot, D.q[l], D.k[l], p)
        nnz[l] = bsr.info(slot)[0]
        U[l] = union_blocks(*bsr.structure(slot), w.sender_heads, R)
        bsr.release_layer(slot)
    return nnz, U


def accounting_of(w, D, nnz, U):
    rcvs = w.receivers
    ret_bytes = sum(retrieval_bytes(w, rcvs[ri], nnz[m]) for ri, j, m in D.reuse)
    ret_flops = sum(2.0 * w.B * w.B * w.d * U[m] * rcvs[ri].heads
                    + 2.0 * w.B * w.B * rcvs[ri].heads * nnz[m] for ri, j, m in D.reuse)
    comp_flops = qk_flops(w) * len(D.layers)
    pk_bytes = sum(pack_bytes(w, nnz[l]) for l in D.layers)
    return ret_bytes, ret_flops, comp_flops, pk_bytes


def rooflines_of(w, prof, n_layers, ret_bytes, comp_flops, pk_bytes, peaks, label, long_step):
    hbm = float(peaks["hbm_gbs"])
    burst = float(peaks["bf16_tflops"])
    sus = float(peaks.get("bf16_tflops_sustained", burst))
    # a kernel timed inside a long step (hundreds of ms of back-to-back
    # launches, under the power cap) is held to the sustained peak, a kernel
    # timed alone to the burst peak; both fractions are reported
    tf, tf_name = (sus, "bf16_tflops_sustained") if long_step else (burst, "bf16_tflops")
    max_blocks = max(-(-L // w.B) for L in w.seqlens)
    out = {}
    n, ms = prof["stats"]
    per = ms / max(n, 1) / 1e3
    ach = comp_flops / n_layers / per / 1e12
    out["stats"] = {"bound": "tensor", "achieved": ach, "peak": tf, "unit": "TFLOP/s",
                    "frac": ach / tf, "frac_of_sustained": ach / sus, "frac_of_burst": ach / burst,
                    "traffic": traffic_for("stats", 2.0 * w.T * (w.sender_heads + w.sender_kv_heads)
                                           * w.d, max_blocks),
                    "launches": n, "ms_per_launch": per * 1e3, "peak_source": f"{tf_name} ({label})"}
    for kind, total in (("pack", pk_bytes), ("retrieve", ret_bytes)):
        n, ms = prof[kind]
        per = ms / max(n, 1) / 1e3
        alg = total / max(n, 1)
        ach = alg / per / 1e9
        out[kind] = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                     "frac": ach / hbm, "traffic": traffic_for(kind, alg), "launches": n,
                     "ms_per_launch": per * 1e3, "algorithmic_bytes_per_launch": alg,
                     "frac_of_8TBs_nominal": ach / 8000.0, "peak_source": f"hbm_gbs ({label})"}
    return out


def measure_streamed(mapflow, D, steps, warmup, world, dev, peaks, label, clocks=True):
    """Warm-up, structure pass, then `steps` timed steps with per-launch
    events; returns the measurement dict (device-resident inputs)."""
    import torch
    w = D.w
    p = w.p[0]
    bsr = mapflow.BSR(2, w.T, w.sender_heads, w.B, w.cu_seqlens)
    nnz, U = structure_pass(bsr, D, p)
    for _ in range(warmup):
        streamed_step(bsr, D, p)
    bsr.device_status()
    ret_bytes, ret_flops, comp_flops, pk_bytes = accounting_of(w, D, nnz, U)
    stream = torch.cuda.current_stream()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device()) if clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    bsr.profile(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.perf_counter()
    e0.record(stream)
    for _ in range(steps):
        streamed_step(bsr, D, p)
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    clk = sampler.stop() if sampler else None
    bsr.device_status()
    prof = bsr.profile_read()
    bsr.profile(False)
    bsr.close()
    t_step = e0.elapsed_time(e1) / 1e3
    t_ret = prof["retrieve"][1] / 1e3
    t_comp = sum(prof[k][1] for k in ("stats", "select", "scan", "pack", "union")) / 1e3
    t_step, t_ret, t_comp = job_times([t_step, t_ret, t_comp], world, dev)
    K = steps
    roofs = rooflines_of(w, prof, len(D.layers) * K, ret_bytes * K, comp_flops * K,
                         pk_bytes * K, peaks, label, True)
    tf_sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    n_cand = w.sender_heads * candidate_blocks(w)
    ret_tensor_frac = ret_flops * K / t_ret / (tf_sus * 1e12)
    res = {
        "retrieval_gbs": job_throughput(ret_bytes * K, world, t_ret) / 1e9,
        "compressor_tokens_per_s": job_throughput(w.T * len(D.layers) * K, world, t_comp),
        "ms_per_step": 1e3 * t_step / K,
        "retrieval_ms_per_step": 1e3 * t_ret / K,
        "compressor_ms_per_step": 1e3 * t_comp / K,
        "retrieval_bytes_per_step": ret_bytes,
        "retrieval_tensor_flops_per_step": ret_flops,
        "retrieval_tensor_frac_of_sustained": ret_tensor_frac,
        "retrieval_binds": "hbm" if roofs["retrieve"]["frac"] >= ret_tensor_frac else "tensor",
        "kept_fraction": float(np.mean([nnz[l] for l in D.layers])) / n_cand,
        "pack_bytes_written_per_step": float(sum(nnz[l] * (2 * w.B * w.B + 4) for l in D.layers)),
        # the pack recomputes the kept tiles' Q.K^T (reported apart from the
        # one causal pass the statistics kernel is held to)
        "pack_recompute_tflops": float(sum(2 * w.d * w.B * w.B * nnz[l] for l in D.layers)) * K
        / (prof["pack"][1] / 1e3) / 1e12,
        "exp2_per_s": float(sum(L * (L + 1) // 2 for L in w.seqlens)) * w.sender_heads
        * len(D.layers) * K * world / t_comp,
        "rooflines": roofs,
        "launches_per_step": {k: v[0] // K for k, v in prof.items()},
        "clocks": clk, "wall_s_timed": t_wall,
    }
    return res, nnz, U


def overlap_probe(torch, bsr, D, p, qhost, comp, h2d):
    """One input copy (a layer's Q from the leg's own pinned buffer) alone,
    one layer's compression alone, and both at once on their two streams:
    where copies and kernels overlap, `both` is near the larger of the two,
    where they do not, near their sum."""
    l0 = D.layers[0]

    def run(copy, kernel):
        e0 = torch.cuda.Event(enable_timing=True)
        ec = torch.cuda.Event(enable_timing=True)
        ek = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(comp)
        h2d.wait_event(e0)
        if copy:
            with torch.cuda.stream(h2d):
                D.q[l0].copy_(qhost, non_blocking=True)
        ec.record(h2d)
        if kernel:
            bsr.compress(0, D.q[l0], D.k[l0], p)
        ek.record(comp)
        torch.cuda.synchronize()
        return max(e0.elapsed_time(ec), e0.elapsed_time(ek))

    run(True, True)
    t_copy = statistics.median([run(True, False) for _ in range(3)])
    t_kern = statistics.median([run(False, True) for _ in range(3)])
    t_both = statistics.median([run(True, True) for _ in range(3)])
    bsr.release_layer(0)
    return {"copy_ms": round(t_copy, 3), "copy_gbs": round(qhost.numel() * qhost.element_size()
                                                          / t_copy / 1e6, 1),
            "compress_ms": round(t_kern, 3), "both_ms": round(t_both, 3)}


def measure_e2e(mapflow, D, nnz, reps, peaks):
    """The same streamed step through the public API with host buffers: every
    step copies each layer's Q/K and each reuse layer's V and W from pinned
    host memory to the device and each O back, inside the timed region.
    Copies run on two copy streams (one per direction), layer by layer, so
    they overlap the neighbouring layers' kernels."""
    import torch
    w = D.w
    p = w.p[0]
    Ls = len(D.layers)
    budget = host_budget_bytes()
    qk_bytes = D.q[D.layers[0]].numel() * 2 + D.k[D.layers[0]].numel() * 2
    keys = [(ri, j) for ri, j, m in D.reuse]
    v_bytes = sum(D.v[k].numel() * 2 for k in keys)
    o_slot_bytes = max(D.o[k].numel() * 2 for k in keys)
    n_o = 4
    n_h = int(max(2, min(Ls, (budget - n_o * o_slot_bytes - min(v_bytes, budget // 4)) // qk_bytes)))
    n_v = len(keys) if v_bytes <= budget // 4 else max(2, int(budget // 4 // (v_bytes / len(keys))))
    # host copies: Q/K of the first n_h sender layers, cycled over the step's
    # layers (layer i carries host slot i mod n_h); V of the first n_v reuse
    # layers, cycled the same way; an O ring of n_o slots per output shape
    qh = [D.q[D.layers[i]].cpu().pin_memory() for i in range(n_h)]
    kh = [D.k[D.layers[i]].cpu().pin_memory() for i in range(n_h)]
    vh = [D.v[keys[i]].cpu().pin_memory() for i in range(n_v)]
    Wh = {k: D.W[k].cpu().pin_memory() for k in keys}
    oh = {}
    for k in keys:
        shape = tuple(D.o[k].shape)
        if shape not in oh:
            oh[shape] = [torch.empty(shape, dtype=D.o[k].dtype).pin_memory() for _ in range(n_o)]
    h2d = torch.cuda.Stream()
    d2h = torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    li = {l: i for i, l in enumerate(D.layers)}
    ki = {k: i for i, k in enumerate(keys)}
    ev_qk = {l: torch.cuda.Event() for l in D.layers}
    ev_v = {k: torch.cuda.Event() for k in keys}
    ev_o = {k: torch.cuda.Event() for k in keys}
    o_count = {}

    def issue_copies_in():
        h2d.wait_stream(comp)  # the previous step is done with the device buffers
        with torch.cuda.stream(h2d):
            for l in D.layers:
                i = li[l] % n_h
                D.q[l].copy_(qh[i], non_blocking=True)
                D.k[l].copy_(kh[i], non_blocking=True)
                ev_qk[l].record(h2d)
                for k in D.by_layer[l]:
                    D.v[k].copy_(vh[ki[k] % n_v], non_blocking=True)
                    D.W[k].copy_(Wh[k], non_blocking=True)
                    ev_v[k].record(h2d)

    def waits(kind, key):
        if kind == "qk":
            comp.wait_event(ev_qk[key])
        elif kind == "v":
            comp.wait_event(ev_v[key])
        else:
            ev_o[key].record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_o[key])
                ring = oh[tuple(D.o[key].shape)]
                c = o_count.get(ring[0].shape, 0)
                o_count[ring[0].shape] = c + 1
                ring[c % n_o].copy_(D.o[key], non_blocking=True)

    bsr = mapflow.BSR(2, w.T, w.sender_heads, w.B, w.cu_seqlens)
    # warm-up repetition, then the timed ones with per-launch events
    issue_copies_in()
    streamed_step(bsr, D, p, waits)
    torch.cuda.synchronize()
    bsr.device_status()
    overlap = overlap_probe(torch, bsr, D, p, qh[0], comp, h2d)
    steps, links = [], []
    host_ms = []
    for _ in range(reps):
        link_before = link_bandwidth()
        bsr.profile(True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        h0 = time.perf_counter()
        issue_copies_in()
        h1 = time.perf_counter()
        streamed_step(bsr, D, p, waits)
        d2h.wait_stream(comp)
        e1.record(d2h)
        h2 = time.perf_counter()
        torch.cuda.synchronize()
        # host time to enqueue the step's input copies and then its kernels and
        # output copies: milliseconds when the copies are asynchronous
        host_ms.append((round(1e3 * (h1 - h0), 2), round(1e3 * (h2 - h1), 2)))
        prof = bsr.profile_read()
        t = e0.elapsed_time(e1) / 1e3
        t_ret = prof["retrieve"][1] / 1e3
        t_comp = sum(prof[k][1] for k in ("stats", "select", "scan", "pack", "union")) / 1e3
        steps.append((t, t_ret, t_comp))
        links.append({"before": link_before, "after": link_bandwidth()})
    bsr.device_status()
    bsr.profile(False)
    bsr.close()
    # layer i of the step carried host slot i mod n_h: its kept tiles are
    # those of that sender layer (compression is deterministic)
    nnz_e = {l: nnz[D.layers[li[l] % n_h]] for l in D.layers}
    rcvs = w.receivers
    ret_bytes = sum(retrieval_bytes(w, rcvs[ri], nnz_e[m]) for ri, j, m in D.reuse)
    h2d_b = sum((D.q[l].numel() + D.k[l].numel()) * 2 for l in D.layers) + \
        sum(D.v[k].numel() * 2 + D.W[k].numel() * 4 for k in keys)
    d2h_b = sum(D.o[k].numel() * 2 for k in keys)
    # each leg's end-to-end time: the step's end-to-end time minus the other
    # leg's kernel time (copy stalls count against both legs)
    ret_gbs = [ret_bytes / (t - tc) / 1e9 for t, tr, tc in steps]
    comp_tps = [w.T * Ls / (t - tr) for t, tr, tc in steps]
    return {"value": statistics.median(ret_gbs), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d_b), "d2h_bytes_per_step": int(d2h_b),
            "compressor_tokens_per_s": statistics.median(comp_tps),
            "ms_per_step": 1e3 * statistics.median([s[0] for s in steps]),
            "reps": {"retrieval_gbs": [round(x, 1) for x in ret_gbs],
                     "compressor_tokens_per_s": [round(x) for x in comp_tps],
                     "ms_per_step": [round(1e3 * s[0], 2) for s in steps],
                     # kernel time inside the end-to-end step (per-launch events)
                     "retrieval_kernel_ms": [round(1e3 * s[1], 2) for s in steps],
                     "compressor_kernel_ms": [round(1e3 * s[2], 2) for s in steps]},
            "spread": {"retrieval_gbs_min": min(ret_gbs), "retrieval_gbs_max": max(ret_gbs)},
            "link_gbs": links,
            "host_enqueue_ms": {"copies_in": [x[0] for x in host_ms],
                                "kernels_and_copies_out": [x[1] for x in host_ms]},
            "overlap_probe": overlap,
            "host_buffers_pinned": bool(all(t.is_pinned() for t in qh + kh + vh)
                                        and all(t.is_pinned() for r in oh.values() for t in r)),
            "host_slots": {"qk_layers_distinct": n_h, "v_layers_distinct": n_v,
                           "o_ring": n_o,
                           "note": "step layer i copies host slot i mod n (host memory bound)"},
            "definition": "each leg's e2e time = the step's end-to-end time (copies in and "
                          "out included) minus the other leg's kernel time"}


def measure_residency(mapflow, D, peaks, reps=3):
    """A compressed sender layer is moved to host memory and fetched back on a
    copy stream while the compute stream compresses and retrieves other
    sender layers (the receiver's own recompute of its first layers stands
    behind this on the pages).  t_copy: the fetch alone; t_compute: the
    compute alone; t_both: both at once; hidden = 1 - (t_both - t_compute) /
    t_copy."""
    import torch
    w = D.w
    p = w.p[0]
    L0 = D.layers[0]
    held = mapflow.BSR(1, w.T, w.sender_heads, w.B, w.cu_seqlens)
    held.compress(0, D.q[L0], D.k[L0], p)
    nnz0 = held.info(0)[0]
    layer_bytes = nnz0 * (2 * w.B * w.B + 4)
    if layer_bytes > host_budget_bytes():
        held.close()
        return {"skipped": f"a layer's {layer_bytes / 1e9:.1f} GB of tiles exceeds the host budget"}
    held.offload(0)
    torch.cuda.synchronize()
    comp = torch.cuda.current_stream()
    cp = torch.cuda.Stream()
    work = mapflow.BSR(2, w.T, w.sender_heads, w.B, w.cu_seqlens)

    def timed(do_copy, n_compute):
        e0 = torch.cuda.Event(enable_timing=True)
        ec = torch.cuda.Event(enable_timing=True)
        ek = torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        cp.wait_stream(comp)
        if do_copy:
            held.prefetch(0, stream=cp)
        ec.record(cp)
        for l in D.layers[1:1 + n_compute]:
            work.compress(l % 2, D.q[l], D.k[l], p)
            for key in D.by_layer[l]:
                work.retrieve(D.W[key], D.v[key], D.o[key], [l % 2])
            work.release_layer(l % 2)
        ek.record(comp)
        torch.cuda.synchronize()
        t_copy = e0.elapsed_time(ec) / 1e3
        t_all = max(t_copy, e0.elapsed_time(ek) / 1e3)
        if do_copy:
            held.offload(0)
            torch.cuda.synchronize()
        return t_copy, t_all

    timed(True, 1)
    t_copy = statistics.median([timed(True, 0)[0] for _ in range(reps)])
    # enough compute to cover the copy
    t_one = statistics.median([timed(False, 1)[1] for _ in range(reps)])
    n = max(1, min(len(D.layers) - 1, math.ceil(1.2 * t_copy / t_one)))
    t_compute = statistics.median([timed(False, n)[1] for _ in range(reps)])
    t_both = statistics.median([timed(True, n)[1] for _ in range(reps)])
    held.prefetch(0)
    torch.cuda.synchronize()
    held.device_status()
    work.close()
    held.close()
    return {"layer_tiles_bytes": layer_bytes, "t_copy_ms": 1e3 * t_copy,
            "copy_gbs": layer_bytes / t_copy / 1e9,
            "compute_layers": n, "t_compute_ms": 1e3 * t_compute, "t_both_ms": 1e3 * t_both,
            "hidden_fraction": 1.0 - (t_both - t_compute) / t_copy}


def measure_density_sweep(mapflow, w, dev, peaks, label, steps=3, warmup=2):
    """The single-layer long-context workload at each of its top-p values."""
    import torch
    D = DeviceWorkload(w, dev)
    out = {}
    for p in w.p:
        bsr = mapflow.BSR(1, w.T, w.sender_heads, w.B, w.cu_seqlens)
        (l,) = D.layers
        bsr.compress(0, D.q[l], D.k[l], p)
        nnz = bsr.info(0)[0]
        R = sum((L + w.B - 1) // w.B for L in w.seqlens)
        U = union_blocks(*bsr.structure(0), w.sender_heads, R)
        for _ in range(warmup):
            bsr.compress(0, D.q[l], D.k[l], p)
            for key in D.by_layer[l]:
                bsr.retrieve(D.W[key], D.v[key], D.o[key], [0])
        bsr.profile(True)
        for _ in range(steps):
            bsr.compress(0, D.q[l], D.k[l], p)
            for key in D.by_layer[l]:
                bsr.retrieve(D.W[key], D.v[key], D.o[key], [0])
        torch.cuda.synchronize()
        bsr.device_status()
        prof = bsr.profile_read()
        bsr.close()
        wp = workloads.scaled(w, w.seqlens, p=(p,))
        ret_bytes = sum(retrieval_bytes(w, w.receivers[ri], nnz) for ri, j, m in D.reuse)
        roofs = rooflines_of(wp, prof, steps, ret_bytes * steps, qk_flops(w) * steps,
                             pack_bytes(w, nnz) * steps, peaks, label, False)
        t_comp = sum(prof[k][1] for k in ("stats", "select", "scan", "pack", "union")) / 1e3
        out[f"p={p:.2f}"] = {
            "kept_fraction": nnz / (w.sender_heads * candidate_blocks(w)),
            "retrieval_gbs": roofs["retrieve"]["achieved"],
            "retrieval_hbm_frac": roofs["retrieve"]["frac"],
            "retrieval_ms": roofs["retrieve"]["ms_per_launch"],
            "compressor_tokens_per_s": w.T * steps / t_comp,
            "stats_tflops": roofs["stats"]["achieved"], "stats_frac": roofs["stats"]["frac"],
            "stats_ms": roofs["stats"]["ms_per_launch"],
            "pack_gbs": roofs["pack"]["achieved"], "pack_ms": roofs["pack"]["ms_per_launch"],
            "union_blocks": U}
    del D
    torch.cuda.empty_cache()
    return out


def run_gpu(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist
    from cross_model_attention_gb300 import mapflow
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    peaks, src = load_peaks()
    label = "of measured" if src == "measured" else "of fallback"
    w = workloads.get(args.workload)

    D = DeviceWorkload(w, dev)
    res, nnz, U = measure_streamed(mapflow, D, args.steps, args.warmup, world, dev, peaks, label)
    roofs = res["rooflines"]
    dominant = max(("stats", "pack", "retrieve"),
                   key=lambda k: roofs[k]["ms_per_launch"] * roofs[k]["launches"])

    e2e = None if args.no_e2e else measure_e2e(mapflow, D, nnz, args.e2e_reps, peaks)
    residency = None
    if not args.no_residency:
        residency = measure_residency(mapflow, D, peaks)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        l0 = D.layers[0]
        key = next(k for k in D.v if k[0] == 0)
        to64 = lambda t: t.float().double().cpu().numpy()  # noqa: E731
        q64, k64, v64 = to64(D.q[l0]), to64(D.k[l0]), to64(D.v[key][0])
        W64 = D.W[key][0].double().cpu().numpy()
    del D
    torch.cuda.empty_cache()

    extra = {}
    if not args.no_extra and args.workload == DEFAULT_WORKLOAD:
        w2 = workloads.get(2)
        D2 = DeviceWorkload(w2, dev)
        r2, _, _ = measure_streamed(mapflow, D2, 3, 3, world, dev, peaks, label, clocks=False)
        del D2
        torch.cuda.empty_cache()
        extra["workload 2: " + w2.name] = {k: r2[k] for k in (
            "retrieval_gbs", "compressor_tokens_per_s", "ms_per_step", "retrieval_ms_per_step",
            "compressor_ms_per_step", "kept_fraction")} | {
            "retrieval_hbm_frac": r2["rooflines"]["retrieve"]["frac"],
            "stats_tflops": r2["rooflines"]["stats"]["achieved"],
            "stats_frac": r2["rooflines"]["stats"]["frac"],
            "pack_gbs": r2["rooflines"]["pack"]["achieved"]}
        w3 = workloads.get(3)
        extra["workload 3: " + w3.name] = measure_density_sweep(mapflow, w3, dev, peaks, label)

    out = None
    if rank == 0:
        if cpu is None and world == 1 and not args.no_cpu_baseline:
            r = oracle_sample(w, q64, k64, v64, W64, budget_rows=args.cpu_rows,
                              heads=args.cpu_heads)
            cpu = {"value": r["retrieval_gbs"], "unit": "GB/s", "cores": os.cpu_count(),
                   "kind": "oracle", "sample": r["sample"],
                   "compressor_tokens_per_s": r["compressor_tokens_per_s"],
                   "seconds": r["seconds"],
                   "threads_note": "numpy BLAS matmul on all host cores; elementwise ops on one"}
        launches = sum(res["launches_per_step"].values()) * args.steps
        out = {
            "metric": METRIC, "value": res["retrieval_gbs"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded, drawn on the device)",
            "config": config_dict(w, world),
            "compressor": {"tokens_per_s": res["compressor_tokens_per_s"],
                           "qk_tensor_frac": roofs["stats"]["frac"],
                           "qk_tflops": roofs["stats"]["achieved"],
                           "exp2_per_s": res["exp2_per_s"],
                           "pack_bytes_written_per_step": res["pack_bytes_written_per_step"],
                           "pack_recompute_tflops": res["pack_recompute_tflops"],
                           "ms_per_step": res["compressor_ms_per_step"]},
            "retrieval": {"ms_per_step": res["retrieval_ms_per_step"],
                          "bytes_per_step": res["retrieval_bytes_per_step"],
                          "hbm_frac": roofs["retrieve"]["frac"],
                          "tensor_flops_per_step": res["retrieval_tensor_flops_per_step"],
                          "tensor_frac_of_sustained": res["retrieval_tensor_frac_of_sustained"],
                          "binds": res["retrieval_binds"],
                          "kept_fraction": res["kept_fraction"]},
            "roofline": roofs[dominant] | {"kernel": dominant},
            "rooflines": roofs,
            "gpu_launches": launches,
            "launches_per_step": res["launches_per_step"],
            "clocks": res["clocks"],
            "e2e": e2e,
            "residency": residency,
            "workloads": extra or None,
            "cpu_baseline": cpu,
            "wall_s_timed": res["wall_s_timed"],
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-reps", type=int, default=8)
    ap.add_argument("--no-residency", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the N = 16384 workload and the N = 32768 density sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=8)
    ap.add_argument("--cpu-heads", type=int, default=2)
    ap.add_argument("--ref-rows", type=int, default=3)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
