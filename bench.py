#!/usr/bin/env python
"""Benchmark of the absorbed MLA decode step on GB300.

One step = one pass of the whole hot path over one batch of the full-step
workload (batch 128, 128 heads, d_model 7168, q_lora 1536, cache of 8191
tokens per sequence + 1 appended = 8192): mla_append_kv -> mla_absorb_q ->
mla_decode_attention (+ split-KV combine) -> mla_out_absorb, all in libmla
kernels. Inputs are synthetic (seeded), resident in HBM before the timed region,
and larger than L2 (1.21 GB latent cache + 374 MB of weights), so no L2 flush is
needed between steps.

`value` is the step's algorithmic bytes (latent cache rows read once, weights read
once, q/out/new-row traffic) per second, summed over all ranks. `e2e` is the same
metric through the public Python API (DecodeStep) with every step's per-token
inputs (hidden states, positions, lengths) copied from pinned host memory and its
output y copied back inside the timed region, on a copy stream with double buffers
so that the transfers overlap the neighbouring steps' kernels, as a serving loop
would; the cache and weights are device-resident state.

The same line carries `configs`: decode attention alone, timed in the same process
after the step, on the V3-shaped (16 x 4096), mixed-length (128 x U[1024, 8192]) and
long-context (32 x 32768, 64 heads) workloads, each with its time, GB/s, TFLOP/s and
fraction of the roofline.

--impl reference times the fp64 CPU oracle (the only other implementation) on a
bounded sample of the same workload on this machine's host cores; its value and
ms_per_step are the sample's own (an estimate for the whole batch is reported in a
separate field).

Multi-GPU: the decode step shards by sequence with no exchange, so N ranks run N
independent replicas of the batch (weak scaling) and rank 0 reports the total.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import threading
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
WORKLOAD = "step"


def _measured_peaks():
    path = os.path.join(HERE, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def step_costs(d):
    """Algorithmic bytes and flops of one full step: every weight read once, every cached row
    read once, the step's activations in and out; flops 2 per weight and batch row for the
    projections, 2 x H x (576 + 512) per cached token for attention."""
    B, H, dm, ql = d["B"], d["H"], d["d_model"], d["q_lora"]
    L = d["seqlens_after"].astype(np.int64)
    weights = 2 * (576 * dm + ql * dm + H * 128 * ql + H * 64 * ql + H * 128 * 512 * 2 +
                   dm * H * 128)
    cache = int(L.sum()) * 576 * 2
    act = B * dm * 2 * 2 + B * 576 * 2 + B * H * (576 * 2 + 512 * 2 + 4)
    attn_flops = int(L.sum()) * 2 * H * (576 + 512)
    proj_flops = 2 * B * (weights // 2)
    return {"bytes": weights + cache + act, "flops": attn_flops + proj_flops,
            "attn_bytes": cache + B * H * (576 * 2 + 512 * 2 + 4), "attn_flops": attn_flops,
            "weight_bytes": weights, "cache_bytes": cache}


class ClockSampler:
    """nvidia-smi clock/throttle samples (every 200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("MLA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _line_config(d, args, world):
    """The `config` object of both arms' lines (the same keys for the GPU and the reference)."""
    return dict(d["_cfg"], parallelism=f"replicas{world}" if world > 1 else "single",
                l2="inputs larger than L2 (1.21 GB cache + 374 MB weights); no flush",
                num_splits=args.num_splits or "auto")


def sample_bytes(d, n_seq: int, heads: int) -> int:
    """Algorithmic bytes of the oracle's sample: the full step of n_seq sequences restricted
    to `heads` heads (the weights of those heads once, the sequences' cached rows once, their
    activations)."""
    H, dm, ql = heads, d["d_model"], d["q_lora"]
    L = d["seqlens_after"][:n_seq].astype(np.int64)
    weights = 2 * (576 * dm + ql * dm + H * 128 * ql + H * 64 * ql + H * 128 * 512 * 2 +
                   dm * H * 128)
    act = n_seq * dm * 2 * 2 + n_seq * 576 * 2 + n_seq * H * (576 * 2 + 512 * 2 + 4)
    return int(weights + int(L.sum()) * 576 * 2 + act)


# --------------------------------------------------------------- CPU oracle leg

def time_oracle(d, n_seq: int):
    """The fp64 oracle's full step on the first n_seq sequences; returns (seconds, info)."""
    import oracle
    rows = list(range(n_seq))
    cache = d["kv_cache"]
    t0 = time.perf_counter()
    oracle.append_kv(d["h"][rows], d["w_dkr"], d["pos"][rows], d["block_table"][rows], cache)
    q_lat, q_rope = oracle.absorb_q(d["h"][rows], d["w_dq"], d["w_uq"], d["w_qr"], d["w_uk"],
                                    d["pos"][rows], d["rope_theta"])
    o_lat, _ = oracle.decode_absorbed(q_lat, q_rope, cache, d["block_table"][rows],
                                      d["seqlens_after"][rows], d["scale"])
    oracle.out_absorb(o_lat, d["w_uv"], d["w_o"])
    return time.perf_counter() - t0


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _head_slice(d, hs):
    """Weights of the first hs heads (the per-head slices of W_UQ, W_QR, W_UK, W_UV, W_O)."""
    H, ql, dm = d["H"], d["q_lora"], d["d_model"]
    return dict(
        w_uq=np.ascontiguousarray(d["w_uq"].reshape(H, 128, ql)[:hs].reshape(-1, ql)),
        w_qr=np.ascontiguousarray(d["w_qr"].reshape(H, 64, ql)[:hs].reshape(-1, ql)),
        w_uk=np.ascontiguousarray(d["w_uk"][:hs]), w_uv=np.ascontiguousarray(d["w_uv"][:hs]),
        w_o=np.ascontiguousarray(d["w_o"].reshape(dm, H, 128)[:, :hs].reshape(dm, -1)))


def time_oracle_heads(d, ws, seq: int = 0) -> float:
    """The oracle's full step for one sequence restricted to the heads in ws; seconds."""
    import oracle
    r = [seq]
    cache = d["kv_cache"]
    t0 = time.perf_counter()
    oracle.append_kv(d["h"][r], d["w_dkr"], d["pos"][r], d["block_table"][r], cache)
    q_lat, q_rope = oracle.absorb_q(d["h"][r], d["w_dq"], ws["w_uq"], ws["w_qr"], ws["w_uk"],
                                    d["pos"][r], d["rope_theta"])
    o_lat, _ = oracle.decode_absorbed(q_lat, q_rope, cache, d["block_table"][r],
                                      d["seqlens_after"][r], d["scale"])
    oracle.out_absorb(o_lat, ws["w_uv"], ws["w_o"])
    return time.perf_counter() - t0


def run_reference(args, d, costs, metric, unit):
    """The fp64 oracle on the host cores. Each step is a sample of the full step sized so
    that warm-up + all steps take about two minutes: the whole step for the first n_seq
    sequences (every head) when one sequence fits the per-step budget, else one sequence
    restricted to a head subset. `value` and `ms_per_step` are the sample's own (its
    algorithmic bytes over its measured time); the whole batch's time, scaled from
    per-sequence and per-head parts calibrated on a 1-head and an all-head run of one
    sequence, is reported separately as an estimate."""
    world, rank, _ = _dist_init()
    if rank != 0:
        return
    B, H = d["B"], d["H"]
    full = _head_slice(d, H)
    one = _head_slice(d, 1)
    t_all = min(time_oracle_heads(d, full) for _ in range(2))
    t_one = min(time_oracle_heads(d, one) for _ in range(2))
    t_head = max((t_all - t_one) / (H - 1), 1e-9)
    t_seq = max(t_one - t_head, 0.0)
    budget = 120.0 / max(1, args.steps + args.warmup)
    if t_all <= budget:
        n_seq, hs = max(1, min(B, int(budget / t_all))), H
        run = lambda: time_oracle(d, n_seq)  # noqa: E731
        what = f"the full step of {n_seq} of {B} sequences (every head)"
    else:
        n_seq, hs = 1, H
        while hs > 1 and t_seq + hs * t_head > budget:
            hs //= 2
        ws = _head_slice(d, hs)
        run = lambda: time_oracle_heads(d, ws)  # noqa: E731
        what = (f"1 of {B} sequences x {hs} of {H} heads of the full step (its whole "
                f"8192-token attention and the projections of those heads)")
    for _ in range(args.warmup):
        run()
    ts = [run() for _ in range(args.steps)]
    t_sample = statistics.median(ts)
    value = sample_bytes(d, n_seq, hs) / t_sample / 1e9
    # estimate only: the whole step scaled from the calibrated per-sequence and per-head parts
    t_step_est = B * (t_seq + H * t_head)
    sample = f"each step: {what}, timed as run; value = its algorithmic bytes / its time"
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_sample * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": _line_config(d, args, 1),
            "implementation": "fp64 CPU oracle",
            "full_step_estimate": {
                "ms": t_step_est * 1e3, "value": costs["bytes"] / t_step_est / 1e9, "unit": unit,
                "how": (f"{B} x (per-sequence {t_seq*1e3:.1f} ms + {H} x per-head "
                        f"{t_head*1e3:.2f} ms), parts calibrated on the same host")},
            "cpu_baseline": {"value": value, "unit": unit, "cores": _host_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- GPU leg

def run_gpu(args, d, costs, metric, unit):
    import torch
    world, rank, local = _dist_init()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from mla_latent_kv_13_gb300 import mla

    def dbf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def di(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    names = ["w_dkr", "w_dq", "w_uq", "w_qr", "w_uk", "w_uv", "w_o"]
    wt = {k: dbf(d[k]) for k in names}
    cache = dbf(d["kv_cache"])
    bt = di(d["block_table"])
    h, pos, L = dbf(d["h"]), di(d["pos"]), di(d["seqlens_after"])
    B, H = d["B"], d["H"]
    max_len = int(d["seqlens_after"].max())
    step = mla.DecodeStep(wt, B, H, max_len, num_splits=args.num_splits)
    stream = torch.cuda.current_stream(dev)

    # ---- device-resident timing, with the decode kernel timed inside each step
    for _ in range(args.warmup):
        step(h, pos, L, bt, cache)
    torch.cuda.synchronize(dev)
    if step.check() != 0:
        raise RuntimeError("device error during warm-up")

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if rank == 0 else None
    _barrier(world)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.start()
        time.sleep(0.3)
    start.record(stream)
    for _ in range(args.steps):
        step(h, pos, L, bt, cache, stream)
    end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop() if clocks else None
    _barrier(world)
    t_ms = start.elapsed_time(end)
    t_ms = _max_over_ranks(t_ms, world, dev)
    if step.check() != 0:
        raise RuntimeError("device error in the timed region")

    # ---- the attention launch inside the step, timed in a second pass with events around
    # it (the same launches as DecodeStep; kept out of the step's own timing, since an event
    # between two launches stops the second one's early start)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    w = step.w
    for i in range(args.steps):
        mla.append_absorb_q(h, w["w_dkr"], pos, bt, cache, w["w_dq"], w["w_uq"], w["w_qr"],
                            w["w_uk"], step.theta, step.q_lat, step.q_rope, step.ws_q, stream)
        mla.decode_prepare(L, B, H, max_len, step.num_splits, step.ws_att, stream)
        ev[i][0].record(stream)
        mla.decode_attention_prepared(step.q_lat, step.q_rope, cache, bt, L, max_len, step.scale,
                                      step.num_splits, step.o_lat, step.lse, step.ws_att, stream)
        ev[i][1].record(stream)
        mla.out_absorb(step.o_lat, w["w_uv"], w["w_o"], step.y, step.ws_out, stream)
    torch.cuda.synchronize(dev)
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if step.check() != 0:
        raise RuntimeError("device error in the attention timing pass")

    # ---- end-to-end through the public API with host buffers
    h_host = torch.from_numpy(d["h"].view(np.int16)).pin_memory()
    pos_host = torch.from_numpy(d["pos"]).pin_memory()
    L_host = torch.from_numpy(d["seqlens_after"]).pin_memory()
    y_host = torch.empty((B, d["d_model"]), dtype=torch.int16).pin_memory()
    h_dev = torch.empty_like(h).view(torch.int16)
    pos_dev, L_dev = torch.empty_like(pos), torch.empty_like(L)
    for _ in range(2):
        h_dev.copy_(h_host, non_blocking=True)
        step(h_dev.view(torch.bfloat16), pos, L, bt, cache)
    torch.cuda.synchronize(dev)
    _barrier(world)
    # A serving loop: each step's inputs go up and its result comes down on a copy stream,
    # double-buffered, so that the transfers overlap the neighbouring steps' kernels; every
    # step's copies are still inside the timed region.
    copy_s = torch.cuda.Stream(dev)
    ins = [(torch.empty_like(h_dev), torch.empty_like(pos_dev), torch.empty_like(L_dev))
           for _ in range(2)]
    ys = [torch.empty((B, d["d_model"]), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    y_done = [torch.cuda.Event() for _ in range(2)]
    y_read = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        k = i % 2
        with torch.cuda.stream(copy_s):
            if i >= 2:
                copy_s.wait_event(in_free[k])  # step i-2 has read this buffer
            ins[k][0].copy_(h_host, non_blocking=True)
            ins[k][1].copy_(pos_host, non_blocking=True)
            ins[k][2].copy_(L_host, non_blocking=True)
            in_ready[k].record(copy_s)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_s.wait_event(e0)
    upload(0)
    for i in range(args.steps):
        k = i % 2
        if i + 1 < args.steps:
            upload(i + 1)
        stream.wait_event(in_ready[k])
        if i >= 2:
            stream.wait_event(y_read[k])  # the result of step i-2 has left this buffer
        step(ins[k][0].view(torch.bfloat16), ins[k][1], ins[k][2], bt, cache, out=ys[k])
        in_free[k].record(stream)
        y_done[k].record(stream)
        with torch.cuda.stream(copy_s):
            copy_s.wait_event(y_done[k])
            y_host.copy_(ys[k].view(torch.int16), non_blocking=True)
            y_read[k].record(copy_s)
    stream.wait_event(y_read[(args.steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = _max_over_ranks(e0.elapsed_time(e1), world, dev)
    h2d = h_host.numel() * 2 + pos_host.numel() * 4 + L_host.numel() * 4
    d2h = y_host.numel() * 2

    # ---- decode attention alone on the other attention workloads (same process), a
    # fixed number of launches each: a few tens of milliseconds per workload, whatever the
    # step count (after a long step run the part sits at its power cap, and thousands of
    # further launches per workload would time that rather than the kernel)
    configs = None
    if rank == 0 and not args.no_configs:
        configs = time_attention_configs(cache, dev, CONFIG_LAUNCHES, args.num_splits)

    if rank != 0:
        return
    peaks = _measured_peaks()
    ms_step = t_ms / args.steps
    value = costs["bytes"] * world * args.steps / (t_ms * 1e-3) / 1e9
    tflops = costs["flops"] * world * args.steps / (t_ms * 1e-3) / 1e12
    roof_s = max(costs["bytes"] / (peaks["hbm_gbs"] * 1e9),
                 costs["flops"] / (peaks["bf16_tflops"] * 1e12))
    attn_gbs = costs["attn_bytes"] / (attn_ms * 1e-3) / 1e9
    traffic = None
    tr_path = os.path.join(HERE, "profiles", "decode_traffic.json")
    if os.path.exists(tr_path):
        try:
            tj = json.load(open(tr_path))
            if tj.get("kernel_source_hash") == _kernel_hash():
                traffic = tj.get("dram_bytes_per_launch")
        except Exception:
            traffic = None
    launches_per_step = step_launches(step)
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": _line_config(d, args, world),
        "tflops": tflops,
        "tokens_per_s": B * world * args.steps / (t_ms * 1e-3),
        "roofline_frac_step": roof_s / (ms_step * 1e-3),
        "roofline": {"kernel": "decode_attention_prepared (attention + merge kernels; the "
                               "step's schedule runs on the side stream, next to absorb_q)",
                     "bound": "hbm", "achieved": attn_gbs,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": attn_gbs / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_source": peaks["source"] + " (burst copy)",
                     "launch_ms": attn_ms,
                     "algorithmic_bytes_per_launch": costs["attn_bytes"]},
        "e2e": {"value": costs["bytes"] * world * args.steps / (e2e_ms * 1e-3) / 1e9,
                "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if configs:
        line["configs"] = configs
    if world == 1 and not args.no_cpu_baseline:
        t_s = time_oracle(d, args.cpu_sample)
        line["cpu_baseline"] = {
            "value": sample_bytes(d, args.cpu_sample, H) / t_s / 1e9, "unit": unit,
            "cores": _host_cores(), "kind": "oracle", "seconds": t_s,
            "sample": (f"the full step of {args.cpu_sample} of {B} sequences (all heads, "
                       f"all weights), timed as run; value = that sample's algorithmic "
                       f"bytes / its time")}
    print(json.dumps(line), flush=True)


def run_gpu_attention(args, w, metric, unit):
    """Decode attention alone on one of the attention workloads (profiling / per-config lines)."""
    import torch
    world, rank, local = _dist_init()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from mla_latent_kv_13_gb300 import mla, synth
    d = synth.make_attention_inputs(w, seed=0)

    def dbf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    ql, qr, cache = dbf(d["q_lat"]), dbf(d["q_rope"]), dbf(d["kv_cache"])
    bt = torch.from_numpy(d["block_table"]).to(dev)
    L = torch.from_numpy(d["seqlens"]).to(dev)
    B, H = d["B"], d["H"]  # H = query rows per sequence (s_q tokens x H / s_q heads)
    s_q = w.s_q
    max_len = int(d["seqlens"].max())
    ws = mla.alloc_workspace(mla.decode_workspace_size(B, H, max_len, args.num_splits))
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    if s_q > 1:  # draft tokens: the same rows, causal among the s_q tokens
        ql, qr = ql.view(B, s_q, H // s_q, 512), qr.view(B, s_q, H // s_q, 64)
        out, lse = out.view(B, s_q, H // s_q, 512), lse.view(B, s_q, H // s_q)

    def attend(c):
        if s_q > 1:
            mla.decode_attention_mq(ql, qr, c, bt, L, max_len, d["scale"], args.num_splits, out,
                                    lse, ws)
        else:
            mla.decode_attention(ql, qr, c, bt, L, max_len, d["scale"], args.num_splits, out,
                                 lse, ws)

    def one():
        attend(cache)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize(dev)
    # inputs below L2 size are rotated through distinct cache copies (cold L2 per step)
    nbytes = d["kv_cache"].nbytes
    copies = [cache]
    if nbytes * 2 < 256 << 20:
        copies += [cache.clone() for _ in range(max(1, (256 << 20) // nbytes))]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize(dev)
    start.record(stream)
    for i in range(args.steps):
        attend(copies[i % len(copies)])
    end.record(stream)
    torch.cuda.synchronize(dev)
    if mla.check_device_status(ws) != 0:
        raise RuntimeError("device error in the timed region")
    t_ms = _max_over_ranks(start.elapsed_time(end), world, dev)
    if rank != 0:
        return
    peaks = _measured_peaks()
    byts = synth.algorithmic_attention_bytes(d["seqlens"], H)
    flops = synth.attention_flops(d["seqlens"], H)
    ms = t_ms / args.steps
    gbs = byts / (ms * 1e-3) / 1e9
    roof_s = max(byts / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
    line = {"metric": metric, "value": gbs * world, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": dict(w.describe(), l2=("rotating %d cache copies" % len(copies))
                           if len(copies) > 1 else "inputs larger than L2"),
            "tflops": flops / (ms * 1e-3) / 1e12, "tokens_per_s": B * s_q / (ms * 1e-3),
            "roofline": {"kernel": "decode_attention", "bound": "hbm", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": roof_s / (ms * 1e-3), "traffic": None,
                         "peak_source": peaks["source"] + " (burst copy)"},
            "gpu_launches": args.steps * mla.decode_plan(B, H, max_len, args.num_splits)[1]}
    print(json.dumps(line), flush=True)


def run_gpu_prefill(args):
    """Chunked prefill of one sequence (expanded form): 128 heads, a 4096-token chunk after a
    4096-token prefix, timed through mla_prefill_attention (row gather, the two per-head
    up-projections and the causal attention) against the bf16 tensor peak."""
    import torch
    world, rank, local = _dist_init()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from mla_latent_kv_13_gb300 import mla, synth
    H, prefix, C = 128, 4096, 4096
    T = prefix + C
    d = synth.make_attention_inputs(synth.Workload("prefill", 1, H, (T,), None, True), seed=0)
    rng = np.random.default_rng(1)

    def dbf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def rnd(shape, sigma):
        return dbf(synth.f32_to_bf16_bits((rng.standard_normal(shape) * sigma).astype(np.float32)))

    qn, qr = rnd((C, H, 128), 1.0), rnd((C, H, 64), 1.0)
    w_uk, w_uv = rnd((H, 128, 512), 0.02), rnd((H, 128, 512), 0.02)
    cache = dbf(d["kv_cache"])
    bt = torch.from_numpy(d["block_table"][0]).to(dev)
    ws = mla.alloc_workspace(mla.prefill_workspace_size(H, prefix, C))
    out = torch.empty((C, H, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((C, H), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def one():
        mla.prefill_attention(qn, qr, cache, bt, prefix, w_uk, w_uv, d["scale"], out, lse, ws)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize(dev)
    start.record(stream)
    for _ in range(args.steps):
        one()
    end.record(stream)
    torch.cuda.synchronize(dev)
    if mla.check_device_status(ws) != 0:
        raise RuntimeError("device error in the timed region")
    t_ms = _max_over_ranks(start.elapsed_time(end), world, dev)
    if rank != 0:
        return
    peaks = _measured_peaks()
    ms = t_ms / args.steps
    visible = sum(prefix + i + 1 for i in range(C))
    attn_flops = 2 * H * (192 + 128) * visible
    proj_flops = 2 * 2 * T * 512 * H * 128
    flops = attn_flops + proj_flops
    tf = flops / (ms * 1e-3) / 1e12
    line = {"metric": "MLA chunked prefill (expanded form): TFLOP/s on 1 GB300", "value": tf * world,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "prefill", "heads": H, "prefix": prefix, "chunk": C,
                       "d_c": 512, "d_nope": 128, "d_rope": 64, "d_v": 128,
                       "l2": "inputs larger than L2 (537 MB of projected K/V)"},
            "tokens_per_s": C / (ms * 1e-3),
            "roofline": {"kernel": "prefill_attention", "bound": "tensor", "achieved": tf,
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": tf / peaks["bf16_tflops"], "traffic": None,
                         "peak_source": peaks["source"] + " (cuBLAS bf16 burst)",
                         "flops_per_launch": flops, "attention_flops": attn_flops},
            "gpu_launches": args.steps * 4}
    print(json.dumps(line), flush=True)


ATTN_CONFIGS = ("v3", "mixed", "long", "long_fp8", "step_prepared")
ATTN_GATE = {"v3": None, "mixed": 0.70, "long": 0.70, "long_fp8": None, "step_prepared": None}


CONFIG_LAUNCHES = 200  # timed launches per attention workload in the `configs` object


def time_attention_configs(pool, dev, launches: int, num_splits: int):
    """mla_decode_attention alone on the v3-shaped, mixed-length and long-context workloads
    (the long one also over the FP8 cache), and mla_decode_attention_prepared on the
    full-step shape with its schedule prepared once, in this process after the step: their
    seqlens, block tables and queries follow the
    seeded recipe of each workload; their cache rows are the step's resident pool (the same
    N(0, 1) bf16 values; every block table indexes into it). Launches back to back on one
    stream between CUDA events; a workload whose cache is under twice the L2 size reads a
    different block range of the pool at each launch (its table shifted by a multiple of its
    block count), so every launch starts from a cold L2."""
    import torch
    from mla_latent_kv_13_gb300 import mla, synth
    peaks = _measured_peaks()
    stream = torch.cuda.current_stream(dev)
    nb_pool = pool.shape[0]
    out_all = {}
    fp8_pool = None
    for name in ATTN_CONFIGS:
        fp8 = name.endswith("_fp8")
        # step_prepared: the full-step shape as the layers of one decode step see it, the
        # schedule prepared once (mla_decode_prepare) and every call skipping it
        prepared = name.endswith("_prepared")
        w = synth.WORKLOADS[name[:-4] if fp8 else (name[:-9] if prepared else name)]
        if fp8 and fp8_pool is None:  # the same pool as e4m3 codes with row exponents
            fp8_pool = mla.quantize_kv_fp8(pool)
        L = synth.draw_seqlens(w, 0)
        bt, nblk = synth.make_block_table(L, w.shuffled, 0)
        if nblk > nb_pool:
            continue
        ql, qr = synth.make_attention_queries(w, seed=0)
        B, H = w.batch, w.heads
        max_len = int(L.max())

        def dbf(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(
                torch.bfloat16)

        q_lat, q_rope = dbf(ql), dbf(qr)
        cache_bytes = int(L.sum()) * 576 * 2
        rot = 1
        if 2 * cache_bytes < (256 << 20):
            rot = max(1, min(nb_pool // nblk, 16))
        bts = []
        for k in range(rot):
            b2 = bt.copy()
            b2[b2 >= 0] += k * nblk
            bts.append(torch.from_numpy(b2).to(dev))
        Ld = torch.from_numpy(L).to(dev)
        ws = mla.alloc_workspace(mla.decode_workspace_size(B, H, max_len, num_splits))
        out = torch.empty((B, H, 512), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H), dtype=torch.float32, device=dev)

        if prepared:
            mla.decode_prepare(Ld, B, H, max_len, num_splits, ws)

        def attend(i):
            if prepared:
                mla.decode_attention_prepared(q_lat, q_rope, pool, bts[i % rot], Ld, max_len,
                                              synth.SCALE_192, num_splits, out, lse, ws)
            elif fp8:
                mla.decode_attention_fp8(q_lat, q_rope, fp8_pool[0], fp8_pool[1], bts[i % rot], Ld,
                                         max_len, synth.SCALE_192, num_splits, out, lse, ws)
            else:
                mla.decode_attention(q_lat, q_rope, pool, bts[i % rot], Ld, max_len,
                                     synth.SCALE_192, num_splits, out, lse, ws)

        for i in range(3):
            attend(i)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(launches):
            attend(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if mla.check_device_status(ws) != 0:
            raise RuntimeError(f"device error in the {name} attention timing")
        ms = e0.elapsed_time(e1) / launches
        byts = synth.algorithmic_attention_bytes(L, H, kv_bytes_per_value=1 if fp8 else 2)
        flops = synth.attention_flops(L, H)
        roof_s = max(byts / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
        out_all[name] = {
            "batch": B, "heads": H,
            "seqlens": w.seqlens[0] if w.seqlens else f"U{list(w.seqlen_range)} seed 0",
            "tokens": int(L.sum()), "ms": ms, "GB/s": byts / (ms * 1e-3) / 1e9,
            "TFLOP/s": flops / (ms * 1e-3) / 1e12, "frac": roof_s / (ms * 1e-3),
            "bound": "hbm" if byts / (peaks["hbm_gbs"] * 1e9) >=
            flops / (peaks["bf16_tflops"] * 1e12) else "tensor",
            "gate": ATTN_GATE[name], "launches": launches,
            "plan": {"splits": mla.decode_plan(B, H, max_len, num_splits)[0]},
            "l2": (f"{rot} disjoint block ranges rotated" if rot > 1
                   else "cache larger than L2"),
            "algorithmic_bytes": byts,
            "cache": "e4m3 codes + one power-of-two scale exponent per token" if fp8 else "bf16",
            "schedule": ("prepared once, outside the timed launches (one decode step's layers "
                         "share it)" if prepared else "computed by every call")}
        del ws, out, lse, bts, q_lat, q_rope
    return out_all


def step_launches(step) -> int:
    """Kernels one DecodeStep launches, by the library's own plans for these shapes on this
    device: append_absorb_q 3-9 (W_DQ with W_DKR in one launch where their clusters fit),
    decode 1-3 (+ merge, + schedule), out_absorb 2-3 (a split-K product reduced inside its
    clusters is one launch, else two)."""
    from mla_latent_kv_13_gb300 import mla
    _, decode = mla.decode_plan(step.B, step.H, step.max_seqlen, step.num_splits)
    _, _, out, both = mla.projection_launches(step.B, step.dm, step.ql, step.H)
    return both + decode + out


DECODE_SOURCES = ("decode_tc.cu", "sm100.cuh", "common.cuh")


def _kernel_hash() -> str:
    """Hash of the decode kernel's sources: recorded DRAM traffic is only reported while
    the kernel it was measured on is unchanged."""
    import hashlib
    hsh = hashlib.sha256()
    csrc = os.path.join(HERE, "mla_latent_kv_13_gb300", "csrc")
    for n in DECODE_SOURCES:
        with open(os.path.join(csrc, n), "rb") as f:
            hsh.update(f.read())
    return hsh.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["step", "tiny", "v3", "mixed", "long", "mtp", "prefill"],
                    help="step = the full decode step (default); the others time decode "
                         "attention alone on that attention workload")
    ap.add_argument("--cpu-sample", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload attention timings in the step line")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    import sys
    sys.path.insert(0, HERE)
    from mla_latent_kv_13_gb300 import synth
    metric = "MLA decode attn: latent-KV GB/s, TFLOP/s and % roofline on 1 GB300"
    if args.workload != "step":
        if args.impl == "reference":
            raise SystemExit("--impl reference is defined on the full-step workload")
        if args.workload == "prefill":
            run_gpu_prefill(args)
        else:
            run_gpu_attention(args, synth.WORKLOADS[args.workload], metric, "GB/s")
        return
    w = synth.WORKLOADS[WORKLOAD]
    d = synth.make_step_inputs(w, seed=0)
    d["_cfg"] = dict(w.describe(), seqlen=int(d["seqlens_after"].max()), prefilled=int(d["pos"][0]))
    costs = step_costs(d)
    if args.impl == "reference":
        run_reference(args, d, costs, metric, "GB/s")
    else:
        run_gpu(args, d, costs, metric, "GB/s")


if __name__ == "__main__":
    main()
