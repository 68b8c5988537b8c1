#!/usr/bin/env python3
"""Benchmark of ragged MLA prefill over a paged latent KV cache on GB300.

One step = one pass of the whole path over one batch: the chunk plan, then
per chunk the paged gather, the K/V up-projection and the causal attention
with LSE merge.  The K timed steps run back to back with CUDA events around
each attention launch only (its duration gives the roofline); the
projection's own duration comes from a few further steps with events around
it as well.  The default workload is the DeepSeek-V3-shaped prefill
(B=1, 4096 new tokens, no cache, 128 heads, page size 128) that the
tensor-peak target is quoted on.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...     (the CPU oracle, timed on host cores)

Prints one JSON line.  `value` is causal-effective TFLOP/s of the whole step
(attention flops counted once per visible query-key pair, 640*H per pair,
plus the up-projection's 2*rows*512*2*H*128), with inputs resident on the
device; `e2e` is the same metric through the fused C entry point with
pinned-host inputs copied in and the output copied back inside the timed
region.  `roofline` describes the attention kernel.  Under torchrun (N>1)
every rank runs its own full replica (no collective) and rank 0 reports.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# DRAM bytes (read + write) per attention launch from one ncu capture of the
# current kernel (dram__bytes_read.sum + dram__bytes_write.sum), keyed by
# (workload, kernel); absent where the kernel has changed since its capture.
ATTN_DRAM_BYTES_PER_LAUNCH = {("v3_prefill", "attn_pair_kernel"): 474_251_776 + 118_507_520}
# CUDA kernel name of each attention variant the library reports.
ATTN_KERNEL_NAMES = {"pair": "attn_pair_kernel", "e4m3": "attn_pair_kernel_e4m3"}


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="v3_prefill")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    ap.add_argument("--no-stages", action="store_true", help="skip the plan / gather stage figures")
    ap.add_argument("--no-paged", action="store_true", help="skip timing the in-place paged stages")
    ap.add_argument("--stage", default=None, choices=["plan", "gather", "cache_write", "decode",
                                                      "sparse_decode"],
                    help="time one HBM-bound stage alone on its stress shape")
    ap.add_argument("--batch", type=int, default=None, help="sequences for --stage")
    return ap.parse_args()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's figure (the whole job ends when its last rank does)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_tflops(flops_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank runs the same step (replicas), so the
    job does world times the per-rank work in the slowest rank's time."""
    return flops_per_rank_step * world / (ms_per_step * 1e-3) / 1e12


def _flops(w, new, cache):
    from workloads import KV_LORA_RANK
    pairs = sum(int(n) * int(c) + int(n) * (int(n) + 1) // 2 for n, c in zip(new, cache))
    attn = 2 * w.H * (128 + 64 + 128) * pairs
    ctx = int(sum(int(n) + int(c) for n, c in zip(new, cache)))
    up = 2 * ctx * KV_LORA_RANK * 2 * w.H * 128
    return attn, up, pairs


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# A timed loop shorter than this runs at the burst clock: the kernel is judged
# against the burst peak; longer loops settle under the power cap.
SUSTAINED_AFTER_S = 2.0


def _attention_roofline(achieved, peaks, src, dtype, timed_s, clk):
    """The attention kernel's roofline entry.  The peak is the measured bf16
    dense burst figure unless the timed loop lasted seconds (then the
    sustained one).  Also reported: the fraction of the sustained figure, and a
    clock-matched fraction (TFLOP/s per SM MHz of this run against the
    sustained GEMM's TFLOP/s per MHz at the median clock it was measured at)."""
    burst = peaks.get("bf16_tflops")
    sustained = peaks.get("bf16_tflops_sustained", burst)
    long_loop = timed_s >= SUSTAINED_AFTER_S
    bf16_peak = sustained if long_loop else burst
    kind = "sustained" if long_loop else "burst"
    why = (f"timed loop {timed_s:.3f} s {'>=' if long_loop else '<'} {SUSTAINED_AFTER_S} s")
    out = {"bound": "tensor", "achieved": achieved, "unit": "TFLOP/s"}
    if dtype == "e4m3":
        # Q.K^T (2*192 of the 640 flops a key pair) runs as e4m3 MMAs and P.V
        # (2*128) as f16 MMAs.  No fp8 peak is measured on this machine: the fp8
        # rate is the measured bf16 figure times the NOMINAL fp8/bf16 ratio
        # (4.5 / 2.25 PFLOP/s dense).
        fp8_peak = 2.0 * bf16_peak
        peak = 640.0 / (384.0 / fp8_peak + 256.0 / bf16_peak)
        out["peak_source"] = (f"{src} bf16 dense {kind} {bf16_peak:.0f} ({why}); QK^T at 2x that "
                              f"(NOMINAL fp8/bf16 ratio, no fp8 peak measured), PV at bf16: "
                              f"flop-weighted {peak:.0f}")
    else:
        peak = bf16_peak
        out["peak_source"] = f"{src} bf16 dense {kind} ({why})"
    out["peak"] = peak
    out["frac"] = achieved / peak
    out["peak_kind"] = kind
    out["frac_of_bf16_burst"] = achieved / burst
    out["frac_of_bf16_sustained"] = achieved / sustained
    cl = peaks.get("clocks_under_load") or {}
    if clk and clk.get("sm_mhz") and cl.get("sm_mhz_median"):
        per_mhz = achieved / clk["sm_mhz"]
        ref_per_mhz = sustained / cl["sm_mhz_median"]
        out["frac_clock_matched"] = per_mhz / ref_per_mhz
        out["clock_matched_note"] = (f"TFLOP/s per SM MHz: this run {per_mhz:.4f} at {clk['sm_mhz']:.0f} MHz; "
                                     f"sustained GEMM {ref_per_mhz:.4f} at {cl['sm_mhz_median']:.0f} MHz")
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r[2] > 200.0] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in busy:
            for n, v in zip(names, r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(busy),
                "power_w_max": max(r[2] for r in rows)}


def _oracle_run(w, inp, codes, heads, rows=None):
    """One timed oracle run over the given heads (and per-sequence query rows,
    all when None).  Returns (seconds, flops the oracle computed): the
    projection of every context row for those heads plus the causal attention
    of the selected rows."""
    import numpy as np
    import oracle as O
    new, cache = inp["new_lens"], inp["cache_lens"]
    t = time.perf_counter()
    O.mla_prefill(codes["q"], codes["kv_cache"], codes["page_table"], inp["page_size"],
                  codes["w_k"], codes["w_uv"], codes["input_row_offsets"], codes["cache_lengths"],
                  w.buffer_token_size, w.max_chunks, inp["scale"], dtype=w.dtype,
                  q_scale=inp["q_scale"], ckv_scale=inp["ckv_scale"], w_scale=inp["w_scale"],
                  heads=heads, rows=rows)
    secs = time.perf_counter() - t
    if rows is None:
        pairs = sum(int(n) * int(c) + int(n) * (int(n) + 1) // 2 for n, c in zip(new, cache))
    else:
        pairs = sum(int(np.sum(int(c) + np.asarray(r) + 1)) for r, c in zip(rows, cache))
    ctx = int(sum(int(n) + int(c) for n, c in zip(new, cache)))
    flops = len(heads) * (2 * 320 * pairs + 2 * ctx * 512 * 256)
    return secs, flops


def _codes(inp):
    import oracle as O
    return {k: O.codes(inp[k]) for k in ("q", "kv_cache", "page_table", "w_k", "w_uv",
                                         "input_row_offsets", "cache_lengths")}


def _oracle_sample(w, inp, budget_s=15.0):
    """The oracle over whole sequences for as many heads (spread over all H)
    as fit in about `budget_s` seconds.  Returns (TFLOP/s, seconds, desc)."""
    codes = _codes(inp)
    secs, flops, heads = 0.0, 0, []
    stride = max(1, w.H // 16)
    for h in range(0, w.H, stride):
        s, f = _oracle_run(w, inp, codes, [h])
        secs += s
        flops += f
        heads.append(h)
        if secs >= budget_s:
            break
    desc = (f"oracle (numpy float64) on the whole path for all {int(sum(inp['new_lens']))} query "
            f"rows of {len(heads)} of {w.H} heads (every {stride}th from 0)")
    return flops / secs / 1e12, secs, desc


def _cores():
    return os.cpu_count() or 1


def _cpu_model():
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: implementer and part)."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return platform.machine()
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return platform.machine()


def _cpu_desc():
    return {"cores": _cores(), "cpu_model": _cpu_model(),
            "omp_num_threads": os.environ.get("OMP_NUM_THREADS")}


def run_reference(a):
    import numpy as np
    rank, world, _ = _dist()
    if rank != 0:
        return
    from workloads import PROFILE_CASES, WORKLOADS, make_inputs
    w = WORKLOADS.get(a.workload) or PROFILE_CASES[a.workload]
    inp = make_inputs(w)
    codes = _codes(inp)
    rng = np.random.default_rng(0)

    def sample(k):
        h = (k * 37) % w.H
        rows = [np.sort(rng.choice(int(n), size=min(256, int(n)), replace=False)) if n else
                np.zeros(0, np.int64) for n in inp["new_lens"]]
        return [h], rows

    for k in range(a.warmup):
        _oracle_run(w, inp, codes, *sample(k))
    secs, flops = 0.0, 0
    for k in range(a.steps):
        s, f = _oracle_run(w, inp, codes, *sample(k))
        secs += s
        flops += f
    value = flops / secs / 1e12
    desc = ("oracle (numpy float64), whole path per step on one head (cycling over the heads) "
            "for 256 random query rows per sequence; flops counted for exactly that work")
    line = {
        "impl": "reference", "metric": "MLA prefill TFLOP/s (causal-effective)", "value": value,
        "unit": "TFLOP/s", "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": secs / a.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(_config(w, inp), parallelism=f"replicas{world}" if world > 1 else "single"),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", **_cpu_desc(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(w, inp):
    return {"workload": w.name, "B": inp["B"], "new_tokens": int(sum(inp["new_lens"])),
            "cache_tokens": int(sum(inp["cache_lens"])), "H": w.H, "q_depth": 192, "v_depth": 128,
            "kv_lora_rank": 512, "page_size": w.page_size,
            "buffer_token_size": w.buffer_token_size, "max_chunks": w.max_chunks,
            "dtype": w.dtype,
            "l2": "inputs larger than L2 (no flush): q, K/V buffers and weights exceed 129 MB"}


def run_ours(a):
    import numpy as np
    import torch
    import torch.distributed as dist

    rank, world, local = _dist()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import mla_prefill_attention_plan_gb300 as mla
    from mla_prefill_attention_plan_gb300 import build as B
    B.build()
    mla.load()
    from workloads import PROFILE_CASES, WORKLOADS, make_inputs
    w = WORKLOADS.get(a.workload) or PROFILE_CASES[a.workload]
    inp = make_inputs(w)
    H, T, Bsz = w.H, inp["T_q"], inp["B"]
    S, mc = w.buffer_token_size, w.max_chunks
    dt = mla.MLA_BF16 if w.dtype == "bf16" else mla.MLA_E4M3
    elt = torch.bfloat16 if w.dtype == "bf16" else torch.float8_e4m3fn
    attn_flops, up_flops, pairs = _flops(w, inp["new_lens"], inp["cache_lens"])
    step_flops = attn_flops + up_flops

    # device-resident inputs
    d = {k: inp[k].to(dev) for k in ("q", "input_row_offsets", "cache_lengths", "kv_cache",
                                     "page_table", "w_k", "w_uv")}
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    bro = torch.empty(mc, Bsz + 1, dtype=torch.int32, device=dev)
    co = torch.empty(mc, Bsz, dtype=torch.int32, device=dev)
    bl = torch.empty(mc, dtype=torch.int32, device=dev)
    ckv = torch.empty(S, 512, dtype=elt, device=dev)
    krope = torch.empty(S, 64, dtype=elt, device=dev)
    knope = torch.empty(S, H, 128, dtype=elt, device=dev)
    # V: bf16, or f16 holding the e4m3-rounded values for e4m3
    vbuf = torch.empty(S, H, 128, dtype=torch.bfloat16 if w.dtype == "bf16" else torch.float16, device=dev)
    oacc = torch.empty(T, H, 128, dtype=torch.float32, device=dev) if mc > 1 else None
    lacc = torch.empty(T, H, dtype=torch.float32, device=dev) if mc > 1 else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    kv_descale = inp["ckv_scale"] if w.dtype == "e4m3" else 1.0
    kv_inv = 1.0 / inp["ckv_scale"] if w.dtype == "e4m3" else 1.0
    launches_per_step = (2 if Bsz > 4096 else 1) + 3 * mc   # plan: one CTA, or two passes
    attn_kernel_name = ATTN_KERNEL_NAMES[mla.mla_attention_kernel(dt)]

    def step(ev=None, attention_only=False):
        mla.check(mla.mla_prefill_plan(bro, co, bl, d["input_row_offsets"], d["cache_lengths"], Bsz,
                                       mc, S, status, stream))
        for ch in range(mc):
            mla.check(mla.mla_gather_latent(ckv, krope, d["kv_cache"], d["page_table"],
                                            inp["num_pages"], inp["page_size"], inp["max_pages"],
                                            bro, co, bl, ch, Bsz, S, dt, status, stream))
            if ev is not None and not attention_only:
                ev[ch][2].record(stream)
            mla.check(mla.mla_upproject(knope, vbuf, ckv, d["w_k"], d["w_uv"], bl, ch, S, H, dt,
                                        inp["ckv_scale"], inp["w_scale"], kv_inv, status, stream))
            if ev is not None:
                if not attention_only:
                    ev[ch][3].record(stream)
                ev[ch][0].record(stream)
            mla.check(mla.mla_prefill_attention(out, lse, oacc, lacc, d["q"], knope, vbuf, krope,
                                                d["input_row_offsets"], d["cache_lengths"], bro, co,
                                                bl, ch, mc, Bsz, H, inp["max_prompt_len"], T, S,
                                                inp["scale"], inp["q_scale"], kv_descale,
                                                kv_descale, dt, status, stream))
            if ev is not None:
                ev[ch][1].record(stream)

    for _ in range(max(3, a.warmup)):
        step()
    torch.cuda.synchronize()
    assert status.item() == 0, mla.status_string(int(status.item()))

    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)]
            for _ in range(mc)] for _ in range(a.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for k in range(a.steps):
        step(evs[k], attention_only=True)
    t1.record(stream)
    # The projection's own time, over a few more steps with events around it
    # too (an event between two kernels keeps the second from launching before
    # the first ends, so the timed steps carry events around the attention
    # only, the kernel the roofline describes).
    n_split = min(a.steps, 50)
    evs_split = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)]
                  for _ in range(mc)] for _ in range(n_split)]
    for k in range(n_split):
        step(evs_split[k])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = _max_over_ranks(t0.elapsed_time(t1), world, dev)
    ms_per_step = total_ms / a.steps
    attn_ms = sum(evs[k][ch][0].elapsed_time(evs[k][ch][1]) for k in range(a.steps) for ch in range(mc))
    used_chunks = int((bl >= 0).sum().item())
    paged = None if a.no_paged else _paged_alternates(mla, d, inp, w, bro, co, bl, ckv, krope, knope, vbuf,
                                                      out, oacc, lacc, status, stream)
    attn_ms_per_launch = attn_ms / (a.steps * max(used_chunks, 1))
    up_ms = sum(evs_split[k][ch][2].elapsed_time(evs_split[k][ch][3]) for k in range(n_split)
                for ch in range(mc)) * a.steps / n_split
    attn_ms_per_chunk = [sum(evs[k][ch][0].elapsed_time(evs[k][ch][1]) for k in range(a.steps)) / a.steps
                         for ch in range(used_chunks)]
    assert status.item() == 0, mla.status_string(int(status.item()))

    # End to end through the fused entry point, as a serving loop runs it: every
    # step's inputs are copied in from pinned host memory and its result copied
    # back, pipelined across steps on three streams (step k+1's inputs go in and
    # step k-1's output comes out while step k computes), two buffer sets.
    e2e = None
    if not a.no_e2e:
        keys = ("q", "input_row_offsets", "cache_lengths", "kv_cache", "page_table")
        host = {k: inp[k].pin_memory() for k in keys}
        outs_host = [torch.empty(T, H, 128, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        bufs = [{k: torch.empty_like(d[k]) for k in keys} for _ in range(2)]
        outs = [torch.empty(T, H, 128, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        nbytes = mla.mla_prefill_workspace_bytes(Bsz, H, T, mc, S, dt)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = outs_host[0].numel() * outs_host[0].element_size()
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        s_comp = stream

        def e2e_run(n):
            """n pipelined steps; returns (start, end) events on the compute stream."""
            in_done = [torch.cuda.Event() for _ in range(n)]
            comp_done = [torch.cuda.Event() for _ in range(n)]
            out_done = [torch.cuda.Event() for _ in range(n)]
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            start.record(s_comp)
            s_in.wait_event(start)
            s_out.wait_event(start)
            for k in range(n):
                buf, o_dev, o_host = bufs[k % 2], outs[k % 2], outs_host[k % 2]
                with torch.cuda.stream(s_in):
                    if k >= 2:
                        s_in.wait_event(comp_done[k - 2])   # its inputs were read
                    for k2 in keys:
                        buf[k2].copy_(host[k2], non_blocking=True)
                    in_done[k].record(s_in)
                s_comp.wait_event(in_done[k])
                if k >= 2:
                    s_comp.wait_event(out_done[k - 2])      # its output buffer was read back
                mla.check(mla.mla_prefill(o_dev, None, buf["q"], buf["input_row_offsets"],
                                          buf["cache_lengths"], buf["kv_cache"], buf["page_table"],
                                          inp["num_pages"], inp["page_size"], inp["max_pages"],
                                          d["w_k"], d["w_uv"], Bsz, H, T, inp["max_prompt_len"], S, mc,
                                          inp["scale"], inp["q_scale"], inp["ckv_scale"],
                                          inp["w_scale"], dt, ws, nbytes, status, s_comp))
                comp_done[k].record(s_comp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[k])
                    o_host.copy_(o_dev, non_blocking=True)
                    out_done[k].record(s_out)
            s_comp.wait_event(out_done[n - 1])
            end.record(s_comp)
            return start, end

        e2e_steps = a.e2e_steps or max(3, min(a.steps, 50))
        e2e_run(3)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = e2e_run(e2e_steps)
        torch.cuda.synchronize()
        e2e_ms = _max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
        assert status.item() == 0, mla.status_string(int(status.item()))
        # the last step's result really came back
        assert torch.equal(outs_host[(e2e_steps - 1) % 2].view(torch.int16), outs[(e2e_steps - 1) % 2].cpu().view(torch.int16))
        e2e = {"value": _job_tflops(step_flops, world, e2e_ms), "unit": "TFLOP/s",
               "ms_per_step": e2e_ms, "steps": e2e_steps, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "api": "mla_prefill",
               "pipeline": "copy-in / compute / copy-out on three streams, two buffer sets"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, src = _peaks()
    achieved = attn_flops / max(used_chunks, 1) / (attn_ms_per_launch * 1e-3) / 1e12
    roofline = _attention_roofline(achieved, peaks, src, w.dtype, total_ms * 1e-3, clk)
    roofline["kernel"] = attn_kernel_name
    roofline["traffic"] = ATTN_DRAM_BYTES_PER_LAUNCH.get((w.name, attn_kernel_name))
    line = {
        "metric": "MLA prefill TFLOP/s (causal-effective)",
        "value": _job_tflops(step_flops, world, ms_per_step),
        "unit": "TFLOP/s",
        "n_gpus": world, "steps": a.steps, "warmup": a.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": dict(_config(w, inp), parallelism=f"replicas{world}" if world > 1 else "single"),
        "attn_tflops": achieved,
        "attn_ms_per_launch": attn_ms_per_launch,
        "attn_ms_per_chunk": attn_ms_per_chunk,
        "upproj_tflops": up_flops / (up_ms / a.steps * 1e-3) / 1e12,
        "upproj_ms_per_step": up_ms / a.steps,
        "step_flops": {"attention": attn_flops, "upproject": up_flops, "visible_pairs": pairs},
        "roofline": roofline,
        "paged_alternates": paged,
        "e2e": e2e,
        "gpu_launches": launches_per_step * a.steps,
        "clocks": clk,
    }
    if not a.no_stages:
        del d, out, lse, ckv, krope, knope, vbuf, oacc, lacc
        torch.cuda.empty_cache()
        line["stages"] = _stages_summary()
    if not a.no_cpu_baseline:
        v, secs, desc = _oracle_sample(w, inp, budget_s=15.0)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", **_cpu_desc(), "kind": "oracle",
                                "sample": desc, "seconds": secs}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def _paged_alternates(mla, d, inp, w, bro, co, bl, ckv, krope, knope, vbuf, out, oacc, lacc, status,
                      stream, reps=10):
    """Chunk 0 of the workload through the stages the fused path uses
    (gather, mla_upproject, mla_prefill_attention) and through the ones that
    read the paged cache in place (mla_chunk_cache_rows, mla_upproject_paged,
    mla_prefill_attention_paged): median per-launch milliseconds of each, CUDA
    events on the launching stream, after the timed region."""
    import statistics
    import torch
    S, mc, Bsz, H, T = w.buffer_token_size, w.max_chunks, inp["B"], w.H, inp["T_q"]
    dt = mla.MLA_BF16 if w.dtype == "bf16" else mla.MLA_E4M3
    paging = (inp["num_pages"], inp["page_size"], inp["max_pages"])
    ncr = inp["num_pages"] * inp["page_size"]
    rows = torch.empty(mc, S, dtype=torch.int32, device=d["q"].device)
    kv_descale = inp["ckv_scale"] if w.dtype == "e4m3" else 1.0
    kv_inv = 1.0 / inp["ckv_scale"] if w.dtype == "e4m3" else 1.0
    attn = dict(lse=None, o_acc=oacc, lse_acc=lacc, q=d["q"], k_nope=knope, v=vbuf,
                input_row_offsets=d["input_row_offsets"], cache_lengths=d["cache_lengths"],
                buffer_row_offsets=bro, cache_offsets=co, buffer_lengths=bl, chunk=0, max_chunks=mc,
                batch_size=Bsz, num_heads=H, max_prompt_len=inp["max_prompt_len"], total_q_tokens=T,
                buffer_token_size=S, scale=inp["scale"], q_scale=inp["q_scale"], k_scale=kv_descale,
                v_scale=kv_descale, dtype=dt, d_status=status, stream=stream)
    calls = {
        "gather": lambda: mla.mla_gather_latent(ckv, krope, d["kv_cache"], d["page_table"], *paging, bro, co,
                                                bl, 0, Bsz, S, dt, status, stream),
        "cache_rows_all_chunks": lambda: mla.mla_chunk_cache_rows(rows, d["page_table"], *paging, bro, co, bl,
                                                                  mc, Bsz, S, status, stream),
        "upproject": lambda: mla.mla_upproject(knope, vbuf, ckv, d["w_k"], d["w_uv"], bl, 0, S, H, dt,
                                               inp["ckv_scale"], inp["w_scale"], kv_inv, status, stream),
        "upproject_paged": lambda: mla.mla_upproject_paged(knope, vbuf, d["kv_cache"], rows[0], ncr, bl, 0, S,
                                                           d["w_k"], d["w_uv"], H, dt, inp["ckv_scale"],
                                                           inp["w_scale"], kv_inv, status, stream),
        "attention": lambda: mla.mla_prefill_attention(out, k_rope=krope, **attn),
        "attention_paged": lambda: mla.mla_prefill_attention_paged(out, kv_cache=d["kv_cache"],
                                                                   cache_rows=rows[0], num_cache_rows=ncr,
                                                                   **attn),
    }
    res = {}
    for k, f in calls.items():
        mla.check(f())
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            mla.check(f())
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        res[k + "_ms"] = statistics.median(ts)
    assert status.item() == 0, mla.status_string(int(status.item()))
    res["chunk"] = 0
    res["note"] = ("per-launch medians on chunk 0; the fused path runs gather + upproject + attention, "
                   "the paged stages read the cache in place and are slower here")
    return res


def measure_stage(stage, batch=None, steps=20, warmup=5):
    """One HBM-bound stage alone on a stress shape, CUDA events around each
    launch.  Before every timed launch the L2 is flushed by a 512 MB write and
    then a 512 MB read, so the launch neither finds its inputs in L2 nor
    inherits the flush's dirty lines to write back.  Returns the stage's JSON
    object (the same keys as the main line)."""
    import numpy as np
    import torch
    import mla_prefill_attention_plan_gb300 as mla
    from mla_prefill_attention_plan_gb300 import build as B
    B.build()
    mla.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(512 << 20, dtype=torch.uint8, device=dev)
    peaks, src = _peaks()
    rng = np.random.default_rng(0)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    if stage == "plan":
        Bsz = batch or (1 << 22)
        mc = 4
        new = rng.integers(0, 64, Bsz)
        cache = rng.integers(0, 64, Bsz)
        S = int(-(-int((new + cache).sum()) // mc))
        iro = torch.as_tensor(np.concatenate([[0], np.cumsum(new)]).astype(np.int32), device=dev)
        cl = torch.as_tensor(cache.astype(np.int32), device=dev)
        bro = torch.empty(mc, Bsz + 1, dtype=torch.int32, device=dev)
        co = torch.empty(mc, Bsz, dtype=torch.int32, device=dev)
        bl = torch.empty(mc, dtype=torch.int32, device=dev)
        nbytes = 4 * (2 * Bsz + 1) + 4 * mc * (2 * Bsz + 2)
        launch = lambda: mla.check(mla.mla_prefill_plan(bro, co, bl, iro, cl, Bsz, mc, S, st, stream))
        kernels = "plan_one_cta" if Bsz <= 4096 else "plan_tile_totals + plan_tile_tables"
        desc = {"workload": "plan_stress", "B": Bsz, "max_chunks": mc, "buffer_token_size": S,
                "new_tokens": "U[0,63]", "cache_tokens": "U[0,63]"}
    elif stage == "cache_write":
        from workloads import WORKLOADS, make_cache_write_operands, make_inputs
        w = WORKLOADS["v3_prefill"]
        inp = make_inputs(w)
        T, H, Bsz = inp["T_q"], w.H, inp["B"]
        L = inp["new_lens"] + inp["cache_lens"]
        lat, gamma, freqs = make_cache_write_operands(w, T, int(L.max()))
        kv = inp["kv_cache"].to(dev)
        q = inp["q"].to(dev)
        lat, gamma, freqs = lat.to(dev), gamma.to(dev), freqs.to(dev)
        iro, cl, pt = (inp[k].to(dev) for k in ("input_row_offsets", "cache_lengths", "page_table"))
        # Per token: latent row read, cache row written, frequency row read,
        # and every head's rope part of q read and written.
        nbytes = T * (576 * 2 + 576 * 2 + 64 * 4 + 2 * H * 64 * 2) + 512 * 4
        launch = lambda: mla.check(mla.mla_latent_cache_write(
            kv, q, lat, gamma, freqs, iro, cl, pt, inp["num_pages"], inp["page_size"], inp["max_pages"],
            Bsz, H, T, freqs.shape[0], 1e-6, 1.0, mla.MLA_BF16, st, stream))
        kernels = "cache_write_kernel<2>"
        desc = {"workload": "latent_cache_write_v3", "tokens": T, "H": H, "cache_dtype": "bf16",
                "q": "bf16, rope part rotated in place"}
    else:
        Bsz = batch or 64
        L = 8192
        ps = 128
        pages = Bsz * L // ps
        perm = torch.as_tensor(rng.permutation(pages).astype(np.int32), device=dev)
        pt = perm.view(Bsz, L // ps)
        kv = torch.randn(pages, ps, 576, device=dev).to(torch.bfloat16)
        S = Bsz * L
        iro = torch.zeros(Bsz + 1, dtype=torch.int32, device=dev)
        cl = torch.full((Bsz,), L, dtype=torch.int32, device=dev)
        bro = torch.empty(1, Bsz + 1, dtype=torch.int32, device=dev)
        co = torch.empty(1, Bsz, dtype=torch.int32, device=dev)
        bl = torch.empty(1, dtype=torch.int32, device=dev)
        mla.check(mla.mla_prefill_plan(bro, co, bl, iro, cl, Bsz, 1, S, st, stream))
        ckv = torch.empty(S, 512, dtype=torch.bfloat16, device=dev)
        kr = torch.empty(S, 64, dtype=torch.bfloat16, device=dev)
        nbytes = 2 * S * 576 * 2 + 4 * Bsz * (L // ps)
        launch = lambda: mla.check(mla.mla_gather_latent(ckv, kr, kv, pt, pages, ps, L // ps, bro, co,
                                                         bl, 0, Bsz, S, mla.MLA_BF16, st, stream))
        kernels = "gather_kernel<2>"
        desc = {"workload": "gather_stress", "B": Bsz, "cached_tokens_per_seq": L, "page_size": ps,
                "pages": "shuffled", "dtype": "bf16"}
    for _ in range(max(3, warmup)):
        launch()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush.fill_(1)
        flush_rd.amax()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    assert st.item() == 0, mla.status_string(int(st.item()))
    ms = statistics.median(times)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    line = {"metric": f"{stage} algorithmic GB/s", "value": gbs, "unit": "GB/s", "n_gpus": 1,
            "steps": steps, "warmup": warmup, "ms_per_step": ms, "ms_min": min(times),
            "higher_is_better": True, "dtype": "int32" if stage == "plan" else "bf16",
            "data": "synthetic", "config": dict(desc, l2="flushed before every timed launch (512 MB write, then 512 MB read)"),
            "roofline": {"bound": "hbm", "kernel": kernels, "achieved": gbs, "peak": peak,
                         "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                         "peak_source": f"{src} copy bandwidth (burst)",
                         "algorithmic_bytes": nbytes}}
    del flush, flush_rd
    torch.cuda.empty_cache()
    return line


def run_stage(a):
    if a.stage in ("decode", "sparse_decode"):
        import torch
        from mla_prefill_attention_plan_gb300 import build as B
        B.build()
        torch.cuda.set_device(0)
        name = "v3_decode" if a.stage == "decode" else "v3_sparse_decode"
        print(json.dumps(measure_decode(name, a.steps, a.warmup)), flush=True)
        return
    print(json.dumps(measure_stage(a.stage, a.batch, a.steps, a.warmup)), flush=True)


def measure_decode(name, steps=20, warmup=5):
    """The absorbed decode (mla_decode, four launches) on a decode workload,
    CUDA events around each call, the L2 flushed before every timed call.
    Algorithmic bytes: every key row a sequence attends to (1152 B) once, q,
    out, w_uk and w_uv; flops: the q_lat and output projections plus 2 * H *
    (576 + 512) per visible (query, key) pair."""
    import numpy as np
    import torch
    import mla_prefill_attention_plan_gb300 as mla
    from workloads import DECODE_WORKLOADS, make_attention_sinks, make_inputs, make_sparse_indices
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)
    w = DECODE_WORKLOADS[name]
    inp = make_inputs(w, with_w_uk=True)
    B, H, T = inp["B"], w.H, inp["T_q"]
    new, cache = inp["new_lens"], inp["cache_lens"]
    sparse = "sparse" in name
    topk_n = 2048
    d = {k: inp[k].to(dev) for k in ("q", "input_row_offsets", "cache_lengths", "kv_cache", "page_table",
                                     "w_uk", "w_uv")}
    if sparse:
        idx, topk = make_sparse_indices(inp, topk_n)
        idx, topk = idx.to(dev), topk.to(dev)
        sink = make_attention_sinks(B).to(dev)
        keys = [int(k) for k in topk.cpu()]
        pairs = sum(int(n) * k for n, k in zip(new, keys))
        rows_read = sum(keys)
    else:
        idx = topk = sink = None
        pairs = sum(int(n) * int(c) + int(n) * (int(n) + 1) // 2 for n, c in zip(new, cache))
        rows_read = int(sum(int(n) + int(c) for n, c in zip(new, cache)))
    max_new = int(new.max())
    max_seq = int((new + cache).max())
    parts = mla.mla_decode_partitions(B, H, max_new, min(topk_n, max_seq) if sparse else max_seq)
    nbytes = mla.mla_decode_workspace_bytes(H, T, parts)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty(T, H, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, H, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def launch():
        mla.check(mla.mla_decode(out, lse, d["q"], d["input_row_offsets"], d["cache_lengths"], d["kv_cache"],
                                 d["page_table"], inp["num_pages"], inp["page_size"], inp["max_pages"], d["w_uk"],
                                 d["w_uv"], B, H, T, max_new, max_seq, 0, inp["scale"], d_indices=idx,
                                 indices_stride=topk_n if sparse else 0, topk_lengths=topk, attn_sink=sink,
                                 workspace=ws, workspace_bytes=nbytes, d_status=st, stream=stream))
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(3, warmup)):
        launch()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush.fill_(1)
        flush_rd.amax()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        launch()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    assert st.item() == 0, mla.status_string(int(st.item()))
    ms = statistics.median(times)
    algo_bytes = rows_read * 1152 + T * H * (192 + 128) * 2 + 2 * H * 512 * 128 * 2
    flops = T * H * 2 * (2 * 128 * 512) + 2 * H * (576 + 512) * pairs
    peaks, src = _peaks()
    gbs = algo_bytes / (ms * 1e-3) / 1e9
    tflops = flops / (ms * 1e-3) / 1e12
    del flush, flush_rd, d, ws
    torch.cuda.empty_cache()
    return {"workload": name, "B": B, "new_tokens": T, "H": H,
            "keys": "top-%d lists, per-batch sinks" % topk_n if sparse else "cached + new context, causal",
            "context_tokens": int(sum(int(n) + int(c) for n, c in zip(new, cache))),
            "partitions": "library choice (at most %d a sequence)" % parts, "kernels": "head_gemm (w_uk), decode_attn_kernel, decode_merge_kernel, head_gemm (w_uv)",
            "ms_median": ms, "ms_min": min(times), "gbs": gbs, "hbm_frac": gbs / peaks["hbm_gbs"],
            "tflops": tflops, "bf16_burst_frac": tflops / peaks["bf16_tflops"],
            "algorithmic_bytes": algo_bytes, "flops": flops, "bound": "hbm",
            "peak_source": f"{src} copy bandwidth {peaks['hbm_gbs']:.0f} GB/s",
            "l2": "flushed before every timed call"}


def _stages_summary():
    """The HBM-bound stages on their stress shapes, for the main line: the
    gather (64 sequences x 8192 cached tokens, shuffled pages, 1.2 GB moved),
    and the plan at 2^20 and 2^24 sequences."""
    out = {}
    for key, stage, batch in (("gather", "gather", None), ("plan_B2^20", "plan", 1 << 20),
                              ("plan_B2^24", "plan", 1 << 24)):
        r = measure_stage(stage, batch, steps=20, warmup=5)
        rf = r["roofline"]
        out[key] = {"workload": r["config"]["workload"], "B": r["config"].get("B"),
                    "kernel": rf["kernel"], "gbs": rf["achieved"], "peak_gbs": rf["peak"],
                    "frac": rf["frac"], "algorithmic_bytes": rf["algorithmic_bytes"],
                    "ms_median": r["ms_per_step"], "ms_min": r["ms_min"],
                    "l2": "flushed before every timed launch"}
    for name in ("v3_decode", "v3_sparse_decode"):
        out["decode_" + name] = measure_decode(name)
    return out


def main():
    a = _args()
    if a.stage is not None:
        run_stage(a)
        return
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
