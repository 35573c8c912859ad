#!/usr/bin/env python
"""Benchmark of the fused attention forward + split-KV decode on GB300.

One step = the whole hot path over one batch of synthetic input:
  attn_fwd on the prefill workload (B=4, H=16, N=2048, d=128, bf16) non-causal,
  attn_fwd on the same inputs causal, and
  attn_decode on the decode workload (B=16, Hq=32, Hkv=8, KV cache 32768 x 128,
  valid lengths uniform in [1024, 32768]).
`value` is forward TFLOPS (algorithmic 4*B*H*N*N*d, halved for causal) over the
two forward launches; the decode's HBM GB/s is reported beside it.  Inputs are
resident in HBM; L2 is flushed (a 512 MiB write) between timed steps.  Each
launch of the step is then timed again over --stat-iters iterations for its
median, min and max.

Beside the step: the long-context (B=1 H=32 N=16384, outlier channels) and GQA
(B=8 Hq=32 Hkv=8 N=4096) causal forwards (`configs`), the backward, the packed
variable-length forward, the FP8 forward and the d=256 forward, each timed
alone; `e2e` runs the whole step through the public API from pinned host
buffers.  The oracle leg (`cpu_baseline`) times the fp64 CPU oracle on whole
heads of the prefill inputs and checks the bench's own last outputs for those
heads against it.

`--impl reference` times the fp64 CPU oracle instead (a bounded sample of the
same workload on the host cores).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("attn fwd TFLOPS & % of GB300 BF16 peak; split-KV decode HBM GB/s & % of peak")


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# The sources each profiled kernel is built from (its own translation unit and
# the headers it includes); a kernel's DRAM figures stay valid while their code
# (comments removed) hashes to the value stored beside them.
KERNEL_SOURCES = {
    "attn_fwd_kernel": ["attn_fwd_sm103.cu", "fwd_sched.h", "ptx.cuh", "internal.h"],
    "attn_decode_split_kernel": ["attn_decode_sm103.cu", "ptx.cuh", "internal.h"],
    "attn_bwd": ["attn_bwd_sm103.cu", "fwd_sched.h", "ptx.cuh", "internal.h"],
    "attn_fp8": ["attn_fp8_sm103.cu", "fwd_sched.h", "ptx.cuh", "internal.h"],
    "attn_fwd_wide": ["attn_fwd_wide_sm103.cu", "fwd_sched.h", "ptx.cuh", "internal.h"],
}


def _code_only(text: str) -> str:
    """C/C++ source with comments removed and trailing blanks stripped: what a
    DRAM-traffic record depends on (string literals in these sources hold no
    comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel: str) -> str:
    """sha256 over name + code (comments removed) of one kernel's sources, in
    the listed order: a comment edit keeps a traffic record valid, a code edit
    does not."""
    import hashlib
    csrc = os.path.join(ROOT, "exact_attention_14_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        h.update(name.encode())
        with open(os.path.join(csrc, name), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()


def read_traffic():
    """DRAM bytes per launch from the committed ncu summaries, for the kernels
    whose code (comments aside) has not changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return {}
    with open(path) as f:
        t = json.load(f)
    return {k: v for k, v in t.get("kernels", {}).items()
            if k in KERNEL_SOURCES and v.get("sources_sha256") == kernel_source_hash(k)}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "reasons": sorted(reasons)}


def fwd_flops(B, H, N, d, causal):
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def oracle_sample(seconds: float, q, k, v, scale, heads=None):
    """Time the fp64 oracle on whole heads of the prefill workload (the same
    inputs the GPU legs use), non-causal and causal alternately, until
    `seconds` of work (or over the given (b, h, causal) heads).  Returns
    (TFLOPS, desc, cores, elapsed, [(b, h, causal, O, LSE), ...])."""
    import oracle
    oracle.build()
    B, H, N, d = q.shape
    flops, t0, done, out = 0.0, time.perf_counter(), 0, []
    while True:
        if heads is not None:
            if done >= len(heads):
                break
            b, h, causal = heads[done]
        else:
            b, h, causal = (done // 2) % B, ((done // 2) // B) % H, bool(done % 2)
        sl = (slice(b, b + 1), slice(h, h + 1))
        o_ref, l_ref = oracle.attention(q[sl], k[sl], v[sl], causal=causal, scale=scale)
        out.append((b, h, causal, o_ref[0, 0], l_ref[0, 0]))
        flops += fwd_flops(1, 1, N, d, causal)
        done += 1
        el = time.perf_counter() - t0
        if heads is None and el >= seconds:
            break
    el = time.perf_counter() - t0
    cores = os.cpu_count() or 1
    desc = (f"{done} whole heads of the prefill workload (N={N}, d={d}), "
            f"alternating non-causal/causal, fp64 three-pass oracle, OpenMP on {cores} threads")
    return flops / el / 1e12, desc, cores, el, out


def stats_ms(times_s):
    """Median, min and max (ms) of per-iteration device times."""
    t = sorted(times_s)
    n = len(t)
    med = t[n // 2] if n % 2 else 0.5 * (t[n // 2 - 1] + t[n // 2])
    return {"median_ms": 1e3 * med, "min_ms": 1e3 * t[0], "max_ms": 1e3 * t[-1], "iters": n}


def time_legs(stream, fns, iters, flush, flush_each=False):
    """Per-launch device times (s) of each callable in `fns`, over `iters`
    iterations after an L2 flush (before every callable if flush_each), CUDA
    events on `stream`.  Returns one list of times per callable."""
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in fns] for _ in range(iters)]
    for i in range(iters):
        flush.zero_()
        for j, fn in enumerate(fns):
            if flush_each and j > 0:
                flush.zero_()
            evs[i][j][0].record(stream)
            fn()
            evs[i][j][1].record(stream)
    torch.cuda.synchronize()
    return [[evs[i][j][0].elapsed_time(evs[i][j][1]) * 1e-3 for i in range(iters)]
            for j in range(len(fns))]


def ranks_barrier(world: int) -> None:
    """Barrier over the launched ranks (no-op for one process)."""
    if world > 1:
        torch.distributed.barrier()


def ranks_max(values, world: int, device) -> list:
    """Element-wise maximum of per-rank timings over all ranks (the job's time
    is its slowest rank's)."""
    if world == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def run_reference(args, rank, world):
    if rank != 0:
        return
    from exact_attention_14_gb300.inputs import PREFILL, make_config_inputs
    q, k, v = make_config_inputs(PREFILL)
    for _ in range(args.warmup):
        oracle_sample(1.0, q, k, v, PREFILL.scale)
    total_flops = total_t = 0.0
    cores = os.cpu_count() or 1
    desc = ""
    for _ in range(args.steps):
        tf, desc, cores, el, _ = oracle_sample(3.0, q, k, v, PREFILL.scale)
        total_flops += tf * el * 1e12
        total_t += el
    value = total_flops / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill fwd B=4 H=16 N=2048 d=128 (oracle sample)"},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import exact_attention_14_gb300 as ea
    from exact_attention_14_gb300.inputs import DECODE, GQA, LONG, PREFILL, VARLEN, \
        hadamard_signs, make_config_inputs, make_decode_config_inputs, make_fwd_inputs, \
        make_varlen_inputs, varlen_lengths

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    ea.load()
    peaks = read_peaks()
    peak_t = peaks["bf16_tflops"]
    traffic = read_traffic()
    cfg = PREFILL
    q_h, k_h, v_h = make_config_inputs(cfg)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    # one output buffer per mask, so both results stay for the parity check
    o = {c: torch.empty(q.shape, dtype=torch.bfloat16, device=dev) for c in (False, True)}
    lse = {c: torch.empty(q.shape[:3], dtype=torch.float32, device=dev) for c in (False, True)}
    fws = {c: torch.empty(max(16, ea.attn_fwd_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N,
                                                             cfg.d, c)),
                          dtype=torch.uint8, device=dev) for c in (False, True)}
    dq_h, dk_h, dv_h, dsl_h = make_decode_config_inputs(DECODE)
    dq, dk, dv, dsl = dq_h.to(dev), dk_h.to(dev), dv_h.to(dev), dsl_h.to(dev)
    d_o = torch.empty(dq.shape, dtype=torch.bfloat16, device=dev)
    d_lse = torch.empty(dq.shape[:3], dtype=torch.float32, device=dev)
    ws = torch.empty(ea.attn_decode_workspace_size(DECODE.B, DECODE.Hq, DECODE.Hkv, DECODE.Nmax,
                                                   DECODE.d, 0), dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    sum_len = int(dsl.sum().item())
    # algorithmic decode bytes: K and V of every valid key, Q read, O (bf16) + LSE written
    dec_bytes = (2.0 * sum_len * DECODE.Hkv * DECODE.d * 2 + dq.numel() * 2 + d_o.numel() * 2
                 + d_lse.numel() * 4)
    f_nc = fwd_flops(cfg.B, cfg.Hq, cfg.N, cfg.d, False)
    f_c = fwd_flops(cfg.B, cfg.Hq, cfg.N, cfg.d, True)
    stream = torch.cuda.current_stream(dev)

    def fwd_launch(c):
        return lambda: ea.attn_fwd(q, k, v, o[c], lse[c], causal=c, workspace=fws[c],
                                   stream=stream)

    def dec_launch():
        ea.attn_decode(dq, dk, dv, dsl, d_o, d_lse, workspace=ws, stream=stream)

    step_fns = [fwd_launch(False), fwd_launch(True), dec_launch]

    def step(ev=None):
        for j, fn in enumerate(step_fns):
            if ev: ev[j].record(stream)
            fn()
        if ev: ev[len(step_fns)].record(stream)

    args.warmup = max(args.warmup, 3)
    # The flush comes first in every step: the GPU is still writing it while
    # the host enqueues the step's launches, so no host gap lands between a
    # step's events.
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if ea.attn_last_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    ranks_barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            step(evs[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        # per-launch statistics over more iterations (same launches, L2 flushed
        # before each step), still under the clock sampler
        n_stat = max(args.stat_iters, args.steps)
        st_nc, st_c, st_dec = time_legs(stream, step_fns, n_stat, flush)
    ranks_barrier(world)
    if ea.attn_last_device_error() != 0:
        raise RuntimeError("device error during the timed region")
    per = [[e[j].elapsed_time(e[j + 1]) * 1e-3 for e in evs] for j in range(3)]
    t_nc, t_c, t_dec = (sum(x) / args.steps for x in per)
    t_nc, t_c, t_dec = ranks_max([t_nc, t_c, t_dec], world, dev)
    t_step = t_nc + t_c + t_dec
    tflops = world * (f_nc + f_c) / (t_nc + t_c) / 1e12
    dec_gbs = world * dec_bytes / t_dec / 1e9

    # end to end through the public API: pinned host inputs -> device -> result
    # to host, for the whole step (both forwards and the decode; the decode's
    # KV cache is resident state, its query and lengths come from the host)
    e2e = None
    if rank == 0 or world > 1:
        e2e = run_e2e(ea, args, world, dev, stream, (q_h, k_h, v_h), (dq_h, dsl_h), (dk, dv),
                      o, lse, d_o, d_lse, ws, fws, f_nc + f_c)

    extra = {}
    if not args.no_configs:
        extra["configs"] = run_configs(ea, args, dev, stream, flush, peaks, traffic)
    if not args.no_bwd:
        extra["bwd"] = run_bwd(ea, args, dev, stream, flush, peaks, q, k, v)
    if not args.no_varlen:
        extra["varlen"] = run_varlen(ea, args, dev, stream, flush, peaks)
    if not args.no_fp8:
        extra["fp8"] = run_fp8(ea, args, dev, stream, flush, peaks)
    if not args.no_wide:
        extra["wide"] = run_wide(ea, args, dev, stream, flush, peaks)
        extra["decode_d256"] = run_decode_wide(ea, args, dev, stream, flush, peaks, traffic)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tf, desc, cores, _, heads = oracle_sample(args.cpu_seconds, q_h, k_h, v_h, cfg.scale)
        cpu = {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": desc,
               "parity_check": parity_of_heads(heads, o, lse)}
        if not cpu["parity_check"]["pass"]:
            raise RuntimeError(f"bench outputs differ from the oracle: {cpu['parity_check']}")

    if rank != 0:
        return
    fwd_time = t_nc + t_c
    tr = traffic.get("attn_fwd_kernel", {})
    roof = {"bound": "tensor", "kernel": "attn_fwd_kernel (non-causal + causal launches)",
            "achieved": (f_nc + f_c) / fwd_time / 1e12, "peak": peak_t, "unit": "TFLOP/s",
            "frac": (f_nc + f_c) / fwd_time / 1e12 / peak_t,
            "traffic": (tr["prefill_noncausal"] + tr["prefill_causal"])
                       if "prefill_noncausal" in tr and "prefill_causal" in tr else None,
            "traffic_note": "DRAM bytes of one non-causal + one causal launch (ncu, profiles/); "
                            "algorithmic bytes 2 x 134.7 MB",
            "peak_source": f"{peaks['source']} bf16_tflops (burst)",
            "noncausal": {"achieved": f_nc / t_nc / 1e12, "frac": f_nc / t_nc / 1e12 / peak_t,
                          "traffic": tr.get("prefill_noncausal"), **stats_ms(st_nc)},
            "causal": {"achieved": f_c / t_c / 1e12, "frac": f_c / t_c / 1e12 / peak_t,
                       "traffic": tr.get("prefill_causal"), **stats_ms(st_c)}}
    trd = traffic.get("attn_decode_split_kernel", {})
    roof_dec = {"bound": "hbm", "kernel": "attn_decode_split_kernel (split-KV with in-kernel merge)",
                "achieved": dec_bytes / t_dec / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dec_bytes / t_dec / 1e9 / peaks["hbm_gbs"],
                "traffic": trd.get("decode"),
                "traffic_note": "DRAM bytes per launch (ncu, profiles/); algorithmic bytes in "
                                "decode.algorithmic_bytes",
                "peak_source": f"{peaks['source']} hbm_gbs", **stats_ms(st_dec)}
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "prefill fwd B=4 H=16 N=2048 d=128 (non-causal + causal) + "
                               "decode B=16 Hq=32 Hkv=8 Nmax=32768 d=128",
                   "global_batch": cfg.B * world, "seq_len": cfg.N,
                   "parallelism": f"replicas x{world}", "l2": "flushed (512 MiB write) between steps"},
        "fwd": {"noncausal_tflops": f_nc / t_nc / 1e12, "causal_tflops": f_c / t_c / 1e12,
                "noncausal_ms": 1e3 * t_nc, "causal_ms": 1e3 * t_c,
                "frac_of_bf16_peak": (f_nc + f_c) / fwd_time / 1e12 / peak_t},
        "decode": {"value": dec_gbs, "unit": "GB/s", "ms": 1e3 * t_dec,
                   "algorithmic_bytes": dec_bytes, "frac_of_hbm": dec_gbs / world / peaks["hbm_gbs"],
                   "sum_seqlen": sum_len},
        "roofline": roof, "roofline_decode": roof_dec, **extra,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (2 + ea.attn_decode_kernel_launches(DECODE.B, DECODE.Hq, DECODE.Hkv,
                                                            DECODE.Nmax, DECODE.d)) * args.steps,
        "wall_s_timed_region": wall,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def parity_of_heads(heads, o, lse):
    """The bench's last outputs (bf16 O, fp32 LSE) on the heads the oracle leg
    computed, against the oracle within the parity tolerances (O compared with
    the oracle rounded to bf16, plus half a bf16 ulp)."""
    import numpy as np
    worst_o = worst_l = 0.0
    ok = True
    for b, h, causal, o_ref, l_ref in heads:
        got = o[causal][b, h].float().cpu().double().numpy()
        ref = torch.from_numpy(o_ref).to(torch.bfloat16).double().numpy()
        half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 8)
        err = np.abs(got - ref)
        ok &= bool((err <= 1e-2 + half_ulp).all())
        worst_o = max(worst_o, float(err.max()))
        dl = float(np.abs(lse[causal][b, h].cpu().double().numpy() - l_ref).max())
        ok &= dl <= 1e-3
        worst_l = max(worst_l, dl)
    return {"heads": len(heads), "rows": sum(x[3].shape[0] for x in heads),
            "max_abs_o": worst_o, "max_abs_lse": worst_l, "pass": ok,
            "tolerance": "|dO| <= 1e-2 + half a bf16 ulp of the bf16-rounded oracle, |dLSE| <= 1e-3"}


def run_e2e(ea, args, world, dev, stream, fwd_host, dec_host, dec_cache, o, lse, d_o, d_lse, ws,
            fws, fwd_flops_total):
    """The whole step through the public API with host buffers: each step
    copies its inputs from pinned host memory (prefill Q, K, V; the decode
    query and lengths) and reads its results back (both forwards' O and LSE,
    the decode's O and LSE).  Steps are pipelined over three streams: step i's
    host-to-device copies overlap step i-1's kernels and step i-2's copies
    back; device buffers alternate between two sets."""
    q_h, k_h, v_h = fwd_host
    dq_h, dsl_h = dec_host
    dk, dv = dec_cache
    inp_h = [t.pin_memory() for t in (q_h, k_h, v_h, dq_h, dsl_h)]
    res_shapes = [(o[False], lse[False]), (o[True], lse[True]), (d_o, d_lse)]
    outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory()
              for pair in res_shapes for t in pair]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ins = [[torch.empty_like(t, device=dev) for t in inp_h] for _ in range(2)]
    outs = [[torch.empty_like(t) for pair in res_shapes for t in pair] for _ in range(2)]
    dws = [torch.empty_like(ws) for _ in range(2)]
    ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    count = [0]

    def e2e_step():
        i = count[0]
        count[0] += 1
        b = i % 2
        qd, kd, vd, dqd, dsld = ins[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[b])       # step i-2's kernels have read ins[b]
            for dst, src in zip(ins[b], inp_h):
                dst.copy_(src, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])          # step i-2's results have left outs[b]
        ob = outs[b]
        for m, c in enumerate((False, True)):
            ea.attn_fwd(qd, kd, vd, ob[2 * m], ob[2 * m + 1], causal=c, workspace=fws[c],
                        stream=stream)
        ea.attn_decode(dqd, dk, dv, dsld, ob[4], ob[5], workspace=dws[b], stream=stream)
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            for dst, src in zip(outs_h, ob):
                dst.copy_(src, non_blocking=True)
            ev_out[b].record(s_out)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    ranks_barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(args.steps):
        e2e_step()
    e1.record(s_out)
    e1.synchronize()
    torch.cuda.synchronize()
    t_e2e = ranks_max([e0.elapsed_time(e1) / args.steps * 1e-3], world, dev)[0]
    # the last step's results, read back through the pipeline, equal the
    # headline step's (same inputs, deterministic kernels)
    dev_res = [t for pair in res_shapes for t in pair]
    if not all(torch.equal(h, d.cpu()) for h, d in zip(outs_h, dev_res)):
        raise RuntimeError("end-to-end leg returned a different result")
    h2d = sum(t.numel() * t.element_size() for t in inp_h)
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    return {"value": world * fwd_flops_total / t_e2e / 1e12, "unit": "TFLOPS",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * t_e2e,
            "covers": "both prefill forwards and the decode of a step (forward FLOPs over the "
                      "whole step's time)",
            "pipeline": "pinned host buffers; step i's H2D, step i-1's kernels and step i-2's "
                        "D2H on three streams, device buffers double-buffered"}


def run_configs(ea, args, dev, stream, flush, peaks, traffic):
    """The long-context (B1 H32 N16384, outlier channels) and GQA (B8 Hq32
    Hkv8 N4096) causal forwards, each timed alone after an L2 flush."""
    from exact_attention_14_gb300.inputs import GQA, LONG, make_config_inputs
    out = {}
    tr = traffic.get("attn_fwd_kernel", {})
    for cfg, key in ((LONG, "long"), (GQA, "gqa")):
        q, k, v = (t.to(dev) for t in make_config_inputs(cfg))
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        wsz = ea.attn_fwd_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N, cfg.d, True)
        w = torch.empty(max(16, wsz), dtype=torch.uint8, device=dev)
        fn = lambda: ea.attn_fwd(q, k, v, o, lse, causal=True, workspace=w, stream=stream)  # noqa
        for _ in range(args.warmup):
            flush.zero_()
            fn()
        t = time_legs(stream, [fn], max(args.stat_iters, args.steps), flush)[0]
        if ea.attn_last_device_error() != 0:
            raise RuntimeError(f"device error in the {key} leg")
        st = stats_ms(t)
        f = cfg.flops(True)
        tf = f / (st["median_ms"] * 1e-3) / 1e12
        out[key] = {"kernel": "attn_fwd_kernel", "workload":
                    f"{cfg.name}: B={cfg.B} Hq={cfg.Hq} Hkv={cfg.Hkv} N={cfg.N} d={cfg.d}",
                    "tflops": tf, "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
                    "flops": f, "traffic": tr.get(f"{key}_causal"), **st}
        del q, k, v, o, lse, w
    return out


def run_bwd(ea, args, dev, stream, flush, peaks, q, k, v):
    """attn_bwd on the prefill inputs, non-causal then causal, O and LSE from
    attn_fwd."""
    from exact_attention_14_gb300.inputs import PREFILL as cfg
    g = torch.Generator().manual_seed(5)
    dout = torch.randn(q.shape, generator=g, dtype=torch.float32).to(torch.bfloat16).to(dev)
    ob = {c: ea.forward(q, k, v, causal=c, out_dtype=torch.bfloat16, stream=stream)
          for c in (False, True)}
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty(ea.attn_bwd_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N, cfg.d),
                      dtype=torch.uint8, device=dev)
    fns = [lambda c=c: ea.attn_bwd(q, k, v, ob[c][0], dout, ob[c][1], dq, dk, dv, causal=c,
                                   workspace=bws, stream=stream) for c in (False, True)]
    for _ in range(args.warmup):
        flush.zero_()
        for fn in fns:
            fn()
    t_nc, t_c = time_legs(stream, fns, max(args.stat_iters, args.steps), flush, flush_each=True)
    if ea.attn_last_device_error() != 0:
        raise RuntimeError("device error in the backward leg")
    s_nc, s_c = stats_ms(t_nc), stats_ms(t_c)
    f_nc = 2.5 * fwd_flops(cfg.B, cfg.Hq, cfg.N, cfg.d, False)  # five GEMMs per tile
    f_c = 2.5 * fwd_flops(cfg.B, cfg.Hq, cfg.N, cfg.d, True)
    tb_nc, tb_c = s_nc["median_ms"] * 1e-3, s_c["median_ms"] * 1e-3
    return {"kernels": "attn_bwd (prep + K/V-outer dK/dV pass + Q-outer dQ pass)",
            "noncausal_tflops": f_nc / tb_nc / 1e12, "causal_tflops": f_c / tb_c / 1e12,
            "noncausal": s_nc, "causal": s_c,
            "tflops": (f_nc + f_c) / (tb_nc + tb_c) / 1e12,
            "frac_of_bf16_peak": (f_nc + f_c) / (tb_nc + tb_c) / 1e12 / peaks["bf16_tflops"],
            "flops_note": "2.5 x the forward formula (S, dP, dV, dK, dQ products); medians"}


def run_varlen(ea, args, dev, stream, flush, peaks):
    """16 causal sequences of U[256, 4096] tokens in one attn_fwd_varlen."""
    from exact_attention_14_gb300.inputs import VARLEN as vc, make_varlen_inputs, varlen_lengths
    lens = varlen_lengths(vc.n_seqs, vc.len_lo, vc.len_hi, vc.seed)
    vq, vk, vv, vcq, vck = (t.to(dev) for t in make_varlen_inputs(lens, lens, vc.Hq, vc.Hkv,
                                                                   vc.d, vc.seed))
    vo = torch.empty(vq.shape, dtype=torch.bfloat16, device=dev)
    vl = torch.empty((vc.Hq, vq.shape[0]), dtype=torch.float32, device=dev)
    fn = lambda: ea.attn_fwd_varlen(vq, vk, vv, vo, vcq, vck, max(lens), max(lens), vl,  # noqa
                                    causal=vc.causal, scale=vc.scale, stream=stream)
    for _ in range(args.warmup):
        flush.zero_()
        fn()
    st = stats_ms(time_legs(stream, [fn], max(args.stat_iters, args.steps), flush)[0])
    if ea.attn_last_device_error() != 0:
        raise RuntimeError("device error in the varlen leg")
    fv = sum(4.0 * vc.Hq * n * n * vc.d / (2 if vc.causal else 1) for n in lens)
    tv = st["median_ms"] * 1e-3
    return {"kernel": "attn_fwd_kernel (packed, ragged tensor maps)",
            "workload": f"{vc.n_seqs} sequences U[{vc.len_lo},{vc.len_hi}] "
                        f"(total {sum(lens)} tokens, max {max(lens)}) Hq={vc.Hq} "
                        f"Hkv={vc.Hkv} d={vc.d} causal={vc.causal}",
            "tflops": fv / tv / 1e12, "frac_of_bf16_peak": fv / tv / 1e12 / peaks["bf16_tflops"],
            **st, "flops_note": "sum over sequences of the forward formula 4*H*L^2*d (/2 causal)"}


def run_fp8(ea, args, dev, stream, flush, peaks):
    """The long-context causal workload quantized with the random-sign
    Hadamard rotation; the three quantize launches and the attention launch
    are timed separately."""
    from exact_attention_14_gb300.inputs import LONG, hadamard_signs, make_config_inputs
    lq, lk, lv = (t.to(dev) for t in make_config_inputs(LONG))
    signs = hadamard_signs(LONG.d, seed=LONG.seed).to(dev)
    q8, qd = ea.fp8_quantize(lq, signs, stream=stream)
    k8, kd = ea.fp8_quantize(lk, signs, stream=stream)
    vt8, vd = ea.fp8_quantize(lv, None, transpose=True, stream=stream)
    o8 = torch.empty(lq.shape, dtype=torch.bfloat16, device=dev)
    l8 = torch.empty(lq.shape[:3], dtype=torch.float32, device=dev)

    def quant():
        ea.attn_fp8_quantize(lq, q8, qd, signs, stream=stream)
        ea.attn_fp8_quantize(lk, k8, kd, signs, stream=stream)
        ea.attn_fp8_quantize(lv, vt8, vd, None, transpose=True, stream=stream)

    def attn():
        ea.attn_fwd_fp8(q8, k8, vt8, qd, kd, vd, o8, l8, causal=True, scale=LONG.scale,
                        rotated=True, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        quant()
        attn()
    tq_, ta_ = time_legs(stream, [quant, attn], max(args.stat_iters, args.steps), flush)
    if ea.attn_last_device_error() != 0:
        raise RuntimeError("device error in the fp8 leg")
    sq, sa = stats_ms(tq_), stats_ms(ta_)
    tq_, ta_ = sq["median_ms"] * 1e-3, sa["median_ms"] * 1e-3
    f8 = LONG.flops(True)
    n_el = lq.numel() + lk.numel() + lv.numel()
    qbytes = 3 * n_el + 4 * (qd.numel() + kd.numel() + vd.numel())   # bf16 in, E4M3 out
    peak8 = 2 * peaks["bf16_tflops"]
    gemm8 = fp8_gemm_tflops(dev)
    return {"kernels": "attn_fp8_quantize (x3: Q, K rotated; V transposed) + attn_fwd_fp8_kernel",
            "fp8_gemm_measured_tflops": gemm8,
            "attn_frac_of_measured_fp8_gemm": (f8 / ta_ / 1e12 / gemm8) if gemm8 else None,
            "fp8_gemm_note": "context: best of 10 library E4M3 GEMMs (torch._scaled_mm, 8192^3, "
                             "bf16 out) on this GPU in the same run; the roofline peak above "
                             "follows the rule for a dtype without a driver-measured peak",
            "workload": "long-context causal B=1 H=32 N=16384 d=128, 4 outlier channels",
            "attn_tflops": f8 / ta_ / 1e12, "attn": sa,
            "attn_frac_of_fp8_peak": f8 / ta_ / 1e12 / peak8,
            "fp8_peak_tflops": peak8,
            "fp8_peak_source": f"nominal: 2 x {peaks['source']} bf16_tflops (the fp8/bf16 "
                               "dense ratio; no measured fp8 peak)",
            "quantize_gbs": qbytes / tq_ / 1e9, "quantize": sq,
            "quantize_frac_of_hbm": qbytes / tq_ / 1e9 / peaks["hbm_gbs"],
            "with_quantize_tflops": f8 / (ta_ + tq_) / 1e12}


def run_decode_wide(ea, args, dev, stream, flush, peaks, traffic):
    """Split-KV decode at d = 256 (the 256-column kernel): B=16 Hq=32 Hkv=8,
    KV cache [16, 8, 16384, 256] bf16 (the d = 128 workload's cache bytes),
    lengths uniform in [512, 16384].  Timing only (parity is in the tests), so
    the cache is drawn on the GPU from a seeded generator."""
    B, Hq, Hkv, Nmax, d = 16, 32, 8, 16384, 256
    g = torch.Generator(device=dev).manual_seed(7)
    q = torch.randn(B, Hq, 1, d, device=dev, generator=g).to(torch.bfloat16)
    kc = torch.randn(B, Hkv, Nmax, d, device=dev, generator=g).to(torch.bfloat16)
    vc = torch.randn(B, Hkv, Nmax, d, device=dev, generator=g).to(torch.bfloat16)
    sl = torch.randint(512, Nmax + 1, (B,), generator=torch.Generator().manual_seed(7),
                       dtype=torch.int64).to(torch.int32).to(dev)
    o = torch.empty(B, Hq, 1, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Hq, 1, dtype=torch.float32, device=dev)
    ws = torch.empty(ea.attn_decode_workspace_size(B, Hq, Hkv, Nmax, d, 0), dtype=torch.uint8,
                     device=dev)
    fn = lambda: ea.attn_decode(q, kc, vc, sl, o, lse, workspace=ws, stream=stream)  # noqa
    for _ in range(args.warmup):
        flush.zero_()
        fn()
    st = stats_ms(time_legs(stream, [fn], max(args.stat_iters, args.steps), flush)[0])
    if ea.attn_last_device_error() != 0:
        raise RuntimeError("device error in the d=256 decode leg")
    sum_len = int(sl.sum().item())
    nbytes = 2.0 * sum_len * Hkv * d * 2 + q.numel() * 2 + o.numel() * 2 + lse.numel() * 4
    t = st["median_ms"] * 1e-3
    del kc, vc
    return {"kernel": "attn_decode_split_kernel<256> (split-KV, in-kernel merge)",
            "workload": f"decode B={B} Hq={Hq} Hkv={Hkv} Nmax={Nmax} d={d}, lengths U[512,{Nmax}]",
            "gbs": nbytes / t / 1e9, "frac_of_hbm": nbytes / t / 1e9 / peaks["hbm_gbs"],
            "algorithmic_bytes": nbytes, "sum_seqlen": sum_len,
            "traffic": traffic.get("attn_decode_split_kernel", {}).get("decode_d256"), **st}


def fp8_gemm_tflops(dev):
    """A measured E4M3 GEMM rate on this GPU (torch._scaled_mm, 8192^3, best of
    10 CUDA-event timings), reported beside the FP8 leg's nominal peak; None if
    the library path is unavailable."""
    try:
        n = 8192
        a = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), device=dev)
        torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = None
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            e1.record()
            e1.synchronize()
            t = e0.elapsed_time(e1) * 1e-3
            best = t if best is None else min(best, t)
        return 2.0 * n ** 3 / best / 1e12
    except Exception:  # noqa: BLE001 -- context only
        return None


def run_wide(ea, args, dev, stream, flush, peaks):
    """The prefill shape B4 H16 N2048 at d = 256 on the one-Q-tile-per-CTA
    kernel, non-causal and causal, each after an L2 flush."""
    from exact_attention_14_gb300.inputs import PREFILL as cfg, make_fwd_inputs
    wq_, wk_, wv_ = (t.to(dev) for t in make_fwd_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N,
                                                         256, seed=6))
    wo = torch.empty(wq_.shape, dtype=torch.bfloat16, device=dev)
    wl = torch.empty(wq_.shape[:3], dtype=torch.float32, device=dev)
    fns = [lambda c=c: ea.attn_fwd(wq_, wk_, wv_, wo, wl, causal=c, stream=stream)
           for c in (False, True)]
    for _ in range(args.warmup):
        for fn in fns:
            flush.zero_()
            fn()
    t_nc, t_c = time_legs(stream, fns, max(args.stat_iters, args.steps), flush, flush_each=True)
    if ea.attn_last_device_error() != 0:
        raise RuntimeError("device error in the d=256 leg")
    s_nc, s_c = stats_ms(t_nc), stats_ms(t_c)
    fw = [fwd_flops(cfg.B, cfg.Hq, cfg.N, 256, c) for c in (False, True)]
    tw = [s_nc["median_ms"] * 1e-3, s_c["median_ms"] * 1e-3]
    # the backward at d = 256 on the same inputs (O and LSE from the forward)
    g = torch.Generator().manual_seed(8)
    dout = torch.randn(wq_.shape, generator=g, dtype=torch.float32).to(torch.bfloat16).to(dev)
    ob = {c: ea.forward(wq_, wk_, wv_, causal=c, out_dtype=torch.bfloat16, stream=stream)
          for c in (False, True)}
    gq, gk, gv = torch.empty_like(wq_), torch.empty_like(wk_), torch.empty_like(wv_)
    bws = torch.empty(ea.attn_bwd_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N, 256),
                      dtype=torch.uint8, device=dev)
    bfns = [lambda c=c: ea.attn_bwd(wq_, wk_, wv_, ob[c][0], dout, ob[c][1], gq, gk, gv, causal=c,
                                    workspace=bws, stream=stream) for c in (False, True)]
    for _ in range(args.warmup):
        for fn in bfns:
            flush.zero_()
            fn()
    tb_nc, tb_c = time_legs(stream, bfns, max(args.stat_iters, args.steps), flush, flush_each=True)
    if ea.attn_last_device_error() != 0:
        raise RuntimeError("device error in the d=256 backward leg")
    sb_nc, sb_c = stats_ms(tb_nc), stats_ms(tb_c)
    fb = [2.5 * f for f in fw]
    tb = [sb_nc["median_ms"] * 1e-3, sb_c["median_ms"] * 1e-3]
    return {"kernel": "attn_fwd_wide_kernel<256> (one Q tile per CTA, two 128-key S buffers, K/V chunks through one ring)",
            "workload": f"prefill B={cfg.B} H={cfg.Hq} N={cfg.N} d=256",
            "noncausal_tflops": fw[0] / tw[0] / 1e12, "causal_tflops": fw[1] / tw[1] / 1e12,
            "noncausal": s_nc, "causal": s_c,
            "frac_of_bf16_peak": sum(fw) / sum(tw) / 1e12 / peaks["bf16_tflops"],
            "bwd": {"kernels": "attn_bwd at d = 256 (prep + dK/dV pass per column half over "
                               "64-row Q tiles + dQ pass over 64-key tiles)",
                    "noncausal_tflops": fb[0] / tb[0] / 1e12, "causal_tflops": fb[1] / tb[1] / 1e12,
                    "noncausal": sb_nc, "causal": sb_c,
                    "frac_of_bf16_peak": sum(fb) / sum(tb) / 1e12 / peaks["bf16_tflops"],
                    "flops_note": "2.5 x the forward formula (S, dP, dV, dK, dQ products); the "
                                  "dK/dV pass computes S and dP once per column half"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--stat-iters", type=int, default=50,
                    help="iterations per leg for the median/min/max statistics")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the long-context and GQA legs")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward leg")
    ap.add_argument("--no-varlen", action="store_true", help="skip the packed varlen leg")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 leg")
    ap.add_argument("--no-wide", action="store_true", help="skip the d=256 leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
