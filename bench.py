#!/usr/bin/env python
"""Benchmark of the fused attention forward + split-KV decode on GB300.

One step = the whole hot path over one batch of synthetic input:
  attn_fwd on the prefill workload (B=4, H=16, N=2048, d=128, bf16) non-causal,
  attn_fwd on the same inputs causal, and
  attn_decode on the decode workload (B=16, Hq=32, Hkv=8, KV cache 32768 x 128,
  valid lengths uniform in [1024, 32768]).
`value` is forward TFLOPS (algorithmic 4*B*H*N*N*d, halved for causal) over the
two forward launches; the decode's HBM GB/s is reported beside it.  Inputs are
resident in HBM; L2 is flushed (a 512 MiB write) between timed steps.

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
    "attn_bwd": ["attn_bwd_sm103.cu", "ptx.cuh", "internal.h"],
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


def oracle_sample(seconds: float, seed: int = 1):
    """Time the fp64 oracle on whole heads of the prefill workload (non-causal
    and causal alternately) until `seconds` of work; returns (TFLOPS, desc, cores)."""
    import numpy as np
    import oracle
    from exact_attention_14_gb300.inputs import PREFILL, make_fwd_inputs
    cfg = PREFILL
    q, k, v = make_fwd_inputs(1, 1, 1, cfg.N, cfg.N, cfg.d, seed=seed)
    oracle.build()
    flops, t0, heads = 0.0, time.perf_counter(), 0
    while True:
        causal = bool(heads % 2)
        oracle.attention(q, k, v, causal=causal, scale=cfg.scale)
        flops += fwd_flops(1, 1, cfg.N, cfg.d, causal)
        heads += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    cores = os.cpu_count() or 1
    desc = (f"{heads} whole heads of the prefill workload (N={cfg.N}, d={cfg.d}), "
            f"alternating non-causal/causal, fp64 three-pass oracle, OpenMP on {cores} threads")
    return flops / el / 1e12, desc, cores, el


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
    steps = []
    for _ in range(args.warmup):
        oracle_sample(1.0)
    total_flops = total_t = 0.0
    cores = os.cpu_count() or 1
    desc = ""
    for _ in range(args.steps):
        tf, desc, cores, el = oracle_sample(3.0)
        total_flops += tf * el * 1e12
        total_t += el
        steps.append(el)
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
    from exact_attention_14_gb300.inputs import DECODE, LONG, PREFILL, VARLEN, hadamard_signs, \
        make_config_inputs, make_decode_config_inputs, make_fwd_inputs, make_varlen_inputs, \
        varlen_lengths

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    ea.load()
    peaks = read_peaks()
    cfg = PREFILL
    q_h, k_h, v_h = make_config_inputs(cfg)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
    dq, dk, dv, dsl = make_decode_config_inputs(DECODE)
    dq, dk, dv, dsl = dq.to(dev), dk.to(dev), dv.to(dev), dsl.to(dev)
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

    def step(ev=None):
        if ev: ev[0].record(stream)
        ea.attn_fwd(q, k, v, o, lse, causal=False, stream=stream)
        if ev: ev[1].record(stream)
        ea.attn_fwd(q, k, v, o, lse, causal=True, stream=stream)
        if ev: ev[2].record(stream)
        ea.attn_decode(dq, dk, dv, dsl, d_o, d_lse, workspace=ws, stream=stream)
        if ev: ev[3].record(stream)

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
    ranks_barrier(world)
    if ea.attn_last_device_error() != 0:
        raise RuntimeError("device error during the timed region")
    t_nc = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps * 1e-3
    t_c = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps * 1e-3
    t_dec = sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps * 1e-3
    t_nc, t_c, t_dec = ranks_max([t_nc, t_c, t_dec], world, dev)
    t_step = t_nc + t_c + t_dec
    tflops = world * (f_nc + f_c) / (t_nc + t_c) / 1e12
    dec_gbs = world * dec_bytes / t_dec / 1e9

    # end to end through the public API: pinned host inputs -> device -> result to host
    e2e = None
    if rank == 0 or world > 1:
        qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
        oh = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
        lh = [torch.empty(lse.shape, dtype=lse.dtype).pin_memory() for _ in range(2)]
        # Steps stream through three CUDA streams: step i's host->device copies
        # (s_in) overlap step i-1's kernels and step i-2's device->host copies
        # (s_out); device buffers alternate between two sets, and events keep
        # each set from being overwritten before its readers are done.
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ins = [tuple(torch.empty_like(t) for t in (q, k, v)) for _ in range(2)]
        outs = [[(torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)] for _ in range(2)]
        ev_in, ev_comp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
        count = [0]

        def e2e_step():
            i = count[0]
            count[0] += 1
            b = i % 2
            qd, kd, vd = ins[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[b])       # step i-2's kernels have read ins[b]
                qd.copy_(qp, non_blocking=True)
                kd.copy_(kp, non_blocking=True)
                vd.copy_(vp, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])          # step i-2's results have left outs[b]
            for m, c in enumerate((False, True)):
                ea.attn_fwd(qd, kd, vd, outs[b][m][0], outs[b][m][1], causal=c, stream=stream)
            ev_comp[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                for m in range(2):
                    oh[m].copy_(outs[b][m][0], non_blocking=True)
                    lh[m].copy_(outs[b][m][1], non_blocking=True)
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
        # the last step's causal result, read back through the pipeline, equals
        # the headline step's (same inputs, deterministic kernel)
        if not (torch.equal(oh[1], o.cpu()) and torch.equal(lh[1], lse.cpu())):
            raise RuntimeError("end-to-end leg returned a different result")
        h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h))
        d2h = sum(t.numel() * t.element_size() for t in oh + lh)
        e2e = {"value": world * (f_nc + f_c) / t_e2e / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": 1e3 * t_e2e,
               "pipeline": "pinned host buffers; step i's H2D, step i-1's two attn_fwd calls and "
                           "step i-2's D2H on three streams, device buffers double-buffered"}

    # Backward (a follow-on row, timed apart from the step): attn_bwd on the
    # prefill inputs, non-causal then causal, O and LSE from attn_fwd.
    bwd = None
    if not args.no_bwd:
        g = torch.Generator().manual_seed(5)
        dout = torch.randn(q.shape, generator=g, dtype=torch.float32).to(torch.bfloat16).to(dev)
        ob = {c: ea.forward(q, k, v, causal=c, out_dtype=torch.bfloat16, stream=stream)
              for c in (False, True)}
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        bws = torch.empty(ea.attn_bwd_workspace_size(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N, cfg.d),
                          dtype=torch.uint8, device=dev)

        def bwd_step(ev=None):
            for idx, c in enumerate((False, True)):
                if ev: ev[idx].record(stream)
                ea.attn_bwd(q, k, v, ob[c][0], dout, ob[c][1], dq, dk, dv, causal=c,
                            workspace=bws, stream=stream)
            if ev: ev[2].record(stream)

        for _ in range(args.warmup):
            flush.zero_()
            bwd_step()
        bev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            bwd_step(bev[i])
        torch.cuda.synchronize()
        if ea.attn_last_device_error() != 0:
            raise RuntimeError("device error in the backward leg")
        tb_nc = sum(e[0].elapsed_time(e[1]) for e in bev) / args.steps * 1e-3
        tb_c = sum(e[1].elapsed_time(e[2]) for e in bev) / args.steps * 1e-3
        fb_nc, fb_c = 2.5 * f_nc, 2.5 * f_c  # five GEMMs per tile against the forward's two
        bwd = {"kernels": "attn_bwd (prep + K/V-outer dK/dV pass + Q-outer dQ pass)",
               "noncausal_tflops": fb_nc / tb_nc / 1e12, "causal_tflops": fb_c / tb_c / 1e12,
               "noncausal_ms": 1e3 * tb_nc, "causal_ms": 1e3 * tb_c,
               "tflops": (fb_nc + fb_c) / (tb_nc + tb_c) / 1e12,
               "frac_of_bf16_peak": (fb_nc + fb_c) / (tb_nc + tb_c) / 1e12 / peaks["bf16_tflops"],
               "flops_note": "2.5 x the forward formula (S, dP, dV, dK, dQ products)"}

    # Packed variable-length prefill (a follow-on row, timed apart from the
    # step): 16 causal sequences of U[256, 4096] tokens in one attn_fwd_varlen.
    varlen = None
    if not args.no_varlen:
        vc = VARLEN
        lens = varlen_lengths(vc.n_seqs, vc.len_lo, vc.len_hi, vc.seed)
        vq, vk, vv, vcq, vck = (t.to(dev) for t in make_varlen_inputs(lens, lens, vc.Hq, vc.Hkv,
                                                                       vc.d, vc.seed))
        vo = torch.empty(vq.shape, dtype=torch.bfloat16, device=dev)
        vl = torch.empty((vc.Hq, vq.shape[0]), dtype=torch.float32, device=dev)

        def varlen_step():
            ea.attn_fwd_varlen(vq, vk, vv, vo, vcq, vck, max(lens), max(lens), vl,
                               causal=vc.causal, scale=vc.scale, stream=stream)

        for _ in range(args.warmup):
            flush.zero_()
            varlen_step()
        vev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            vev[i][0].record(stream)
            varlen_step()
            vev[i][1].record(stream)
        torch.cuda.synchronize()
        if ea.attn_last_device_error() != 0:
            raise RuntimeError("device error in the varlen leg")
        tv = sum(e[0].elapsed_time(e[1]) for e in vev) / args.steps * 1e-3
        fv = sum(4.0 * vc.Hq * n * n * vc.d / (2 if vc.causal else 1) for n in lens)
        varlen = {"kernel": "attn_fwd_kernel (packed, ragged tensor maps)",
                  "workload": f"{vc.n_seqs} sequences U[{vc.len_lo},{vc.len_hi}] "
                              f"(total {sum(lens)} tokens, max {max(lens)}) Hq={vc.Hq} "
                              f"Hkv={vc.Hkv} d={vc.d} causal={vc.causal}",
                  "tflops": fv / tv / 1e12, "ms": 1e3 * tv,
                  "frac_of_bf16_peak": fv / tv / 1e12 / peaks["bf16_tflops"],
                  "flops_note": "sum over sequences of the forward formula 4*H*L^2*d (/2 causal)"}

    # FP8 forward (a follow-on row, timed apart from the step): the long-context
    # causal workload (B1 H32 N16384 d128, 4 outlier channels in Q and K),
    # quantized with the random-sign Hadamard rotation; the three quantize
    # launches and the attention launch are timed separately.
    fp8 = None
    if not args.no_fp8:
        lq, lk, lv = (t.to(dev) for t in make_config_inputs(LONG))
        signs = hadamard_signs(LONG.d, seed=LONG.seed).to(dev)
        q8, qd = ea.fp8_quantize(lq, signs, stream=stream)
        k8, kd = ea.fp8_quantize(lk, signs, stream=stream)
        vt8, vd = ea.fp8_quantize(lv, None, transpose=True, stream=stream)
        o8 = torch.empty(lq.shape, dtype=torch.bfloat16, device=dev)
        l8 = torch.empty(lq.shape[:3], dtype=torch.float32, device=dev)
        eff = LONG.scale / LONG.d

        def quant_step():
            ea.attn_fp8_quantize(lq, q8, qd, signs, stream=stream)
            ea.attn_fp8_quantize(lk, k8, kd, signs, stream=stream)
            ea.attn_fp8_quantize(lv, vt8, vd, None, transpose=True, stream=stream)

        def fp8_step():
            ea.attn_fwd_fp8(q8, k8, vt8, qd, kd, vd, o8, l8, causal=True, scale=eff, stream=stream)

        for _ in range(args.warmup):
            flush.zero_()
            quant_step()
            fp8_step()
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush.zero_()
            fev[i][0].record(stream)
            quant_step()
            fev[i][1].record(stream)
            fp8_step()
            fev[i][2].record(stream)
        torch.cuda.synchronize()
        if ea.attn_last_device_error() != 0:
            raise RuntimeError("device error in the fp8 leg")
        tq_ = sum(e[0].elapsed_time(e[1]) for e in fev) / args.steps * 1e-3
        ta_ = sum(e[1].elapsed_time(e[2]) for e in fev) / args.steps * 1e-3
        f8 = LONG.flops(True)
        n_el = lq.numel() + lk.numel() + lv.numel()
        qbytes = 3 * n_el + 4 * (qd.numel() + kd.numel() + vd.numel())   # bf16 in, E4M3 out
        peak8 = 2 * peaks["bf16_tflops"]
        fp8 = {"kernels": "attn_fp8_quantize (x3: Q, K rotated; V transposed) + attn_fwd_fp8_kernel",
               "workload": "long-context causal B=1 H=32 N=16384 d=128, 4 outlier channels",
               "attn_tflops": f8 / ta_ / 1e12, "attn_ms": 1e3 * ta_,
               "attn_frac_of_fp8_peak": f8 / ta_ / 1e12 / peak8,
               "fp8_peak_tflops": peak8,
               "fp8_peak_source": f"{peaks['source']} bf16_tflops x 2 (nominal fp8/bf16 ratio)",
               "quantize_gbs": qbytes / tq_ / 1e9, "quantize_ms": 1e3 * tq_,
               "quantize_frac_of_hbm": qbytes / tq_ / 1e9 / peaks["hbm_gbs"],
               "with_quantize_tflops": f8 / (ta_ + tq_) / 1e12}

    # Head dim 256 (a follow-on row, timed apart from the step): the prefill
    # shape B4 H16 N2048 at d = 256 on the one-Q-tile-per-CTA kernel.
    wide = None
    if not args.no_wide:
        wq_, wk_, wv_ = (t.to(dev) for t in make_fwd_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N,
                                                             256, seed=6))
        wo = torch.empty(wq_.shape, dtype=torch.bfloat16, device=dev)
        wl = torch.empty(wq_.shape[:3], dtype=torch.float32, device=dev)
        for _ in range(args.warmup):
            for c in (False, True):
                flush.zero_()
                ea.attn_fwd(wq_, wk_, wv_, wo, wl, causal=c, stream=stream)
        wev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        torch.cuda.synchronize()
        for i in range(args.steps):
            for m, c in enumerate((False, True)):
                flush.zero_()
                wev[i][2 * m].record(stream)
                ea.attn_fwd(wq_, wk_, wv_, wo, wl, causal=c, stream=stream)
                wev[i][2 * m + 1].record(stream)
        torch.cuda.synchronize()
        if ea.attn_last_device_error() != 0:
            raise RuntimeError("device error in the d=256 leg")
        tw = [sum(e[2 * m].elapsed_time(e[2 * m + 1]) for e in wev) / args.steps * 1e-3 for m in range(2)]
        fw = [fwd_flops(cfg.B, cfg.Hq, cfg.N, 256, c) for c in (False, True)]
        wide = {"kernel": "attn_fwd_wide_kernel<256> (one Q tile per CTA, 64-key tiles, two S buffers)",
                "workload": f"prefill B={cfg.B} H={cfg.Hq} N={cfg.N} d=256",
                "noncausal_tflops": fw[0] / tw[0] / 1e12, "causal_tflops": fw[1] / tw[1] / 1e12,
                "noncausal_ms": 1e3 * tw[0], "causal_ms": 1e3 * tw[1],
                "frac_of_bf16_peak": sum(fw) / sum(tw) / 1e12 / peaks["bf16_tflops"]}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tf, desc, cores, _ = oracle_sample(args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOPS", "cores": cores, "kind": "oracle", "sample": desc}

    if rank != 0:
        return
    fwd_time = t_nc + t_c
    peak_t = peaks["bf16_tflops"]
    traffic = read_traffic()
    roof = {"bound": "tensor", "kernel": "attn_fwd_kernel (non-causal + causal launches)",
            "achieved": (f_nc + f_c) / fwd_time / 1e12, "peak": peak_t, "unit": "TFLOP/s",
            "frac": (f_nc + f_c) / fwd_time / 1e12 / peak_t,
            "traffic": (traffic["attn_fwd_kernel"]["prefill_noncausal"]
                        + traffic["attn_fwd_kernel"]["prefill_causal"])
                       if "attn_fwd_kernel" in traffic else None,
            "traffic_note": "DRAM bytes of one non-causal + one causal launch (ncu, profiles/); "
                            "algorithmic bytes 2 x 134.7 MB",
            "peak_source": f"{peaks['source']} bf16_tflops (burst)"}
    roof_dec = {"bound": "hbm", "kernel": "attn_decode_split_kernel (split-KV with in-kernel merge)",
                "achieved": dec_bytes / t_dec / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dec_bytes / t_dec / 1e9 / peaks["hbm_gbs"],
                "traffic": traffic["attn_decode_split_kernel"]["decode"]
                           if "attn_decode_split_kernel" in traffic else None,
                "traffic_note": "DRAM bytes per launch (ncu, profiles/); algorithmic bytes in "
                                "decode.algorithmic_bytes",
                "peak_source": f"{peaks['source']} hbm_gbs"}
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
        "roofline": roof, "roofline_decode": roof_dec, "bwd": bwd, "varlen": varlen, "fp8": fp8,
        "wide": wide,
        "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": (2 + ea.attn_decode_kernel_launches(DECODE.B, DECODE.Hq, DECODE.Hkv,
                                                            DECODE.Nmax, DECODE.d)) * args.steps,
        "wall_s_timed_region": wall,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
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
