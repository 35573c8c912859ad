"""Runs one kernel of the library on a named workload a few times, for
profiler captures (ncu) of a single launch configuration.

    python -m exact_attention_14_gb300.profile_case --kernel fwd --workload prefill2x
    python -m exact_attention_14_gb300.profile_case --kernel decode --workload decode
    python -m exact_attention_14_gb300.profile_case --kernel bwd --workload prefill --causal 0

Workloads: prefill (B=4 H=16 N=2048 d=128), prefill2x (B=8: inputs larger
than L2), long (B=1 H=32 N=16384), gqa (B=8 Hq=32 Hkv=8 N=4096), decode
(B=16 Hq=32 Hkv=8 Nmax=32768, lengths 1024..32768) and decode_quarter (the
same with Nmax=8192, lengths 256..8192: a 512 MiB cache, still larger than
L2, for multi-pass captures).  Inputs come from the seeded generators.
"""
from __future__ import annotations

import argparse

import torch

import exact_attention_14_gb300 as ea
from exact_attention_14_gb300.inputs import (DECODE, GQA, LONG, PREFILL, make_decode_config_inputs,
                                             make_decode_inputs, make_fwd_inputs)

FWD = {
    "prefill": PREFILL,
    "prefill2x": PREFILL.__class__(**{**PREFILL.__dict__, "name": "prefill x2", "B": 8}),
    "long": LONG,
    "gqa": GQA,
}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=["fwd", "decode", "bwd"], required=True)
    ap.add_argument("--workload", default="prefill")
    ap.add_argument("--causal", type=int, default=-1, help="-1: the workload's first mode")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    if args.kernel == "bwd":
        cfg = FWD[args.workload]
        causal = cfg.causal[0] if args.causal < 0 else bool(args.causal)
        q, k, v = (t.to(dev) for t in make_fwd_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N, cfg.d,
                                                     cfg.seed, cfg.outlier_channels))
        g = torch.Generator().manual_seed(cfg.seed + 100)
        dout = torch.randn(q.shape, generator=g, dtype=torch.float32).to(torch.bfloat16).to(dev)
        o, lse = ea.forward(q, k, v, causal=causal)
        for _ in range(args.iters):
            ea.backward(q, k, v, o, dout, lse, causal=causal)
    elif args.kernel == "fwd":
        cfg = FWD[args.workload]
        causal = cfg.causal[0] if args.causal < 0 else bool(args.causal)
        q, k, v = (t.to(dev) for t in make_fwd_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N, cfg.d,
                                                     cfg.seed, cfg.outlier_channels))
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        for _ in range(args.iters):
            ea.attn_fwd(q, k, v, o, lse, causal=causal)
    else:
        if args.workload == "decode_quarter":
            host = make_decode_inputs(DECODE.B, DECODE.Hq, DECODE.Hkv, DECODE.Nmax // 4, DECODE.d,
                                      seed=DECODE.seed, len_lo=DECODE.len_lo // 4,
                                      len_hi=DECODE.len_hi // 4)
        else:
            host = make_decode_config_inputs(DECODE)
        q, kc, vc, sl = (t.to(dev) for t in host)
        for _ in range(args.iters):
            ea.decode(q, kc, vc, sl)
    torch.cuda.synchronize()
    if ea.attn_last_device_error() != 0:
        raise SystemExit("device error")
    print("ok")


if __name__ == "__main__":
    main()
