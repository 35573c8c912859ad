"""Runs one kernel of the library on a named workload a few times, for
profiler captures (ncu) of a single launch configuration.

    python profile_case.py --kernel fwd --workload prefill2x
    python profile_case.py --kernel decode --workload decode
    python profile_case.py --kernel bwd --workload prefill --causal 0
    python profile_case.py --kernel fp8 --workload long
    python profile_case.py --kernel fp8quant --workload long
    python profile_case.py --kernel varlen

Workloads: prefill (B=4 H=16 N=2048 d=128), prefill2x (B=8: inputs larger
than L2), prefill256 (the prefill shape at d=256), long (B=1 H=32 N=16384), gqa (B=8 Hq=32 Hkv=8 N=4096), decode
(B=16 Hq=32 Hkv=8 Nmax=32768, lengths 1024..32768) and decode_quarter (the
same with Nmax=8192, lengths 256..8192: a 512 MiB cache, still larger than
L2, for multi-pass captures), decode256 (d = 256: B=16 Hq=32 Hkv=8 Nmax=16384,
lengths 512..16384); varlen is the packed causal prefill batch (16
sequences of 256..4096 tokens).  fp8 runs attn_fwd_fp8 on E4M3 operands of the
workload (Q and K rotated by the random-sign Hadamard matrix), fp8quant the
rotating quantization of its Q.  Inputs come from the seeded generators.
"""
from __future__ import annotations

import argparse

import torch

import exact_attention_14_gb300 as ea
from exact_attention_14_gb300.inputs import (DECODE, GQA, LONG, PREFILL, VARLEN, hadamard_signs,
                                             make_decode_config_inputs, make_decode_inputs,
                                             make_fwd_inputs, make_varlen_inputs, varlen_lengths)

FWD = {
    "prefill": PREFILL,
    "prefill2x": PREFILL.__class__(**{**PREFILL.__dict__, "name": "prefill x2", "B": 8}),
    "prefill256": PREFILL.__class__(**{**PREFILL.__dict__, "name": "prefill d256", "d": 256,
                                       "seed": 6}),
    "long": LONG,
    "gqa": GQA,
}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=["fwd", "decode", "bwd", "fp8", "fp8quant", "varlen"],
                    required=True)
    ap.add_argument("--workload", default="prefill")
    ap.add_argument("--causal", type=int, default=-1, help="-1: the workload's first mode")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    if args.kernel in ("fp8", "fp8quant"):
        cfg = FWD[args.workload]
        causal = cfg.causal[0] if args.causal < 0 else bool(args.causal)
        q, k, v = (t.to(dev) for t in make_fwd_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N, cfg.d,
                                                     cfg.seed, cfg.outlier_channels))
        signs = hadamard_signs(cfg.d, seed=cfg.seed).to(dev)
        q8, qd = ea.fp8_quantize(q, signs)
        k8, kd = ea.fp8_quantize(k, signs)
        vt8, vd = ea.fp8_quantize(v, None, transpose=True)
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        for _ in range(args.iters):
            if args.kernel == "fp8":
                ea.attn_fwd_fp8(q8, k8, vt8, qd, kd, vd, o, lse, causal=causal,
                                scale=cfg.scale, rotated=True)
            else:
                ea.attn_fp8_quantize(q, q8, qd, signs)
    elif args.kernel == "varlen":
        lens = varlen_lengths(VARLEN.n_seqs, VARLEN.len_lo, VARLEN.len_hi, VARLEN.seed)
        q, k, v, cq, ck = (t.to(dev) for t in make_varlen_inputs(lens, lens, VARLEN.Hq, VARLEN.Hkv,
                                                                 VARLEN.d, VARLEN.seed))
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty((VARLEN.Hq, q.shape[0]), dtype=torch.float32, device=dev)
        for _ in range(args.iters):
            ea.attn_fwd_varlen(q, k, v, o, cq, ck, max(lens), max(lens), lse, causal=VARLEN.causal)
    elif args.kernel == "bwd":
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
    elif args.workload == "decode256":
        # decode at d = 256: B16 Hq32 Hkv8, cache [16, 8, 16384, 256], lengths U[512, 16384]
        # (the bench's d = 256 decode leg; drawn on the GPU from seeded generators)
        g = torch.Generator(device=dev).manual_seed(7)
        q = torch.randn(16, 32, 1, 256, device=dev, generator=g).to(torch.bfloat16)
        kc = torch.randn(16, 8, 16384, 256, device=dev, generator=g).to(torch.bfloat16)
        vc = torch.randn(16, 8, 16384, 256, device=dev, generator=g).to(torch.bfloat16)
        sl = torch.randint(512, 16385, (16,), generator=torch.Generator().manual_seed(7),
                           dtype=torch.int64).to(torch.int32).to(dev)
        for _ in range(args.iters):
            ea.decode(q, kc, vc, sl)
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
