"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic.  Every tensor is drawn on the CPU with a
``torch.Generator`` so the same seed gives the same bits on any machine, then
handed unchanged to both the CUDA library and the CPU oracle.

Workload recipes follow the five configurations the library is measured on:
values i.i.d. N(0, 1) drawn in fp32 and rounded to bf16 (round-to-nearest-even);
the long-context case scales 4 head-dim channels per head by 8 in Q and K (the
same channels in both -- the reading that keeps the outliers aligned in QK^T);
decode draws each sequence's valid length uniformly from an inclusive integer
range and fills the cache tail (positions >= length) with N(0, 1) or, for the
leak test, with NaN.  Packed variable-length batches draw each sequence's
length uniformly from an inclusive range and lay the sequences end to end.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class FwdConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: tuple  # causal modes the config is run in
    seed: int
    outlier_channels: int = 0
    outlier_scale: float = 8.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self, causal: bool) -> float:
        """Algorithmic FLOPs: 4*B*Hq*Nq*Nk*d, halved for causal."""
        f = 4.0 * self.B * self.Hq * self.N * self.N * self.d
        return f / 2 if causal else f


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    Hq: int
    Hkv: int
    Nmax: int
    d: int
    len_lo: int
    len_hi: int
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads, seeds 0..4 in this order.
TINY = FwdConfig("tiny fwd", 1, 1, 1, 256, 64, (False,), seed=0)
PREFILL = FwdConfig("prefill fwd", 4, 16, 16, 2048, 128, (False, True), seed=1)
LONG = FwdConfig("long-context causal fwd", 1, 32, 32, 16384, 128, (True,), seed=2,
                 outlier_channels=4)
GQA = FwdConfig("GQA causal fwd", 8, 32, 8, 4096, 128, (True,), seed=3)
DECODE = DecodeConfig("decode split-KV", 16, 32, 8, 32768, 128, 1024, 32768, seed=4)

FWD_CONFIGS = (TINY, PREFILL, LONG, GQA)


@dataclass(frozen=True)
class VarlenConfig:
    """A packed batch of n_seqs sequences, each of length U[len_lo, len_hi]
    (the same length for its queries and keys)."""
    name: str
    n_seqs: int
    Hq: int
    Hkv: int
    d: int
    len_lo: int
    len_hi: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# A prefill batch of mixed lengths, 16 sequences of 256..4096 tokens.
VARLEN = VarlenConfig("varlen causal prefill", 16, 16, 16, 128, 256, 4096, True, seed=5)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def make_fwd_inputs(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, seed: int,
                    outlier_channels: int = 0, outlier_scale: float = 8.0):
    """q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d] as bf16 CPU tensors (contiguous)."""
    g = _gen(seed)
    q = torch.randn(B, Hq, Nq, d, dtype=torch.float32, generator=g)
    k = torch.randn(B, Hkv, Nk, d, dtype=torch.float32, generator=g)
    v = torch.randn(B, Hkv, Nk, d, dtype=torch.float32, generator=g)
    if outlier_channels > 0:
        group = Hq // Hkv
        for b in range(B):
            for h in range(Hkv):
                ch = torch.randperm(d, generator=g)[:outlier_channels]
                k[b, h, :, ch] *= outlier_scale
                q[b, h * group:(h + 1) * group, :, ch] *= outlier_scale
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def make_config_inputs(cfg: FwdConfig):
    return make_fwd_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.N, cfg.N, cfg.d, cfg.seed,
                           cfg.outlier_channels, cfg.outlier_scale)


def make_decode_inputs(B: int, Hq: int, Hkv: int, Nmax: int, d: int, seed: int,
                       len_lo: int, len_hi: int, tail: str = "normal"):
    """q [B,Hq,1,d], k/v caches [B,Hkv,Nmax,d] (bf16), seqlens [B] int32.

    tail: "normal" keeps the N(0,1) draws past each length; "nan" overwrites
    them with NaN so a kernel that reads them shows it."""
    g = _gen(seed)
    q = torch.randn(B, Hq, 1, d, dtype=torch.float32, generator=g)
    kc = torch.randn(B, Hkv, Nmax, d, dtype=torch.float32, generator=g)
    vc = torch.randn(B, Hkv, Nmax, d, dtype=torch.float32, generator=g)
    seqlens = torch.randint(len_lo, len_hi + 1, (B,), generator=g, dtype=torch.int64)
    seqlens = seqlens.to(torch.int32)
    q, kc, vc = (t.to(torch.bfloat16) for t in (q, kc, vc))
    if tail == "nan":
        for b in range(B):
            L = int(seqlens[b])
            kc[b, :, L:, :] = float("nan")
            vc[b, :, L:, :] = float("nan")
    elif tail != "normal":
        raise ValueError(f"unknown tail fill {tail!r}")
    return q.contiguous(), kc.contiguous(), vc.contiguous(), seqlens


def make_decode_config_inputs(cfg: DecodeConfig, tail: str = "normal"):
    return make_decode_inputs(cfg.B, cfg.Hq, cfg.Hkv, cfg.Nmax, cfg.d, cfg.seed,
                              cfg.len_lo, cfg.len_hi, tail=tail)


def varlen_lengths(n_seqs: int, len_lo: int, len_hi: int, seed: int) -> list:
    """n_seqs lengths drawn uniformly from [len_lo, len_hi] (inclusive)."""
    g = _gen(seed)
    return torch.randint(len_lo, len_hi + 1, (n_seqs,), generator=g).tolist()


def make_varlen_inputs(lens_q, lens_k, Hq: int, Hkv: int, d: int, seed: int,
                       extra_rows: int = 0, extra_value: float = float("nan")):
    """Packed q [total_q, Hq, d], k, v [total_k, Hkv, d] (bf16, CPU) for
    sequences of lengths lens_q / lens_k laid end to end, and the row offsets
    cu_q, cu_k (int32 [B + 1]).  extra_rows rows past the last sequence hold
    extra_value (they belong to no sequence)."""
    g = _gen(seed)
    cu_q = [0]
    for n in lens_q:
        cu_q.append(cu_q[-1] + int(n))
    cu_k = [0]
    for n in lens_k:
        cu_k.append(cu_k[-1] + int(n))
    tq, tk = cu_q[-1] + extra_rows, cu_k[-1] + extra_rows
    q = torch.randn((tq, Hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((tk, Hkv, d), generator=g, dtype=torch.float32)
    v = torch.randn((tk, Hkv, d), generator=g, dtype=torch.float32)
    if extra_rows:
        q[cu_q[-1]:] = extra_value
        k[cu_k[-1]:] = extra_value
        v[cu_k[-1]:] = extra_value
    return (q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16),
            torch.tensor(cu_q, dtype=torch.int32), torch.tensor(cu_k, dtype=torch.int32))


def make_outlier_inputs(B: int, Hq: int, Hkv: int, N: int, d: int, seed: int,
                        frac: float = 1e-3, magnitude: float = 25.0):
    """q [B,Hq,N,d], k, v [B,Hkv,N,d] bf16: N(0, 1) values with a fraction
    `frac` of the entries of q and k (random positions) replaced by
    +-magnitude (random signs) -- normal data with rare large values."""
    g = _gen(seed)
    q = torch.randn((B, Hq, N, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, Hkv, N, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, Hkv, N, d), generator=g, dtype=torch.float32)
    for t in (q, k):
        hit = torch.rand(t.shape, generator=g) < frac
        sgn = torch.where(torch.rand(t.shape, generator=g) < 0.5, -1.0, 1.0)
        t[hit] = (magnitude * sgn)[hit]
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def hadamard_signs(d: int, seed: int) -> torch.Tensor:
    """d random signs (int8, +-1) for the rotation of Q and K."""
    g = _gen(seed)
    return torch.where(torch.rand(d, generator=g) < 0.5, -1, 1).to(torch.int8)
