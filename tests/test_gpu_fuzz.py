"""Seeded random shapes through every entry point against the fp64 oracle:
forward (both kernels, every supported head dim class), packed batches
(forward and backward), backward and decode.  Each case is small (the oracle takes
well under a second), and the draws reach the corners the fixed cases leave
out: head dims from 8 to 256, lengths from 1 up, GQA groups of 1 to 8,
Nq != Nk (bottom-right causal), and the bf16 output."""
import math

import numpy as np
import pytest
import torch

import exact_attention_14_gb300 as ea
import oracle
from exact_attention_14_gb300.inputs import make_decode_inputs, make_fwd_inputs, make_varlen_inputs

from test_gpu_bwd import _check as bwd_check, _dout
from test_gpu_decode import assert_close as dec_close
from test_gpu_fwd import assert_close, assert_close_bf16

pytestmark = pytest.mark.gpu


def _fwd_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        d = int(rng.integers(1, 33)) * 8                 # 8 .. 256
        hkv = int(rng.integers(1, 4))
        group = int(rng.choice([1, 2, 4, 8]))
        causal = bool(rng.integers(0, 2))
        nq = int(rng.integers(1, 700))
        nk = int(rng.integers(nq if causal else 1, 900))
        b = int(rng.integers(1, 3))
        f32 = bool(rng.integers(0, 4) != 0)
        cases.append((b, hkv * group, hkv, nq, nk, d, causal, f32))
    return cases


@pytest.mark.parametrize("case", _fwd_cases(48, 20261202), ids=lambda c: "x".join(map(str, c)))
def test_fuzz_forward(case):
    B, Hq, Hkv, Nq, Nk, d, causal, f32 = case
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=hash(case) % (2 ** 31))
    scale = 1 / math.sqrt(d)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                        out_dtype=torch.float32 if f32 else torch.bfloat16)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    o = o.float().cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    ro, rl = oracle.attention(q, k, v, causal=causal, scale=scale)
    if f32:
        assert_close(o, lse, ro, rl, str(case))
    else:
        assert_close_bf16(o, ro, str(case))
        assert np.abs(lse - rl).max() <= 1e-3


@pytest.mark.parametrize("case", _fwd_cases(24, 777), ids=lambda c: "x".join(map(str, c)))
def test_fuzz_backward(case):
    B, Hq, Hkv, Nq, Nk, d, causal, _ = case
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=hash(case) % (2 ** 31))
    do = _dout(q.shape, seed=hash(case) % 1000 + 1)
    scale = 1 / math.sqrt(d)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                        out_dtype=torch.float32)
    dq, dk, dv = ea.backward(q.cuda(), k.cuda(), v.cuda(), o, do.cuda(), lse, causal=causal,
                             scale=scale, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale)
    for got, ref, n in ((dq, rq, "dQ"), (dk, rk, "dK"), (dv, rv, "dV")):
        bwd_check(got.cpu().double().numpy(), ref, f"{n} {case}")


def _varlen_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        d = int(rng.integers(1, 33)) * 8
        hkv = int(rng.integers(1, 3))
        group = int(rng.choice([1, 2, 4]))
        causal = bool(rng.integers(0, 2))
        nseq = int(rng.integers(1, 6))
        lq = [int(x) for x in rng.integers(0, 400, nseq)]
        lk = [max(x, int(y)) if causal else int(y) for x, y in zip(lq, rng.integers(1, 500, nseq))]
        lk = [max(1, y) if x > 0 else y for x, y in zip(lq, lk)]
        cases.append((tuple(lq), tuple(lk), hkv * group, hkv, d, causal))
    return cases


@pytest.mark.parametrize("case", _varlen_cases(24, 4242), ids=lambda c: str(abs(hash(c)) % 10 ** 8))
def test_fuzz_varlen(case):
    lq, lk, Hq, Hkv, d, causal = case
    if sum(lq) == 0 or sum(lk) == 0:
        pytest.skip("an empty packed batch is rejected by the entry point")
    q, k, v, cu_q, cu_k = make_varlen_inputs(list(lq), list(lk), Hq, Hkv, d, seed=abs(hash(case)) % (2 ** 31))
    scale = 1 / math.sqrt(d)
    o = torch.full(q.shape, float("nan"), dtype=torch.float32).cuda()
    lse = torch.full((Hq, q.shape[0]), float("nan"), dtype=torch.float32).cuda()
    ea.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), o, cu_q.cuda(), cu_k.cuda(), max(max(lq), 1),
                       max(max(lk), 1), lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    ro, rl = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=causal, scale=scale)
    n = int(cu_q[-1])
    assert_close(o.cpu().double().numpy()[:n], lse.cpu().double().numpy()[:, :n], ro[:n], rl[:, :n],
                 str(case))


@pytest.mark.parametrize("case", _varlen_cases(16, 5151), ids=lambda c: str(abs(hash(c)) % 10 ** 8))
def test_fuzz_varlen_backward(case):
    lq, lk, Hq, Hkv, d, causal = case
    if sum(lq) == 0 or sum(lk) == 0:
        pytest.skip("an empty packed batch is rejected by the entry point")
    q, k, v, cu_q, cu_k = make_varlen_inputs(list(lq), list(lk), Hq, Hkv, d, seed=abs(hash(case)) % (2 ** 31))
    do = _dout(q.shape, seed=abs(hash(case)) % 1000 + 3)
    scale = 1 / math.sqrt(d)
    mq, mk = max(max(lq), 1), max(max(lk), 1)
    qd, kd, vd, cq, ck = q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda()
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((Hq, q.shape[0]), dtype=torch.float32, device="cuda")
    ea.attn_fwd_varlen(qd, kd, vd, o, cq, ck, mq, mk, lse, causal=causal, scale=scale)
    dq, dk, dv = ea.backward_varlen(qd, kd, vd, o, do.cuda(), lse, cq, ck, mq, mk, causal=causal,
                                    scale=scale, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    rq, rk, rv = oracle.attention_bwd_varlen(q, k, v, do, cu_q, cu_k, causal=causal, scale=scale)
    for got, ref, n in ((dq, rq, "dQ"), (dk, rk, "dK"), (dv, rv, "dV")):
        bwd_check(got.cpu().double().numpy(), ref, f"{n} {case}")


def _decode_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        d = int(rng.integers(1, 33)) * 8
        hkv = int(rng.integers(1, 5))
        group = int(rng.choice([1, 2, 4, 8, 16]))
        b = int(rng.integers(1, 6))
        nmax = int(rng.integers(1, 3000))
        lo = int(rng.integers(1, nmax + 1))
        splits = int(rng.choice([0, 0, 1, 3, 16]))
        cases.append((b, hkv * group, hkv, nmax, d, lo, splits))
    return cases


@pytest.mark.parametrize("case", _decode_cases(32, 99), ids=lambda c: "x".join(map(str, c)))
def test_fuzz_decode(case):
    B, Hq, Hkv, Nmax, d, lo, splits = case
    q, kc, vc, sl = make_decode_inputs(B, Hq, Hkv, Nmax, d, seed=hash(case) % (2 ** 31), len_lo=lo,
                                       len_hi=Nmax, tail="nan")
    o, lse = ea.decode(q.cuda(), kc.cuda(), vc.cuda(), sl.cuda(), num_splits=splits,
                       out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
    dec_close(o.cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref, str(case))
