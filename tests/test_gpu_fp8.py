"""GPU parity of the FP8 path against the FP8 oracle, through the C ABI.

attn_fp8_quantize is integer work once its fp32 arithmetic is fixed (the
rotation's butterflies, the block amax, the two scale divisions, the scaled
products): its codes and scales must equal the oracle's bit for bit.

attn_fwd_fp8 runs on codes made by the oracle's quantizer and is compared with
exact attention over the dequantized operands.  Its one approximation beyond
fp32 accumulation is the E4M3 rounding of the probabilities: every element of
O must lie within the oracle's bound for that rounding (2^-3 sum_j P_ij |V_jc|
+ 2^-8 max|V|), the relative L2 error of O must stay below 2^-4 (the largest
relative rounding of a normal E4M3 value; with V independent of the rounding,
O and its error both scale with sqrt(sum_j P_ij^2), so the relative error is
the root-mean-square relative rounding, about 2^-4 / sqrt(3)), and max |dLSE|
<= 1e-3 (the LSE comes from the unrounded probabilities).
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_14_gb300 as ea
import oracle
from oracle import fp8
from exact_attention_14_gb300.inputs import (LONG, FwdConfig, hadamard_signs, make_config_inputs,
                                             make_fwd_inputs)

pytestmark = pytest.mark.gpu

REL_L2 = 2.0 ** -4
MAX_LSE = 1e-3


@pytest.mark.parametrize("B,H,N,rotate,transpose", [
    (1, 1, 128, False, False), (2, 3, 300, True, False), (1, 4, 1, True, False),
    (2, 2, 300, False, True), (1, 1, 1000, False, True), (1, 2, 130, True, True),
])
def test_quantize_bit_exact(B, H, N, rotate, transpose):
    x, _, _ = make_fwd_inputs(B, H, H, N, N, 128, seed=900 + N)
    s = hadamard_signs(128, seed=901) if rotate else None
    codes, ds = ea.fp8_quantize(x.cuda(), None if s is None else s.cuda(), transpose=transpose)
    torch.cuda.synchronize()
    rc, rd = fp8.quantize(x, signs=s, transpose=transpose)
    assert np.array_equal(ds.cpu().numpy(), rd)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quantize_outliers_and_zero_blocks():
    q, k, _ = make_config_inputs(FwdConfig("o", 1, 2, 2, 700, 128, (True,), seed=LONG.seed,
                                           outlier_channels=4))
    q[0, 1, 128:256] = 0
    s = hadamard_signs(128, seed=902)
    for x, sg in ((q, s), (k, None)):
        codes, ds = ea.fp8_quantize(x.cuda(), None if sg is None else sg.cuda())
        rc, rd = fp8.quantize(x, signs=sg)
        assert np.array_equal(ds.cpu().numpy(), rd) and np.array_equal(codes.cpu().numpy(), rc)


def _oracle_operands(q, k, v, signs):
    q8, qd = fp8.quantize(q, signs=signs)
    k8, kd = fp8.quantize(k, signs=signs)
    vt8, vd = fp8.quantize(v, transpose=True)
    return q8, k8, vt8, qd, kd, vd


def _run_fp8(ops, causal, scale, out_dtype=torch.float32, rotated=False):
    """The kernel on the oracle's codes; `scale` is the original problem's
    (the kernel divides it by d when rotated)."""
    q8, k8, vt8, qd, kd, vd = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in ops)
    B, Hq, Nq, d = q8.shape
    o = torch.empty((B, Hq, Nq, d), dtype=out_dtype, device="cuda")
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device="cuda")
    ea.attn_fwd_fp8(q8, k8, vt8, qd, kd, vd, o, lse, causal=causal, scale=scale, rotated=rotated)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def _check(o, lse, ro, rl, bound, what):
    assert np.isfinite(o).all(), what
    err = np.abs(o - ro)
    assert (err <= bound).all(), f"{what}: {(err / bound).max():.3f} of the bound"
    rel = np.linalg.norm(o - ro) / np.linalg.norm(ro)
    assert rel <= REL_L2, f"{what}: relL2 {rel:.3e}"
    assert np.abs(lse - rl).max() <= MAX_LSE, f"{what}: LSE {np.abs(lse - rl).max():.3e}"


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,causal,rotate", [
    (1, 1, 1, 128, 128, False, False),
    (2, 4, 2, 300, 300, True, True),       # GQA, ragged tails, rotated
    (1, 4, 1, 200, 520, False, True),      # MQA, Nq < Nk
    (1, 2, 2, 100, 333, True, False),      # bottom-right causal
    (1, 4, 4, 1000, 1000, True, True),
])
def test_fwd_fp8_parity(B, Hq, Hkv, Nq, Nk, causal, rotate):
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, 128, seed=910 + Nq + Nk)
    s = hadamard_signs(128, seed=911) if rotate else None
    scale = 1 / math.sqrt(128)
    eff = scale / 128 if rotate else scale   # rotated operands' scores carry a factor d
    ops = _oracle_operands(q, k, v, s)
    o, lse = _run_fp8(ops, causal, scale, rotated=rotate)
    ro, rl, bound = fp8.attention_fp8(*ops[:3], *ops[3:], Nk, causal=causal, scale=eff)
    _check(o, lse, ro, rl, bound, f"{(B, Hq, Hkv, Nq, Nk, causal, rotate)}")


def test_fwd_fp8_bf16_output_and_one_hot_rows():
    """A +40 score on one key per row: the row's output is that key's V row
    (the largest probability's rounding is carried into the normaliser)."""
    q, k, v = make_fwd_inputs(1, 2, 2, 256, 256, 128, seed=920)
    ops = list(_oracle_operands(q, k, v, None))
    o, _ = _run_fp8(ops, False, 1 / math.sqrt(128), out_dtype=torch.bfloat16)
    ro, _, bound = fp8.attention_fp8(*ops[:3], *ops[3:], 256, causal=False,
                                     scale=1 / math.sqrt(128))
    assert (np.abs(o - ro) <= bound + 2.0 ** -8 * np.abs(ro)).all()
    # one-hot: scores scaled so that key i dominates row i
    q8 = np.zeros((1, 1, 128, 128), np.uint8)
    k8 = np.zeros((1, 1, 128, 128), np.uint8)
    for i in range(128):
        q8[0, 0, i, i] = 0x7E     # 448
        k8[0, 0, i, i] = 0x7E
    vt8, vd = fp8.quantize(v[:, :1, :128], transpose=True)
    ones = np.ones((1, 1, 1), np.float32)
    ops1 = (q8, k8, vt8, ones * (1 / 448.0), ones * (1 / 448.0), vd)
    o1, _ = _run_fp8(ops1, False, 40.0)
    ro1, _, _ = fp8.attention_fp8(q8, k8, vt8, *ops1[3:], 128, causal=False, scale=40.0)
    assert np.abs(o1 - ro1).max() <= 1e-5


def test_fwd_fp8_long_context_sampled():
    """The long-context workload at full size (B1 H32 N16384 d128, causal,
    4 outlier channels), rotated; the oracle checks sampled rows."""
    q, k, v = make_config_inputs(LONG)
    s = hadamard_signs(128, seed=LONG.seed)
    scale = LONG.scale / 128    # over the rotated operands
    ops = _oracle_operands(q, k, v, s)
    o, lse = _run_fp8(ops, True, LONG.scale, out_dtype=torch.bfloat16, rotated=True)
    rng = np.random.default_rng(5)
    rows = np.stack([np.zeros(48, int), rng.integers(0, 32, 48),
                     np.concatenate([rng.integers(0, 16384, 40), np.arange(8) * 2047])], 1)
    ro, rl, bound = fp8.attention_fp8_rows(*ops[:3], *ops[3:], 16384, rows, causal=True,
                                           scale=scale)
    got = np.stack([o[b, h, i] for b, h, i in rows])
    gl = np.array([lse[b, h, i] for b, h, i in rows])
    assert (np.abs(got - ro) <= bound + 2.0 ** -8 * np.abs(ro)).all()   # + bf16 output rounding
    assert np.abs(gl - rl).max() <= MAX_LSE


def test_forward_fp8_end_to_end_rotation_helps():
    """bf16 -> quantize -> attention, against exact attention on the bf16
    inputs, with outlier channels shared by Q and K: the rotation lowers the
    error of O (lecture notes 4.4)."""
    q, k, v = make_config_inputs(FwdConfig("o", 1, 4, 4, 1024, 128, (True,), seed=LONG.seed,
                                           outlier_channels=4))
    ro, _ = oracle.attention(q, k, v, causal=True)
    errs = []
    for s in (None, hadamard_signs(128, seed=7)):
        o, _ = ea.forward_fp8(q.cuda(), k.cuda(), v.cuda(), causal=True,
                              signs=None if s is None else s.cuda(), out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert ea.attn_last_device_error() == 0
        on = o.cpu().double().numpy()
        errs.append(np.linalg.norm(on - ro) / np.linalg.norm(ro))
    assert errs[0] / errs[1] > 1.5, errs   # measured 3.4x (the pages: 1.6x on their data)
