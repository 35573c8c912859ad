"""Pins of the FP8 oracle (CPU).

- E4M3 rounding and decoding against torch's float8_e4m3fn conversion (a
  library routine), over every code and over random and tie values;
  saturation at 448 from the format's definition.
- The fp32 fast Walsh-Hadamard transform against scipy's Hadamard matrix
  (exact on integer inputs; within fp32 rounding otherwise) and the identity
  (Q D H)(K D H)^T = d Q K^T.
- Block quantization: the block's largest magnitude encodes as +-448, every
  value is within half an E4M3 spacing, all-zero blocks, the transposed layout,
  ragged last blocks.
- attention_fp8 against the C oracle when the dequantized values are exact in
  bf16.
- The pages' claim (lecture notes 4.4): with outlier channels shared by Q and
  K the rotation lowers the quantization error of Q K^T (and, E4M3 being a
  float format, isolated large values leave it nothing to gain).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from exact_attention_14_gb300.inputs import (LONG, FwdConfig, hadamard_signs, make_config_inputs,
                                             make_fwd_inputs, make_outlier_inputs)

scipy_linalg = pytest.importorskip("scipy.linalg")


def test_decode_every_code_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    got = fp8.e4m3_decode(codes)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(np.where(both_nan, 0, got), np.where(both_nan, 0, ref))


def test_rounding_matches_torch():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    # exact ties between neighbouring E4M3 values (round half to even)
    vals = fp8.e4m3_decode(np.arange(0, 126, dtype=np.uint8))
    mids = torch.from_numpy(((vals[:-1] + vals[1:]) / 2).astype(np.float32))
    x = torch.cat([x, mids, -mids]).clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = fp8.e4m3_encode(x.numpy())
    assert np.array_equal(got, ref)


def test_saturation_and_signed_zero():
    assert fp8.e4m3_round(np.float32(500.0)) == 448.0
    assert fp8.e4m3_round(np.float32(-1e9)) == -448.0
    assert fp8.e4m3_encode(np.float32(460.0)) == 0x7E
    assert fp8.e4m3_encode(np.float32(-1e-6)) == 0x80       # rounds to -0
    assert fp8.e4m3_encode(np.float32(2.0 ** -9)) == 0x01   # smallest subnormal


def test_fwht_matches_hadamard_matrix():
    d = 128
    H = scipy_linalg.hadamard(d).astype(np.float64)
    rng = np.random.default_rng(4)
    xi = rng.integers(-50, 50, size=(7, d)).astype(np.float32)
    assert np.array_equal(fp8.fwht_f32(xi).astype(np.float64), xi.astype(np.float64) @ H)
    xr = rng.standard_normal((9, d)).astype(np.float32)
    ref = xr.astype(np.float64) @ H
    assert np.abs(fp8.fwht_f32(xr) - ref).max() <= 1e-5 * np.abs(ref).max()
    for dd in (8, 64):
        Hd = scipy_linalg.hadamard(dd).astype(np.float64)
        xs = rng.integers(-9, 9, size=(3, dd)).astype(np.float32)
        assert np.array_equal(fp8.fwht_f32(xs).astype(np.float64), xs.astype(np.float64) @ Hd)


def test_rotation_preserves_scores_up_to_d():
    d = 64
    rng = np.random.default_rng(5)
    q = rng.integers(-8, 8, size=(10, d)).astype(np.float32)
    k = rng.integers(-8, 8, size=(12, d)).astype(np.float32)
    s = np.where(rng.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
    qr, kr = fp8.fwht_f32(q * s), fp8.fwht_f32(k * s)     # exact for integers
    assert np.array_equal(qr.astype(np.float64) @ kr.T.astype(np.float64),
                          d * (q.astype(np.float64) @ k.T.astype(np.float64)))


def test_quantize_block_properties():
    q, _, _ = make_fwd_inputs(2, 3, 3, 300, 300, 128, seed=6)
    codes, ds = fp8.quantize(q)
    assert codes.shape == (2, 3, 300, 128) and ds.shape == (2, 3, 3)
    x = q.float().numpy().astype(np.float64)
    deq = fp8.dequantize(codes, ds, 300)
    for b in range(2):
        for h in range(3):
            for blk in range(3):
                rows = slice(128 * blk, min(300, 128 * blk + 128))
                xb, db = x[b, h, rows], deq[b, h, rows]
                amax = np.abs(xb).max()
                assert ds[b, h, blk] == np.float32(np.float32(amax) / np.float32(448))
                i = np.unravel_index(np.abs(xb).argmax(), xb.shape)
                assert abs(fp8.e4m3_decode(codes[b, h, rows][i])) == 448.0
                sub = np.abs(xb) < 2.0 ** -6 * ds[b, h, blk]   # inputs in the subnormal range
                err = np.abs(db - xb)
                tol = np.where(sub, 2.0 ** -10 * ds[b, h, blk], 2.0 ** -4 * np.abs(xb))
                assert (err <= tol * (1 + 1e-6) + 1e-12).all()


def test_quantize_zero_block_transpose_and_rotation():
    x = torch.zeros((1, 2, 200, 64), dtype=torch.bfloat16)
    x[0, 1, 150] = 3.0
    codes, ds = fp8.quantize(x)
    assert ds[0, 0, 0] == 1.0 and ds[0, 0, 1] == 1.0 and not codes[0, 0].any()
    assert ds[0, 1, 0] == 1.0 and ds[0, 1, 1] == np.float32(3.0) / np.float32(448.0)
    q, _, _ = make_fwd_inputs(1, 2, 2, 130, 130, 64, seed=7)
    c, d1 = fp8.quantize(q)
    t, d2 = fp8.quantize(q, transpose=True)
    assert t.shape == (1, 2, 64, 144) and np.array_equal(d1, d2)
    assert np.array_equal(t[..., :130], c.transpose(0, 1, 3, 2)) and not t[..., 130:].any()
    s = hadamard_signs(64, seed=8)
    cr, dr = fp8.quantize(q, signs=s)
    rot = fp8.fwht_f32(q.float().numpy() * s.numpy().astype(np.float32))
    ref_c, ref_d = fp8.quantize(rot)
    assert np.array_equal(cr, ref_c) and np.array_equal(dr, ref_d)


def test_attention_fp8_matches_c_oracle_on_exact_values():
    rng = np.random.default_rng(9)
    B, Hq, Hkv, N, d = 1, 4, 2, 200, 64

    def rand_codes(shape):
        c = rng.integers(0, 0x7E, size=shape).astype(np.uint8)
        return c | (rng.integers(0, 2, size=shape).astype(np.uint8) << 7)

    q8, k8 = rand_codes((B, Hq, N, d)), rand_codes((B, Hkv, N, d))
    vt8 = rand_codes((B, Hkv, d, 208))
    ds = lambda h: np.full((B, h, 2), 2.0 ** -7, np.float32)  # noqa: E731
    for causal in (False, True):
        o, lse, _ = fp8.attention_fp8(q8, k8, vt8, ds(Hq), ds(Hkv), ds(Hkv), N, causal=causal,
                                      scale=0.05)
        qb = torch.from_numpy(fp8.dequantize(q8, ds(Hq), N)).to(torch.bfloat16)
        kb = torch.from_numpy(fp8.dequantize(k8, ds(Hkv), N)).to(torch.bfloat16)
        vb = torch.from_numpy(fp8.dequantize(vt8, ds(Hkv), N, transposed=True)).to(torch.bfloat16)
        assert np.array_equal(qb.double().numpy(), fp8.dequantize(q8, ds(Hq), N))  # exact in bf16
        ro, rl = oracle.attention(qb, kb, vb, causal=causal, scale=0.05)
        assert np.abs(o - ro).max() < 1e-12 and np.abs(lse - rl).max() < 1e-12


def _score_error(q, k, signs):
    qf, kf = q.double().numpy()[0, 0], k.double().numpy()[0, 0]
    exact = qf @ kf.T
    cq, dq = fp8.quantize(q, signs=signs)
    ck, dk = fp8.quantize(k, signs=signs)
    sc = fp8.dequantize(cq, dq, q.shape[2])[0, 0] @ fp8.dequantize(ck, dk, k.shape[2])[0, 0].T
    if signs is not None:
        sc = sc / q.shape[3]
    return np.linalg.norm(sc - exact) / np.linalg.norm(exact)


def test_rotation_lowers_score_error_with_outlier_channels():
    """Lecture notes 4.4 / FA3 notes: outliers in the same channels of Q and K
    (the long-context workload's recipe, N = 1024, d = 128).  E4M3 rounds
    relative to each value, so the score error of a dot product grows with
    sum_c q_c^2 k_c^2, which aligned outlier channels dominate; the rotation
    spreads them over all channels and the error falls."""
    cfg = LONG
    q, k, _ = make_config_inputs(FwdConfig("outlier channels", 1, 1, 1, 1024, 128, (True,),
                                           seed=cfg.seed, outlier_channels=4))
    s = hadamard_signs(128, seed=11)
    plain, rotated = _score_error(q, k, None), _score_error(q, k, s)
    assert plain / rotated > 1.5, (plain, rotated)
    # max / RMS of Q falls (the pages: 26.9 -> 5.0 on their data)
    qf = q.float().numpy()[0, 0]
    qr = fp8.fwht_f32(qf * s.numpy().astype(np.float32))
    ratio = lambda a: np.abs(a).max() / np.sqrt((a.astype(np.float64) ** 2).mean())  # noqa: E731
    assert ratio(qf) > 2 * ratio(qr)


def test_rotation_gains_nothing_for_isolated_outliers():
    """With the large values at random positions (rarely in the same channel
    of q and k) the relative rounding of E4M3 leaves the rotation no error to
    remove: the measured score error stays within 1.5x either way."""
    q, k, _ = make_outlier_inputs(1, 1, 1, 1024, 128, seed=10)
    plain, rotated = _score_error(q, k, None), _score_error(q, k, hadamard_signs(128, seed=11))
    assert 1 / 1.5 < plain / rotated < 1.5, (plain, rotated)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk", [
    (1, 2, 2, 130, 130),     # a ragged second 128-row block on both sides
    (2, 4, 1, 200, 333),     # MQA, Nq < Nk: bottom-right causal alignment
    (1, 6, 3, 257, 300),     # GQA, three Q blocks
])
def test_attention_fp8_rows_equals_attention_fp8(B, Hq, Hkv, Nq, Nk, causal):
    """The per-row variant (which checks the full-size long-context launch)
    gives, row for row, what attention_fp8 gives over the whole matrices: the
    same dequantization and block descales (row i uses block i // 128), the
    same causal cut (keys j <= i + Nk - Nq), the same GQA head, the same
    bound.  An off-by-one in any of these fails here."""
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, 128, seed=77 + Nq)
    s = hadamard_signs(128, seed=78)
    q8, qd = fp8.quantize(q, signs=s)
    k8, kd = fp8.quantize(k, signs=s)
    vt8, vd = fp8.quantize(v, transpose=True)
    # distinct descales per block, so a wrong block index shows
    qd = qd * (1.0 + np.arange(qd.size, dtype=np.float32).reshape(qd.shape) / 16)
    kd = kd * (1.0 + np.arange(kd.size, dtype=np.float32).reshape(kd.shape) / 32)
    scale = 0.5 / 128
    o, lse, bound = fp8.attention_fp8(q8, k8, vt8, qd, kd, vd, Nk, causal=causal, scale=scale)
    rows = np.array([(b, h, i) for b in range(B) for h in range(Hq) for i in range(Nq)])
    ro, rl, rb = fp8.attention_fp8_rows(q8, k8, vt8, qd, kd, vd, Nk, rows, causal=causal,
                                        scale=scale)
    assert np.abs(ro - o.reshape(-1, 128)).max() <= 1e-12
    assert np.abs(rl - lse.reshape(-1)).max() <= 1e-12
    assert np.abs(rb - bound.reshape(-1, 128)).max() <= 1e-12


def test_attention_fp8_bound_covers_rounded_probabilities():
    """The bound attention_fp8 returns covers the error of O when the
    probabilities are rounded to E4M3 before the P.V product, as the kernel
    does: P~ = 2^(s*c - m + 4) in the frame of a running max m, rounded,
    with the row sum of the unrounded P~ as the normaliser.  Emulated here in
    fp64 with the oracle's E4M3 rounding on rows of mixed sharpness; the
    bound must hold and must not be loose by orders of magnitude."""
    rng = np.random.default_rng(11)
    Nq, Nk, d = 64, 512, 128
    q8 = fp8.e4m3_encode(rng.standard_normal((1, 1, Nq, d)) * 4)
    k8 = fp8.e4m3_encode(rng.standard_normal((1, 1, Nk, d)) * 4)
    v = rng.standard_normal((1, 1, Nk, d))
    vt8, vd = fp8.quantize(torch.from_numpy(v).to(torch.bfloat16), transpose=True)
    ones = lambda n: np.ones((1, 1, n), np.float32)  # noqa: E731
    for scale in (0.002, 0.01, 0.05):
        o, _, bound = fp8.attention_fp8(q8, k8, vt8, ones(1), ones(4), vd, Nk, causal=False,
                                        scale=scale)
        qv = fp8.e4m3_decode(q8)[0, 0]
        kv = fp8.e4m3_decode(k8)[0, 0]
        vv = fp8.dequantize(vt8, vd, Nk, transposed=True)[0, 0]
        s = scale * qv @ kv.T / math.log(2)                   # base-2 scores
        m = s.max(axis=1, keepdims=True)
        pt = np.exp2(s - m + 4)                               # frame with the factor 2^4
        o_emul = (fp8.e4m3_round(pt) @ vv) / pt.sum(axis=1, keepdims=True)
        err = np.abs(o_emul - o[0, 0])
        assert (err <= bound[0, 0]).all(), scale
        assert err.max() > 1e-3 * bound[0, 0].max(), scale   # the case has real error
