"""FP8 (E4M3) forward oracle -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module; the product path never does and shares
no code with it.

What the FP8 forward computes (lecture notes "Optimizing Attention for Modern
Hardware: FlashAttention 1-4", 4.4 FP8 and incoherent processing; "Flash
Attention 3/4 notes", FA3 section 2, block quantization and incoherent
processing):

- Block quantization: every block of 128 consecutive rows of one (batch, head)
  (a query tile of Q, a key tile of K or V) across all d columns gets its own
  scale, instead of one scale per tensor.
- Incoherent processing: Q and K are both multiplied by the same random
  orthogonal-up-to-scale matrix J = diag(s) H (s random signs, H the Hadamard
  matrix), so (QJ)(KJ)^T is QK^T times d and the scores do not change once
  the softmax scale is divided by d; every rotated channel is a +-1 mix of all
  input channels, which spreads outlier channels out.  V is not rotated (no
  factor on the output side would undo it).

Readings taken where the pages leave a step open:
1. E4M3 is the 8-bit float with 1 sign, 4 exponent bits (bias 7) and 3
   mantissa bits, no infinities, largest finite value 448, subnormals down to
   2^-9.  Conversions round to nearest, ties to even; magnitudes above 448
   saturate to 448.
2. A block's scale: amax = max |x| over the block (after the rotation);
   inv = 448 / amax and descale = amax / 448, both rounded to fp32; the code
   of x is e4m3(fp32(x * inv)).  An all-zero block has inv = 0, descale = 1.
   The dequantized value is code * descale.
3. The rotation is x -> H (s o x) with the unnormalised Sylvester-Hadamard H
   (entries +-1), computed in fp32 by the fast Walsh-Hadamard transform:
   stages h = 1, 2, 4, ..., d/2; in each, every pair (i, i + h) of a block of
   2h entries becomes (a + b, a - b).  Each add rounds to fp32, so the
   transform is a fixed sequence of roundings that any implementation taking
   the same pairs reproduces bit for bit.
4. V's codes are stored transposed, [B, H, d, Np] with the key count padded
   to Np = ceil(N / 16) * 16 (the padding holds zero codes).
5. The attention over the quantized operands is exact attention over the
   dequantized values (computed here in fp64).  The FP8 kernel additionally
   rounds the probabilities to E4M3 before the P.V product; that rounding is
   the kernel's, and attention_fp8 returns the bound the tests hold it to.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 128


def e4m3_round(x) -> np.ndarray:
    """Nearest E4M3 value (ties to even, saturating at +-448) of fp32 values,
    returned as float64 (exact)."""
    x = np.asarray(x, np.float32).astype(np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN has no E4M3 rounding here")
    sign = np.where(np.signbit(x), -1.0, 1.0)
    a = np.minimum(np.abs(x), E4M3_MAX)
    _, e = np.frexp(a)                 # a = f * 2^e with f in [0.5, 1)
    e = np.clip(e - 1, -6, 8)          # binade 2^e (subnormals share the 2^-6 spacing)
    step = np.ldexp(1.0, e - 3)        # 3 mantissa bits: spacing 2^(e-3)
    q = np.round(a / step) * step      # np.round rounds halves to even
    q = np.minimum(q, E4M3_MAX)
    return sign * q


def e4m3_encode(x) -> np.ndarray:
    """Codes (uint8) of the E4M3 rounding of fp32 values."""
    v = e4m3_round(x)
    neg = np.signbit(v)
    a = np.abs(v)
    code = np.zeros(a.shape, np.int64)
    sub = a < 2.0 ** -6
    code = np.where(sub, np.round(a / 2.0 ** -9).astype(np.int64), code)
    _, e = np.frexp(np.where(sub, 1.0, a))
    E = e - 1 + 7                      # biased exponent of a normal value
    M = np.round((np.where(sub, 1.0, a) / np.ldexp(1.0, e - 1) - 1.0) * 8).astype(np.int64)
    code = np.where(sub, code, (E << 3) | M)
    return (code | (neg.astype(np.int64) << 7)).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    """float64 values of E4M3 codes (0x7F / 0xFF, the NaN codes, decode to NaN)."""
    c = np.asarray(codes, np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    M = c & 0x7
    val = np.where(E == 0, M * 2.0 ** -9, (1.0 + M / 8.0) * np.ldexp(1.0, E - 7))
    val = np.where((E == 15) & (M == 7), np.nan, val)
    return s * val


def fwht_f32(x) -> np.ndarray:
    """Unnormalised fast Walsh-Hadamard transform along the last axis, in fp32,
    stages h = 1, 2, ..., d/2 with pairs (i, i + h) -> (a + b, a - b)."""
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    if d & (d - 1):
        raise ValueError("d must be a power of two")
    lead = y.shape[:-1]
    h = 1
    while h < d:
        y = y.reshape(lead + (d // (2 * h), 2, h))
        a = y[..., 0, :].copy()
        b = y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        y = y.reshape(lead + (d,))
        h *= 2
    return y


def _as_f32(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().float().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, np.float32)


def quantize(x, signs=None, transpose: bool = False):
    """Block-quantize x [B, H, N, d] (bf16 tensor or fp32 array) to E4M3.

    signs: None, or d values +-1: rotate each row by H (s o row) first.
    Returns (codes uint8 [B, H, N, d], or [B, H, d, Np] when transpose,
    descale float32 [B, H, ceil(N / 128)])."""
    xf = _as_f32(x)
    B, H, N, d = xf.shape
    if signs is not None:
        s = np.asarray(signs, np.float32).reshape(d)
        xf = fwht_f32(xf * s)          # sign flips are exact
    nblk = -(-N // BLOCK)
    descale = np.empty((B, H, nblk), np.float32)
    codes = np.zeros((B, H, N, d), np.uint8)
    for blk in range(nblk):
        rows = slice(blk * BLOCK, min(N, (blk + 1) * BLOCK))
        xb = xf[:, :, rows, :]
        amax = np.abs(xb).max(axis=(2, 3)).astype(np.float32)
        zero = amax == 0
        safe = np.where(zero, np.float32(1), amax).astype(np.float32)
        inv = np.where(zero, np.float32(0), np.float32(E4M3_MAX) / safe).astype(np.float32)
        descale[:, :, blk] = np.where(zero, np.float32(1),
                                      safe / np.float32(E4M3_MAX)).astype(np.float32)
        prod = (xb * inv[:, :, None, None]).astype(np.float32)
        codes[:, :, rows, :] = e4m3_encode(prod)
    if transpose:
        npad = -(-N // 16) * 16
        t = np.zeros((B, H, d, npad), np.uint8)
        t[..., :N] = codes.transpose(0, 1, 3, 2)
        return t, descale
    return codes, descale


def dequantize(codes, descale, N: int, transposed: bool = False) -> np.ndarray:
    """float64 values [B, H, N, d] of block-quantized codes."""
    c = np.asarray(codes)
    if transposed:
        c = c[..., :N].transpose(0, 1, 3, 2)
    v = e4m3_decode(c)
    rows = np.arange(N) // BLOCK
    return v * np.asarray(descale, np.float64)[:, :, rows][..., None]


def attention_dequantized(q, k, v, *, causal: bool, scale: float):
    """Exact attention in fp64 over float64 operands q [B,Hq,Nq,d], k/v
    [B,Hkv,Nk,d] (bottom-right causal, contiguous GQA groups).  Returns
    (O, LSE, P) with P the probabilities [B, Hq, Nq, Nk]."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    grp = Hq // Hkv
    kk = np.repeat(k, grp, axis=1)
    vv = np.repeat(v, grp, axis=1)
    s = scale * np.einsum("bhid,bhjd->bhij", q, kk)
    if causal:
        mask = np.arange(Nk)[None, :] > np.arange(Nq)[:, None] + (Nk - Nq)
        s = np.where(mask, -np.inf, s)
    mx = s.max(axis=-1, keepdims=True)
    e = np.exp(s - mx)
    tot = e.sum(axis=-1, keepdims=True)
    p = e / tot
    o = np.einsum("bhij,bhjd->bhid", p, vv)
    lse = (mx + np.log(tot))[..., 0]
    return o, lse, p


def attention_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, Nk: int, *, causal: bool,
                  scale: float):
    """Exact attention over the dequantized FP8 operands (q8, k8 [B, H, N, d]
    codes, vt8 [B, Hkv, d, Np] transposed codes).  Returns (O, LSE, bound).

    bound [B, Hq, Nq, d] allows for the kernel's E4M3 rounding of the
    probabilities: a normal E4M3 value is within 2^-4 (relative) of what it
    rounds, so the products change O by at most 2^-4 sum_j P_ij |V_jc| and the
    normaliser by as much again (2^-3 in all); probabilities below the
    smallest normal value (2^-10 of the row's largest, with the kernel's
    factor 2^4 above a maximum that lags the true one by at most 2^4) carry
    an absolute error of at most 2^-14 of the largest each, for which
    2^-8 max|V| is allowed in total (a statistical allowance: those errors
    have both signs)."""
    q8 = np.asarray(q8)
    Nq = q8.shape[2]
    q = dequantize(q8, q_descale, Nq)
    k = dequantize(k8, k_descale, Nk)
    v = dequantize(vt8, v_descale, Nk, transposed=True)
    o, lse, p = attention_dequantized(q, k, v, causal=causal, scale=scale)
    grp = q.shape[1] // k.shape[1]
    va = np.abs(np.repeat(v, grp, axis=1))
    bound = 2.0 ** -3 * np.einsum("bhij,bhjd->bhid", p, va) + \
        2.0 ** -8 * va.max(axis=(2, 3), keepdims=True)
    return o, lse, bound


def attention_fp8_rows(q8, k8, vt8, q_descale, k_descale, v_descale, Nk: int, rows, *,
                       causal: bool, scale: float):
    """Selected rows (b, hq, i) of attention_fp8, for shapes whose full score
    matrix is too large.  Returns (O [n, d], LSE [n], bound [n, d])."""
    q8, k8, vt8 = np.asarray(q8), np.asarray(k8), np.asarray(vt8)
    Nq = q8.shape[2]
    grp = q8.shape[1] // k8.shape[1]
    rows = np.asarray(rows).reshape(-1, 3)
    heads = {}
    out_o, out_l, out_b = [], [], []
    for b, h, i in rows:
        hk = h // grp
        if (b, hk) not in heads:
            kk = dequantize(k8[b:b + 1, hk:hk + 1], np.asarray(k_descale)[b:b + 1, hk:hk + 1], Nk)
            vv = dequantize(vt8[b:b + 1, hk:hk + 1], np.asarray(v_descale)[b:b + 1, hk:hk + 1], Nk,
                            transposed=True)
            heads[(b, hk)] = (kk[0, 0], vv[0, 0])
        kk, vv = heads[(b, hk)]
        blk = i // BLOCK
        qrow = e4m3_decode(q8[b, h, i]) * float(np.asarray(q_descale)[b, h, blk])
        n_allowed = min(Nk, i + 1 + (Nk - Nq)) if causal else Nk
        s = scale * (kk[:n_allowed] @ qrow)
        mx = s.max()
        e = np.exp(s - mx)
        p = e / e.sum()
        out_o.append(p @ vv[:n_allowed])
        out_l.append(mx + np.log(e.sum()))
        va = np.abs(vv[:n_allowed])
        out_b.append(2.0 ** -3 * (p @ va) + 2.0 ** -8 * np.abs(vv).max())
    return np.array(out_o), np.array(out_l), np.array(out_b)
