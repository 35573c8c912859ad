"""GPU parity of attn_bwd against the fp64 oracle, through the C ABI.

The kernel's inputs O and LSE come from the oracle (rounded to fp32), so the
comparison isolates the backward's own arithmetic; one test chains attn_fwd
into attn_bwd.

Tolerance, from the arithmetic: scores and every product accumulate in fp32,
while P and dS are rounded to bf16 (relative error <= 2^-9 each) before the
P.dO, dS.Q and dS.K products.  Those rounding errors are independent across
the summed terms, so each gradient's relative L2 error is a small multiple of
2^-9 ~ 2e-3; the bound is relL2 <= 1e-2 per gradient, and max |error| <=
2e-2 * max |reference| per gradient (fp32 gradients compared; bf16 gradients
add half a bf16 ulp of each reference value).
"""
import math

import numpy as np
import pytest
import torch

import exact_attention_14_gb300 as ea
import oracle
from exact_attention_14_gb300.inputs import make_fwd_inputs

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_REL_TO_PEAK = 2e-2


def _dout(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _errors(got, ref):
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    peak = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
    return rel, peak


def _check(got, ref, what, bf16=False):
    assert np.isfinite(got).all(), f"{what}: non-finite"
    rel, peak = _errors(got, ref)
    if bf16:
        r = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(r), 1e-30))) - 8)
        err = np.abs(got - r)
        assert (err <= MAX_REL_TO_PEAK * np.abs(ref).max() + half_ulp).all(), f"{what}: bf16 bound"
    else:
        assert peak <= MAX_REL_TO_PEAK, f"{what}: max|err|/max|ref| = {peak:.3e}"
    assert rel <= REL_L2, f"{what}: relL2 = {rel:.3e}"


def _run(q, k, v, do, causal, scale, grad_dtype=torch.float32, o=None, lse=None):
    if o is None:
        o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=scale)
        o = torch.from_numpy(o_ref).float()
        lse = torch.from_numpy(lse_ref).float()
    dq, dk, dv = ea.backward(q.cuda(), k.cuda(), v.cuda(), o.cuda(), do.cuda(), lse.cuda(),
                             causal=causal, scale=scale, grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    return tuple(t.float().cpu().double().numpy() for t in (dq, dk, dv))


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 1, 1, 128, 128, 64, False),
    (1, 2, 2, 256, 256, 128, False),
    (1, 2, 2, 384, 384, 128, True),
    (2, 4, 2, 300, 300, 64, True),       # GQA, ragged tails
    (1, 4, 1, 200, 200, 128, False),     # MQA
    (1, 2, 2, 100, 333, 128, True),      # bottom-right causal, Nq < Nk
    (1, 2, 2, 700, 90, 64, False),       # Nq > Nk
    (2, 8, 2, 1000, 1000, 128, True),
])
def test_bwd_parity(B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=300 + Nq + Nk + d)
    do = _dout(q.shape, seed=Nq + 1)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = _run(q, k, v, do, causal, scale)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale)
    what = f"{(B, Hq, Hkv, Nq, Nk, d, causal)}"
    _check(dq, rq, "dQ " + what)
    _check(dk, rk, "dK " + what)
    _check(dv, rv, "dV " + what)


def test_bwd_bf16_gradients():
    q, k, v = make_fwd_inputs(1, 4, 2, 333, 333, 128, seed=77)
    do = _dout(q.shape, seed=78)
    dq, dk, dv = _run(q, k, v, do, True, 1 / math.sqrt(128), grad_dtype=torch.bfloat16)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=True)
    for got, ref, n in ((dq, rq, "dQ"), (dk, rk, "dK"), (dv, rv, "dV")):
        _check(got, ref, n, bf16=True)


def test_bwd_prefill_heads_sampled():
    """The prefill workload's shape (B4 H16 N2048 d128) at full size; the oracle
    checks two whole heads (MHA heads are independent)."""
    B, H, N, d = 4, 16, 2048, 128
    q, k, v = make_fwd_inputs(B, H, H, N, N, d, seed=1)
    do = _dout(q.shape, seed=2)
    for causal in (False, True):
        dq, dk, dv = _run(q, k, v, do, causal, 1 / math.sqrt(d))
        for (b, h) in ((0, 0), (3, 15)):
            sl = (slice(b, b + 1), slice(h, h + 1))
            rq, rk, rv = oracle.attention_bwd(q[sl], k[sl], v[sl], do[sl], causal=causal)
            _check(dq[sl], rq, f"dQ head {(b, h)} causal={causal}")
            _check(dk[sl], rk, f"dK head {(b, h)} causal={causal}")
            _check(dv[sl], rv, f"dV head {(b, h)} causal={causal}")


def test_fwd_then_bwd_end_to_end():
    """attn_fwd's own O (bf16) and LSE feed attn_bwd."""
    q, k, v = make_fwd_inputs(2, 4, 4, 512, 512, 128, seed=91)
    do = _dout(q.shape, seed=92)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = ea.forward(qd, kd, vd, causal=True, out_dtype=torch.bfloat16)
    dq, dk, dv = _run(q, k, v, do, True, 1 / math.sqrt(128), o=o.cpu(), lse=lse.cpu())
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=True)
    _check(dq, rq, "dQ")
    _check(dk, rk, "dK")
    _check(dv, rv, "dV")


def test_bwd_repeatable():
    """Every gradient is accumulated on chip in a fixed order (no atomics):
    bit-identical runs."""
    q, k, v = make_fwd_inputs(1, 4, 2, 640, 640, 128, seed=93)
    do = _dout(q.shape, seed=94)
    a = _run(q, k, v, do, True, 1 / math.sqrt(128))
    b = _run(q, k, v, do, True, 1 / math.sqrt(128))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("d,causal", [(48, True), (96, False), (96, True)])
def test_bwd_head_dims_padded(d, causal):
    q, k, v = make_fwd_inputs(2, 4, 2, 300, 300, d, seed=700 + d)
    do = _dout(q.shape, seed=701)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = _run(q, k, v, do, causal, scale)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale)
    _check(dq, rq, f"dQ d={d}")
    _check(dk, rk, f"dK d={d}")
    _check(dv, rv, f"dV d={d}")


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 2, 2, 128, 128, 256, False),
    (1, 2, 1, 300, 300, 256, True),      # MQA, ragged 64-row Q tiles and 64-key tiles
    (2, 4, 2, 200, 200, 192, False),     # the 256-column kernels with zero columns past d
    (1, 2, 2, 100, 333, 136, True),      # bottom-right causal, Nq < Nk
    (1, 2, 2, 450, 130, 256, False),     # Nq > Nk, a ragged key tile
    (1, 8, 2, 700, 700, 256, True),      # GQA group of 4, several key tiles per CTA half
])
def test_bwd_wide_head_dims(B, Hq, Hkv, Nq, Nk, d, causal):
    """Head dims above 128 (the 256-column kernels: the dK/dV pass per column
    half of d over 64-row Q tiles, the dQ pass over 64-key tiles)."""
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=1400 + Nq + Nk + d)
    do = _dout(q.shape, seed=1401 + d)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = _run(q, k, v, do, causal, scale)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale)
    what = f"{(B, Hq, Hkv, Nq, Nk, d, causal)}"
    _check(dq, rq, "dQ " + what)
    _check(dk, rk, "dK " + what)
    _check(dv, rv, "dV " + what)


def test_bwd_wide_chained_bf16_and_repeatable():
    """d = 256: attn_fwd's own O and LSE into attn_bwd with bf16 gradients,
    twice, bit-identical."""
    q, k, v = make_fwd_inputs(1, 4, 2, 512, 512, 256, seed=1500)
    do = _dout(q.shape, seed=1501)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, out_dtype=torch.bfloat16)
    a = _run(q, k, v, do, True, 1 / 16, grad_dtype=torch.bfloat16, o=o.cpu(), lse=lse.cpu())
    b = _run(q, k, v, do, True, 1 / 16, grad_dtype=torch.bfloat16, o=o.cpu(), lse=lse.cpu())
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=True, scale=1 / 16)
    for got, ref, n in zip(a, (rq, rk, rv), ("dQ", "dK", "dV")):
        _check(got, ref, n, bf16=True)


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [
    (2, 16, 16, 1024, 128, False),
    (2, 16, 16, 1024, 128, True),
    (2, 32, 8, 2048, 64, True),   # GQA: four query heads per dK/dV item
])
def test_bwd_persistent_many_items(B, Hq, Hkv, N, d, causal):
    """More dK/dV and dQ items than SMs, so each persistent CTA runs several
    items back to back (rings, barrier phases and TMEM accumulators carried
    from one item into the next); every head against the oracle."""
    q, k, v = make_fwd_inputs(B, Hq, Hkv, N, N, d, seed=950 + N + d)
    do = _dout(q.shape, seed=951)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = _run(q, k, v, do, causal, scale)
    rq, rk, rv = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale)
    what = f"{(B, Hq, Hkv, N, d, causal)}"
    _check(dq, rq, "dQ " + what)
    _check(dk, rk, "dK " + what)
    _check(dv, rv, "dV " + what)
