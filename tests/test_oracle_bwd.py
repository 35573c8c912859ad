"""Pins of the fp64 backward oracle (CPU).

The oracle's backward follows the lecture notes' section 2.6 formulas.  These
tests check it against things other than those formulas:
- torch autograd in float64 differentiating the plain forward definition
  O = softmax(scale * Q K^T, masked) V (a library routine, not a retyped
  backward);
- a central finite difference of L = sum(O * dO) along a random direction;
- invariants of the softmax Jacobian: every row's dS sums to zero, so the
  keys' dK sum to zero, and every row's P sums to one, so the keys' dV sum to
  the sum of dO over the rows;
- scale = 0 (uniform attention): dQ = dK = 0 and dV_j = sum over the rows
  that see key j of dO_i / (number of keys row i sees);
- GQA equals the sum over the group of the expanded (MHA) heads.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_14_gb300.inputs import make_fwd_inputs

pytestmark = pytest.mark.filterwarnings("ignore")


def _dout(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _autograd(q, k, v, do, causal, scale):
    """torch float64 autograd of the forward definition (heads expanded for GQA)."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    grp = Hq // Hkv
    qd = q.double().requires_grad_(True)
    kd = k.double().requires_grad_(True)
    vd = v.double().requires_grad_(True)
    ke = kd.repeat_interleave(grp, dim=1)
    ve = vd.repeat_interleave(grp, dim=1)
    s = scale * qd @ ke.transpose(-1, -2)
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        s = s.masked_fill(j > i + (Nk - Nq), float("-inf"))
    o = torch.softmax(s, dim=-1) @ ve
    o.backward(do.double())
    return qd.grad.numpy(), kd.grad.numpy(), vd.grad.numpy()


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 2, 2, 37, 37, 16, False),
    (2, 4, 2, 50, 50, 32, True),     # GQA, causal
    (1, 3, 1, 20, 45, 16, True),     # MQA, bottom-right causal with Nq < Nk
    (1, 2, 2, 60, 24, 8, False),     # Nq > Nk
    (1, 2, 1, 129, 129, 64, True),
])
def test_oracle_bwd_matches_autograd(B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=Nq + Nk + d)
    do = _dout(q.shape, seed=Nq)
    scale = 1.0 / np.sqrt(d)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale)
    rq, rk, rv = _autograd(q, k, v, do, causal, scale)
    for got, ref, name in ((dq, rq, "dQ"), (dk, rk, "dK"), (dv, rv, "dV")):
        assert np.abs(got - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max()), name


def _loss_np(qf, kf, vf, dof, causal, scale):
    """L = sum(O * dO) with O from the forward definition, numpy float64, one head."""
    s = scale * qf @ kf.T
    if causal:
        Nq, Nk = s.shape
        mask = np.arange(Nk)[None, :] > np.arange(Nq)[:, None] + (Nk - Nq)
        s = np.where(mask, -np.inf, s)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return float(np.sum((p @ vf) * dof))


@pytest.mark.parametrize("causal", [False, True])
def test_oracle_bwd_matches_finite_differences(causal):
    q, k, v = make_fwd_inputs(1, 1, 1, 12, 12, 8, seed=5)
    do = _dout(q.shape, seed=6)
    scale = 0.4
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=causal, scale=scale)
    qf, kf, vf, dof = (t[0, 0].double().numpy() for t in (q, k, v, do))
    rng = np.random.default_rng(7)
    eps = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        r = rng.standard_normal(qf.shape)
        args = [qf, kf, vf]
        plus = [a.copy() for a in args]
        minus = [a.copy() for a in args]
        plus[which] += eps * r
        minus[which] -= eps * r
        fd = (_loss_np(*plus, dof, causal, scale) - _loss_np(*minus, dof, causal, scale)) / (2 * eps)
        an = float(np.sum(grad[0, 0] * r))
        assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), (which, fd, an)


@pytest.mark.parametrize("causal", [False, True])
def test_oracle_bwd_invariants(causal):
    q, k, v = make_fwd_inputs(2, 4, 2, 70, 70, 32, seed=11)
    do = _dout(q.shape, seed=12)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=causal)
    # sum over keys of dK is zero (each row's dS sums to zero)
    assert np.abs(dk.sum(axis=2)).max() <= 1e-12 * np.abs(dk).max() * dk.shape[2]
    # sum over keys of dV equals the sum of dO over the group's rows
    grp = q.shape[1] // k.shape[1]
    do_sum = do.double().numpy().reshape(2, 2, grp, 70, 32).sum(axis=(2, 3))
    assert np.allclose(dv.sum(axis=2), do_sum, atol=1e-10)


def test_oracle_bwd_scale_zero_closed_form():
    B, Hq, Hkv, N, d = 1, 2, 1, 40, 16
    q, k, v = make_fwd_inputs(B, Hq, Hkv, N, N, d, seed=13)
    do = _dout(q.shape, seed=14)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=True, scale=0.0)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0
    dof = do.double().numpy()
    ref = np.zeros((N, d))
    for h in range(Hq):
        for i in range(N):
            ref[: i + 1] += dof[0, h, i] / (i + 1)   # row i sees keys 0..i uniformly
    assert np.allclose(dv[0, 0], ref, atol=1e-12)


def test_oracle_bwd_gqa_is_the_sum_of_expanded_heads():
    q, k, v = make_fwd_inputs(1, 6, 2, 33, 33, 16, seed=15)
    do = _dout(q.shape, seed=16)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal=True)
    ke, ve = k.repeat_interleave(3, dim=1), v.repeat_interleave(3, dim=1)
    dq2, dk2, dv2 = oracle.attention_bwd(q, ke, ve, do, causal=True)
    assert np.allclose(dq, dq2, atol=1e-13)
    assert np.allclose(dk, dk2.reshape(1, 2, 3, 33, 16).sum(axis=2), atol=1e-12)
    assert np.allclose(dv, dv2.reshape(1, 2, 3, 33, 16).sum(axis=2), atol=1e-12)
