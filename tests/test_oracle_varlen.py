"""Pins of the packed variable-length oracle (CPU).

A packed batch is a set of independent attention problems laid end to end.
The oracle is pinned by (1) a numpy softmax written per sequence on a tiny
batch, (2) the dense oracle on the same sequences stored [B, H, N, d] when all
lengths are equal, (3) independence: the rows of one sequence do not change
when another sequence's values (NaN included) change, and (4) a zero-length
sequence between two others changes nothing.
"""
import numpy as np
import torch

import oracle
from exact_attention_14_gb300.inputs import make_varlen_inputs


def _numpy_reference(q, k, v, cu_q, cu_k, causal, scale):
    qf, kf, vf = (t.double().numpy() for t in (q, k, v))
    Hq, Hkv = q.shape[1], k.shape[1]
    grp = Hq // Hkv
    o = np.full(qf.shape, np.nan)
    lse = np.full((Hq, qf.shape[0]), np.nan)
    for b in range(len(cu_q) - 1):
        qs, qe, ks, ke = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        nq, nk = qe - qs, ke - ks
        for h in range(Hq):
            s = scale * qf[qs:qe, h] @ kf[ks:ke, h // grp].T
            if causal:
                mask = np.arange(nk)[None, :] > np.arange(nq)[:, None] + (nk - nq)
                s = np.where(mask, -np.inf, s)
            mx = s.max(axis=1, keepdims=True)
            e = np.exp(s - mx)
            o[qs:qe, h] = (e / e.sum(axis=1, keepdims=True)) @ vf[ks:ke, h // grp]
            lse[h, qs:qe] = mx[:, 0] + np.log(e.sum(axis=1))
    return o, lse


def test_varlen_oracle_matches_numpy_per_sequence():
    for causal in (False, True):
        lq, lk = [5, 17, 1, 9], [7, 17, 3, 12]
        q, k, v, cu_q, cu_k = make_varlen_inputs(lq, lk, 4, 2, 16, seed=21)
        o, lse = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=causal, scale=0.3)
        ro, rl = _numpy_reference(q, k, v, cu_q, cu_k, causal, 0.3)
        assert np.abs(o - ro).max() < 1e-12
        assert np.abs(lse - rl).max() < 1e-12


def test_varlen_oracle_equal_lengths_is_the_dense_oracle():
    B, H, N, d = 3, 2, 40, 32
    q, k, v, cu_q, cu_k = make_varlen_inputs([N] * B, [N] * B, H, H, d, seed=22)
    o, lse = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=True)
    qd = q.reshape(B, N, H, d).permute(0, 2, 1, 3)
    kd = k.reshape(B, N, H, d).permute(0, 2, 1, 3)
    vd = v.reshape(B, N, H, d).permute(0, 2, 1, 3)
    od, ld = oracle.attention(qd, kd, vd, causal=True)
    assert np.array_equal(o, od.transpose(0, 2, 1, 3).reshape(B * N, H, d))
    assert np.array_equal(lse, ld.transpose(1, 0, 2).reshape(H, B * N))


def test_varlen_oracle_sequences_are_independent():
    lq = [30, 20, 25]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lq, lq, 2, 1, 16, seed=23, extra_rows=5)
    o1, l1 = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=False)
    k2, v2 = k.clone(), v.clone()
    k2[30:50] = float("nan")
    v2[30:50] = float("inf")
    o2, l2 = oracle.attention_varlen(q, k2, v2, cu_q, cu_k, causal=False)
    for rows in (slice(0, 30), slice(50, 75)):
        assert np.array_equal(o1[rows], o2[rows])
        assert np.array_equal(l1[:, rows], l2[:, rows])
    assert np.isnan(o1[75:]).all()          # rows past the last sequence: no result
    assert np.isfinite(o1[:75]).all()


def test_varlen_oracle_empty_sequence_changes_nothing():
    q, k, v, cu_q, cu_k = make_varlen_inputs([12, 0, 8], [12, 0, 8], 2, 2, 8, seed=24)
    o, lse = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=True)
    cu2 = torch.tensor([0, 12, 20], dtype=torch.int32)
    o2, l2 = oracle.attention_varlen(q, k, v, cu2, cu2, causal=True)
    assert np.array_equal(o, o2) and np.array_equal(lse, l2)


# ---------------------------------------------------------------- backward --
def _autograd_reference(q, k, v, do, cu_q, cu_k, causal, scale):
    """float64 autograd of a plain softmax attention, sequence by sequence."""
    Hq, Hkv = q.shape[1], k.shape[1]
    grp = Hq // Hkv
    qf, kf, vf = (t.double().clone().requires_grad_(True) for t in (q, k, v))
    dof = do.double()
    for b in range(len(cu_q) - 1):
        qs, qe, ks, ke = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        nq, nk = qe - qs, ke - ks
        if nq == 0:
            continue
        for h in range(Hq):
            s = scale * qf[qs:qe, h] @ kf[ks:ke, h // grp].T
            if causal:
                mask = torch.arange(nk)[None, :] > torch.arange(nq)[:, None] + (nk - nq)
                s = s.masked_fill(mask, float("-inf"))
            o = torch.softmax(s, dim=1) @ vf[ks:ke, h // grp]
            (o * dof[qs:qe, h]).sum().backward()
    return tuple(t.grad.numpy() for t in (qf, kf, vf))


def test_varlen_bwd_oracle_matches_autograd_per_sequence():
    """The packed backward oracle against float64 autograd of plain softmax
    attention, GQA, causal (bottom-right) and not, with a sequence without
    queries between two others (its keys get zero gradients)."""
    for causal in (False, True):
        lq, lk = [5, 0, 9, 1], [7, 4, 12, 3]
        q, k, v, cu_q, cu_k = make_varlen_inputs(lq, lk, 4, 2, 16, seed=61)
        g = torch.Generator().manual_seed(62)
        do = torch.randn(q.shape, generator=g).to(torch.bfloat16)
        gq, gk, gv = oracle.attention_bwd_varlen(q, k, v, do, cu_q, cu_k, causal=causal, scale=0.3)
        rq, rk, rv = _autograd_reference(q, k, v, do, cu_q, cu_k, causal, 0.3)
        np.testing.assert_allclose(gq, rq, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(gk, rk, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(gv, rv, rtol=1e-10, atol=1e-12)
        assert (gk[7:11] == 0).all() and (gv[7:11] == 0).all()   # the keys of sequence 1


def test_varlen_bwd_oracle_equal_lengths_is_the_dense_oracle():
    B, H, N, d = 3, 2, 20, 8
    q, k, v, cu_q, cu_k = make_varlen_inputs([N] * B, [N] * B, H, H, d, seed=63)
    do = torch.randn(q.shape, generator=torch.Generator().manual_seed(64)).to(torch.bfloat16)
    gq, gk, gv = oracle.attention_bwd_varlen(q, k, v, do, cu_q, cu_k, causal=True)
    dense = lambda t: t.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous()  # noqa: E731
    rq, rk, rv = oracle.attention_bwd(dense(q), dense(k), dense(v), dense(do), causal=True)
    back = lambda a: a.transpose(0, 2, 1, 3).reshape(B * N, H, d)  # noqa: E731
    assert np.array_equal(gq, back(rq)) and np.array_equal(gk, back(rk)) and np.array_equal(gv, back(rv))
