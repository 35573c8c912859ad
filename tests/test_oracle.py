"""Pins for the fp64 oracle: each test checks it against something other than
itself -- a library routine, a closed form, an invariant of the definition, or
brute force on tiny inputs -- so that a dropped term, a wrong sign or index, or
a transposed operand anywhere in it fails at least one test.

Definition pinned (lecture notes "Optimizing Attention for Modern Hardware:
FlashAttention 1-4", sections 0.4, 1.4, 2.2, 2.5, 6.1, exercise 3):
O = softmax(scale * Q K^T) V per row, LSE = log sum exp, causal keeps j <= i,
and partial results over disjoint key sets merge exactly by log-sum-exp.
"""
import itertools
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle
from exact_attention_14_gb300.inputs import make_fwd_inputs


def as_f64(t):
    return t.to(torch.float64).numpy()


def bf16(a):
    return torch.tensor(np.asarray(a, np.float64), dtype=torch.float64).to(torch.bfloat16)


def scipy_reference(q, k, v, causal, scale, kv_len=None):
    """Same quantity through numpy matmul + scipy's logsumexp/softmax."""
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    B, Hq, Nq, d = qd.shape
    Hkv, Nk = kd.shape[1], kd.shape[2]
    grp = Hq // Hkv
    O = np.zeros((B, Hq, Nq, d))
    L = np.zeros((B, Hq, Nq))
    for b in range(B):
        for h in range(Hq):
            S = scale * qd[b, h] @ kd[b, h // grp].T
            mask = np.ones((Nq, Nk), bool)
            if causal:
                mask &= np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
            if kv_len is not None:
                mask &= np.arange(Nk)[None, :] < kv_len[b]
            S = np.where(mask, S, -np.inf)
            L[b, h] = logsumexp(S, axis=1)
            O[b, h] = softmax(S, axis=1) @ vd[b, h // grp]
    return O, L


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 1, 1, 5, 5, 4, False),
    (2, 4, 2, 37, 37, 16, False),
    (2, 4, 2, 37, 37, 16, True),
    (1, 6, 3, 13, 29, 8, True),    # Nq < Nk, causal bottom-right
    (1, 8, 1, 20, 9, 32, False),   # MQA, Nq > Nk
    (3, 2, 2, 1, 17, 64, False),
])
def test_matches_scipy_logsumexp_softmax(B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=11 + Nq)
    scale = 1.0 / math.sqrt(d)
    o, lse = oracle.attention(q, k, v, causal=causal, scale=scale)
    O, L = scipy_reference(q, k, v, causal, scale)
    np.testing.assert_allclose(lse, L, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, O, rtol=0, atol=1e-12)


def test_brute_force_pure_python_tiny():
    """Element-by-element loops with math.exp / math.log on a tiny case."""
    B, Hq, Hkv, N, d = 1, 4, 2, 6, 3
    q, k, v = make_fwd_inputs(B, Hq, Hkv, N, N, d, seed=5)
    qd, kd, vd = as_f64(q), as_f64(k), as_f64(v)
    scale = 0.7
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal=causal, scale=scale)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            for i in range(N):
                keys = [j for j in range(N) if (not causal or j <= i)]
                s = {j: scale * sum(qd[0, h, i, c] * kd[0, g, j, c] for c in range(d))
                     for j in keys}
                denom = sum(math.exp(s[j]) for j in keys)
                assert abs(lse[0, h, i] - math.log(denom)) < 1e-12
                for c in range(d):
                    ref = sum(math.exp(s[j]) / denom * vd[0, g, j, c] for j in keys)
                    assert abs(o[0, h, i, c] - ref) < 1e-12


def test_identical_keys_give_mean_of_values():
    """All keys equal => uniform weights over the allowed keys:
    O_i = mean of allowed V rows, LSE_i = s + log(#allowed)."""
    N, d = 9, 8
    q, _, v = make_fwd_inputs(1, 1, 1, N, N, d, seed=3)
    krow = torch.randn(d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    k = krow.expand(1, 1, N, d).contiguous()
    scale = 0.5
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal=causal, scale=scale)
        vd, qd, kd = as_f64(v)[0, 0], as_f64(q)[0, 0], as_f64(krow)
        for i in range(N):
            n = i + 1 if causal else N
            np.testing.assert_allclose(o[0, 0, i], vd[:n].mean(0), atol=1e-13)
            s = scale * float(qd[i] @ kd)
            assert abs(lse[0, 0, i] - (s + math.log(n))) < 1e-12


def test_single_allowed_key():
    """One key (Nk = 1), or causal row 0: O = that V row, LSE = its score."""
    q, k, v = make_fwd_inputs(1, 2, 2, 1, 1, 16, seed=8)
    o, lse = oracle.attention(q, k, v, scale=0.3)
    for h in range(2):
        np.testing.assert_allclose(o[0, h, 0], as_f64(v)[0, h, 0], atol=0)
        s = 0.3 * float(as_f64(q)[0, h, 0] @ as_f64(k)[0, h, 0])
        assert abs(lse[0, h, 0] - s) < 1e-13
    q, k, v = make_fwd_inputs(1, 1, 1, 7, 7, 16, seed=9)
    o, lse = oracle.attention(q, k, v, causal=True)
    np.testing.assert_allclose(o[0, 0, 0], as_f64(v)[0, 0, 0], atol=0)


def test_large_gap_gives_one_hot():
    """A key whose score exceeds all others by ~50 takes all the weight."""
    d, N = 4, 10
    q = bf16(np.array([[[[1.0, 0, 0, 0]]]]))
    kk = np.zeros((1, 1, N, d))
    kk[0, 0, :, 1] = np.arange(N)          # orthogonal to q: score 0
    kk[0, 0, 6, 0] = 50.0                  # score 50 for key 6
    k = bf16(kk)
    v = make_fwd_inputs(1, 1, 1, 1, N, d, seed=2)[2]
    o, lse = oracle.attention(q, k, v, scale=1.0)
    np.testing.assert_allclose(o[0, 0, 0], as_f64(v)[0, 0, 6], atol=1e-19 + 20 * math.exp(-50))
    assert abs(lse[0, 0, 0] - (50 + math.log1p((N - 1) * math.exp(-50)))) < 1e-12


def test_zero_scale_is_uniform_average_with_causal_counts():
    """scale = 0: every allowed key weighs the same, so row i of a causal head
    averages exactly i + 1 + (Nk - Nq) value rows and LSE = log(count)."""
    Nq, Nk, d = 5, 11, 6
    q, k, v = make_fwd_inputs(1, 1, 1, Nq, Nk, d, seed=4)
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.0)
    vd = as_f64(v)[0, 0]
    for i in range(Nq):
        n = i + 1 + (Nk - Nq)
        np.testing.assert_allclose(o[0, 0, i], vd[:n].mean(0), atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-14


def test_probabilities_sum_to_one_via_identity_values():
    """With V = identity rows, O_i is the probability row P_i: it sums to 1 and
    P_ij = exp(s_ij - LSE_i)."""
    N = d = 16
    q, k, _ = make_fwd_inputs(1, 1, 1, N, N, d, seed=6)
    v = torch.eye(N, dtype=torch.float32).to(torch.bfloat16).reshape(1, 1, N, d)
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal=causal, scale=0.4)
        P = o[0, 0]
        np.testing.assert_allclose(P.sum(1), np.ones(N), atol=1e-14)
        S = 0.4 * as_f64(q)[0, 0] @ as_f64(k)[0, 0].T
        for i in range(N):
            for j in range(N):
                want = 0.0 if (causal and j > i) else math.exp(S[i, j] - lse[0, 0, i])
                assert abs(P[i, j] - want) < 1e-14


def test_key_permutation_invariance():
    """Non-causal attention does not depend on the order of (k_j, v_j) pairs."""
    q, k, v = make_fwd_inputs(2, 2, 2, 12, 23, 16, seed=12)
    perm = torch.randperm(23, generator=torch.Generator().manual_seed(3))
    o1, l1 = oracle.attention(q, k, v)
    o2, l2 = oracle.attention(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous())
    np.testing.assert_allclose(o1, o2, atol=1e-14)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_shift_invariance():
    """k_j -> k_j + u for every j adds scale*q_i.u to all of row i's scores:
    O is unchanged and LSE moves by exactly that amount.  Small integers keep
    every value exact in bf16."""
    rng = np.random.default_rng(0)
    Nq, Nk, d = 6, 10, 8
    qi = rng.integers(-3, 4, (1, 1, Nq, d)).astype(np.float64)
    ki = rng.integers(-3, 4, (1, 1, Nk, d)).astype(np.float64)
    ui = rng.integers(-2, 3, (d,)).astype(np.float64)
    v = make_fwd_inputs(1, 1, 1, Nq, Nk, d, seed=13)[2]
    scale = 0.125
    for causal in (False, True):
        o1, l1 = oracle.attention(bf16(qi), bf16(ki), v, causal=causal, scale=scale)
        o2, l2 = oracle.attention(bf16(qi), bf16(ki + ui), v, causal=causal, scale=scale)
        np.testing.assert_allclose(o1, o2, atol=1e-13)
        np.testing.assert_allclose(l2 - l1, scale * (qi[0, 0] @ ui)[None, None], atol=1e-12)


def test_gqa_equals_expanded_heads():
    """Hq = 4*Hkv is ordinary multi-head attention with each KV head repeated
    for a contiguous group of 4 query heads."""
    q, k, v = make_fwd_inputs(2, 8, 2, 15, 15, 16, seed=14)
    for causal in (False, True):
        o1, l1 = oracle.attention(q, k, v, causal=causal)
        kx = k.repeat_interleave(4, dim=1).contiguous()
        vx = v.repeat_interleave(4, dim=1).contiguous()
        o2, l2 = oracle.attention(q, kx, vx, causal=causal)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def test_causal_row_equals_truncated_noncausal():
    """Causal row i is non-causal attention over keys 0..i+(Nk-Nq) only."""
    Nq, Nk, d = 7, 12, 8
    q, k, v = make_fwd_inputs(1, 2, 2, Nq, Nk, d, seed=15)
    o, lse = oracle.attention(q, k, v, causal=True)
    for i in range(Nq):
        n = i + 1 + (Nk - Nq)
        o2, l2 = oracle.attention(q[:, :, i:i + 1].contiguous(), k[:, :, :n].contiguous(),
                                  v[:, :, :n].contiguous())
        np.testing.assert_allclose(o[:, :, i], o2[:, :, 0], atol=1e-14)
        np.testing.assert_allclose(lse[:, :, i], l2[:, :, 0], atol=1e-13)


def test_kv_len_equals_truncated_cache_and_ignores_tail():
    """Decode over the first L_b keys equals attention over a cache cut at
    L_b; NaN written past L_b never reaches the result."""
    B, Hq, Hkv, Nmax, d = 3, 4, 2, 20, 16
    q, k, v = make_fwd_inputs(B, Hq, Hkv, 1, Nmax, d, seed=16)
    lens = np.array([1, 13, 20], np.int32)
    o, lse = oracle.decode(q, k, v, lens)
    kn, vn = k.clone(), v.clone()
    for b in range(B):
        o2, l2 = oracle.attention(q[b:b + 1].contiguous(), k[b:b + 1, :, :lens[b]].contiguous(),
                                  v[b:b + 1, :, :lens[b]].contiguous())
        np.testing.assert_allclose(o[b], o2[0], atol=1e-14)
        np.testing.assert_allclose(lse[b], l2[0], atol=1e-13)
        kn[b, :, lens[b]:] = float("nan")
        vn[b, :, lens[b]:] = float("nan")
    o3, l3 = oracle.decode(q, kn, vn, lens)
    np.testing.assert_array_equal(o, o3)
    np.testing.assert_array_equal(lse, l3)


def test_lse_merge_of_key_splits_is_exact_in_any_order():
    """Split the keys at random points, attend to each part, merge the parts by
    log-sum-exp in random orders and as a tree: all equal the unsplit result
    (exercise 3: the merge is associative and commutative)."""
    rng = np.random.default_rng(7)
    Nk, d = 97, 32
    q, k, v = make_fwd_inputs(1, 2, 1, 3, Nk, d, seed=17)
    o_full, l_full = oracle.attention(q, k, v)
    rows = [(0, h, i) for h in range(2) for i in range(3)]
    for n_parts in (1, 2, 5, 17, 64):
        cuts = np.sort(rng.choice(np.arange(1, Nk), size=n_parts - 1, replace=False))
        bounds = list(zip([0, *cuts], [*cuts, Nk]))
        parts = [oracle.attention_rows(q, k, v, rows, window=(lo, hi)) for lo, hi in bounds]
        for r, (b, h, i) in enumerate(rows):
            lses = np.array([p[1][r] for p in parts])
            os_ = np.stack([p[0][r] for p in parts])
            order = rng.permutation(n_parts)
            lse, o = oracle.lse_merge(lses[order], os_[order])
            assert abs(lse - l_full[b, h, i]) < 1e-12
            np.testing.assert_allclose(o, o_full[b, h, i], atol=1e-13)
            # pairwise tree
            items = [(lses[s], os_[s]) for s in range(n_parts)]
            while len(items) > 1:
                nxt = []
                for a in range(0, len(items) - 1, 2):
                    l2, o2 = oracle.lse_merge([items[a][0], items[a + 1][0]],
                                              np.stack([items[a][1], items[a + 1][1]]))
                    nxt.append((l2, o2))
                if len(items) % 2:
                    nxt.append(items[-1])
                items = nxt
            assert abs(items[0][0] - l_full[b, h, i]) < 1e-12
            np.testing.assert_allclose(items[0][1], o_full[b, h, i], atol=1e-13)


def test_empty_key_set_reading():
    """No allowed key (an empty window): O = 0, LSE = -inf."""
    q, k, v = make_fwd_inputs(1, 1, 1, 2, 8, 4, seed=18)
    o, lse = oracle.attention_rows(q, k, v, [(0, 0, 0)], window=(5, 5))  # hi <= lo
    assert lse[0] == -np.inf
    np.testing.assert_array_equal(o[0], np.zeros(4))
    lm, om = oracle.lse_merge([-np.inf, -np.inf], np.zeros((2, 4)))
    assert lm == -np.inf


def test_rows_api_matches_full():
    q, k, v = make_fwd_inputs(2, 4, 2, 33, 40, 16, seed=19)
    o, lse = oracle.attention(q, k, v, causal=True)
    rows = [(b, h, i) for b, h, i in itertools.product(range(2), range(4), (0, 5, 32))]
    o2, l2 = oracle.attention_rows(q, k, v, rows, causal=True)
    for r, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(o2[r], o[b, h, i])
        assert l2[r] == lse[b, h, i]


def test_rejects_bad_rows():
    q, k, v = make_fwd_inputs(1, 1, 1, 4, 4, 4, seed=20)
    with pytest.raises(ValueError):
        oracle.attention_rows(q, k, v, [(0, 0, 4)])
