"""GPU parity of attn_fwd_varlen (packed variable-length batches) against the
fp64 oracle, through the C ABI.  Tolerances as attn_fwd: max |dO| <= 1e-2,
relative L2(O) <= 5e-3, max |dLSE| <= 1e-3 (fp32 output); bf16 output within
1e-2 plus half a bf16 ulp of the rounded reference."""
import math

import numpy as np
import pytest
import torch

import exact_attention_14_gb300 as ea
import oracle
from exact_attention_14_gb300.inputs import VARLEN, make_varlen_inputs, varlen_lengths

from test_gpu_fwd import assert_close, assert_close_bf16

pytestmark = pytest.mark.gpu


def gpu_varlen(q, k, v, cu_q, cu_k, causal, scale=None, out_dtype=torch.float32, o_init=None,
               expect_error=0):
    lq = (cu_q[1:] - cu_q[:-1]).tolist()
    lk = (cu_k[1:] - cu_k[:-1]).tolist()
    mq, mk = max(max(lq), 1), max(max(lk), 1)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = (torch.full(q.shape, float("nan"), dtype=out_dtype) if o_init is None else o_init).cuda()
    lse = torch.full((q.shape[1], q.shape[0]), float("nan"), dtype=torch.float32).cuda()
    ea.attn_fwd_varlen(qd, kd, vd, o, cu_q.cuda(), cu_k.cuda(), mq, mk, lse, causal=causal,
                       scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == expect_error
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def _rows(cu):
    """Rows that belong to a sequence."""
    return np.arange(int(cu[-1]))


LENS = [1, 127, 128, 129, 0, 255, 256, 257, 600, 33]


@pytest.mark.parametrize("d", [64, 128, 96])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_parity(d, causal):
    q, k, v, cu_q, cu_k = make_varlen_inputs(LENS, LENS, 8, 2, d, seed=800 + d)
    scale = 1 / math.sqrt(d)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, causal, scale)
    ro, rl = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=causal, scale=scale)
    r = _rows(cu_q)
    assert_close(o[r], lse[:, r], ro[r], rl[:, r], f"d={d} causal={causal}")


@pytest.mark.parametrize("d", [192, 256, 136])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_wide_head_dims(d, causal):
    """Head dims above 128 (the 192- and 256-column kernels, 128-key tiles):
    empty, single-row and ragged sequences, GQA, against the oracle."""
    q, k, v, cu_q, cu_k = make_varlen_inputs(LENS, LENS, 8, 2, d, seed=850 + d)
    scale = 1 / math.sqrt(d)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, causal, scale)
    ro, rl = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=causal, scale=scale)
    r = _rows(cu_q)
    assert_close(o[r], lse[:, r], ro[r], rl[:, r], f"d={d} causal={causal}")


def test_varlen_wide_cross_lengths_and_neighbours():
    """d = 256 with queries and keys of different lengths (bottom-right causal),
    NaN / inf in one sequence's keys, and rows past the last sequence that are
    never written."""
    lq = [100, 300, 1, 257]
    lk = [400, 300, 700, 260]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lq, lk, 4, 4, 256, seed=852, extra_rows=40)
    for causal in (False, True):
        o, lse = gpu_varlen(q, k, v, cu_q, cu_k, causal)
        ro, rl = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=causal)
        n = int(cu_q[-1])
        assert_close(o[:n], lse[:, :n], ro[:n], rl[:, :n], f"cross lengths causal={causal}")
        assert np.isnan(o[n:]).all() and np.isnan(lse[:, n:]).all()
    k2, v2 = k.clone(), v.clone()
    k2[400:700] = float("nan")
    v2[400:700] = float("inf")
    o1, l1 = gpu_varlen(q, k, v, cu_q, cu_k, False)
    o2, l2 = gpu_varlen(q, k2, v2, cu_q, cu_k, False)
    for rows in (slice(0, 100), slice(400, 658)):
        assert np.array_equal(o1[rows], o2[rows]) and np.array_equal(l1[:, rows], l2[:, rows])


def test_varlen_wide_equal_lengths_bit_identical_to_dense():
    """All sequences of one length at d = 256: the dense 256-column kernel's
    tiles and arithmetic in the packed layout."""
    B, H, N, d = 2, 4, 500, 256
    q, k, v, cu_q, cu_k = make_varlen_inputs([N] * B, [N] * B, H, H, d, seed=853)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, True)
    qd = q.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().cuda()
    kd = k.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().cuda()
    vd = v.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().cuda()
    od, ld = ea.forward(qd, kd, vd, causal=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    od = od.permute(0, 2, 1, 3).reshape(B * N, H, d).cpu().double().numpy()
    ld = ld.permute(1, 0, 2).reshape(H, B * N).cpu().double().numpy()
    assert np.array_equal(o, od) and np.array_equal(lse, ld)


def test_varlen_wide_bad_offsets_reported_and_skipped():
    """d = 192: a sequence longer than max_seqlen is not computed, the device
    error word reports it, the other sequences are exact."""
    lens = [64, 236, 64]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lens, lens, 2, 2, 192, seed=854)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full(q.shape, 7.0, dtype=torch.float32).cuda()
    ea.attn_fwd_varlen(qd, kd, vd, o, cu_q.cuda(), cu_k.cuda(), 200, 236, None, causal=False)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == ea.ATTN_ERR_INVALID_ARG
    o = o.cpu().double().numpy()
    assert (o[64:300] == 7.0).all()
    ro, rl = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=False)
    for rows in (slice(0, 64), slice(300, 364)):
        assert np.abs(o[rows] - ro[rows]).max() <= 1e-2


def test_varlen_keys_differ_from_queries():
    """Cross lengths: non-causal any Nq/Nk; causal needs Nq <= Nk (bottom-right)."""
    lq = [100, 300, 1, 512, 129]
    lk = [400, 300, 700, 513, 1000]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lq, lk, 4, 4, 128, seed=811)
    for causal in (False, True):
        o, lse = gpu_varlen(q, k, v, cu_q, cu_k, causal)
        ro, rl = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=causal)
        assert_close(o, lse, ro, rl, f"causal={causal}")
    lq2 = [300, 20, 50]
    lk2 = [10, 700, 1]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lq2, lk2, 4, 4, 64, seed=812)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, False)
    ro, rl = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=False)
    assert_close(o, lse, ro, rl, "Nq > Nk non-causal")


def test_varlen_bf16_output():
    q, k, v, cu_q, cu_k = make_varlen_inputs(LENS, LENS, 8, 8, 128, seed=813)
    o, _ = gpu_varlen(q, k, v, cu_q, cu_k, True, out_dtype=torch.bfloat16)
    ro, _ = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=True)
    assert_close_bf16(o, ro, "bf16 O")


def test_varlen_neighbours_never_leak():
    """NaN and inf in one sequence, and NaN in rows past the last sequence,
    leave every other sequence's result bit-identical; rows outside every
    sequence are never written."""
    lens = [200, 130, 70]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lens, lens, 4, 2, 128, seed=814, extra_rows=90)
    o1, l1 = gpu_varlen(q, k, v, cu_q, cu_k, False)
    k2, v2 = k.clone(), v.clone()
    k2[200:330] = float("nan")
    v2[200:330] = float("inf")
    o2, l2 = gpu_varlen(q, k2, v2, cu_q, cu_k, False)
    for rows in (slice(0, 200), slice(330, 400)):
        assert np.isfinite(o1[rows]).all()
        assert np.array_equal(o1[rows], o2[rows]) and np.array_equal(l1[:, rows], l2[:, rows])
    assert np.isnan(o1[400:]).all() and np.isnan(l1[:, 400:]).all()   # untouched
    ro, rl = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=False)
    assert_close(o1[:400], l1[:, :400], ro[:400], rl[:, :400], "with NaN neighbours")


def test_varlen_equal_lengths_bit_identical_to_dense():
    """All sequences of one length: the same tiles and arithmetic as attn_fwd
    (causal, so no tail split), in the packed layout."""
    B, H, N, d = 3, 4, 700, 128
    q, k, v, cu_q, cu_k = make_varlen_inputs([N] * B, [N] * B, H, H, d, seed=815)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, True)
    qd = q.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().cuda()
    kd = k.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().cuda()
    vd = v.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().cuda()
    od, ld = ea.forward(qd, kd, vd, causal=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    od = od.permute(0, 2, 1, 3).reshape(B * N, H, d).cpu().double().numpy()
    ld = ld.permute(1, 0, 2).reshape(H, B * N).cpu().double().numpy()
    assert np.array_equal(o, od) and np.array_equal(lse, ld)


def test_varlen_bad_offsets_reported_and_skipped():
    """A sequence longer than max_seqlen, or causal with more queries than keys,
    is not computed; the device error word reports it; the others are exact."""
    lens = [64, 236, 64]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lens, lens, 2, 2, 64, seed=816)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full(q.shape, 7.0, dtype=torch.float32).cuda()
    ea.attn_fwd_varlen(qd, kd, vd, o, cu_q.cuda(), cu_k.cuda(), 200, 236, None, causal=False)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == ea.ATTN_ERR_INVALID_ARG
    o = o.cpu().double().numpy()
    assert (o[64:300] == 7.0).all()
    ro, rl = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=False)
    for rows in (slice(0, 64), slice(300, 364)):
        assert np.abs(o[rows] - ro[rows]).max() <= 1e-2
    lk = [64, 100, 64]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lens, lk, 2, 2, 64, seed=817)
    o2, _ = gpu_varlen(q, k, v, cu_q, cu_k, True, expect_error=ea.ATTN_ERR_INVALID_ARG)
    assert np.isnan(o2[64:300]).all()


@pytest.mark.parametrize("d", [128, 256])
def test_varlen_repeatable_and_graph_capture(d):
    q, k, v, cu_q, cu_k = make_varlen_inputs(LENS, LENS, 8, 2, d, seed=818)
    qd, kd, vd, cq, ck = q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda()
    o = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((8, q.shape[0]), dtype=torch.float32, device="cuda")
    ea.attn_fwd_varlen(qd, kd, vd, o, cq, ck, 600, 600, lse, causal=True)
    torch.cuda.synchronize()
    ref_o, ref_l = o.clone(), lse.clone()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        o.zero_()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            ea.attn_fwd_varlen(qd, kd, vd, o, cq, ck, 600, 600, lse, causal=True, stream=s)
    for _ in range(3):
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
    assert ea.attn_last_device_error() == 0


def test_varlen_prefill_workload_sampled():
    """The packed causal prefill workload at full size (16 sequences of
    U[256, 4096] tokens, H16, d128); the oracle checks whole heads of three
    sequences."""
    cfg = VARLEN
    lens = varlen_lengths(cfg.n_seqs, cfg.len_lo, cfg.len_hi, cfg.seed)
    q, k, v, cu_q, cu_k = make_varlen_inputs(lens, lens, cfg.Hq, cfg.Hkv, cfg.d, cfg.seed)
    o, lse = gpu_varlen(q, k, v, cu_q, cu_k, cfg.causal, cfg.scale)
    for b in (0, int(np.argmax(lens)), cfg.n_seqs - 1):
        s, e = int(cu_q[b]), int(cu_q[b + 1])
        qb = q[s:e, 0:2].permute(1, 0, 2).unsqueeze(0)
        kb = k[s:e, 0:2].permute(1, 0, 2).unsqueeze(0)
        vb = v[s:e, 0:2].permute(1, 0, 2).unsqueeze(0)
        ro, rl = oracle.attention(qb, kb, vb, causal=True, scale=cfg.scale)
        assert_close(o[s:e, 0:2], lse[0:2, s:e], ro[0].transpose(1, 0, 2), rl[0], f"seq {b}")


# ---------------------------------------------------------------- backward --
def _dout_packed(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def gpu_bwd_varlen(q, k, v, do, cu_q, cu_k, causal, scale=None, grad_dtype=torch.float32,
                   init=float("nan"), expect_error=0, max_q=None, max_k=None):
    lq = (cu_q[1:] - cu_q[:-1]).tolist()
    lk = (cu_k[1:] - cu_k[:-1]).tolist()
    mq = max_q or max(max(lq), 1)
    mk = max_k or max(max(lk), 1)
    qd, kd, vd, dod, cq, ck = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu_q.cuda(), cu_k.cuda()
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device="cuda")
    ea.attn_fwd_varlen(qd, kd, vd, o, cq, ck, mq, mk, lse, causal=causal, scale=scale)
    dq = torch.full(q.shape, init, dtype=grad_dtype, device="cuda")
    dk = torch.full(k.shape, init, dtype=grad_dtype, device="cuda")
    dv = torch.full(v.shape, init, dtype=grad_dtype, device="cuda")
    ea.attn_bwd_varlen(qd, kd, vd, o, dod, lse, dq, dk, dv, cq, ck, mq, mk, causal=causal,
                       scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == expect_error
    return tuple(t.float().cpu().double().numpy() for t in (dq, dk, dv))


def _bwd_close(got, ref, rows, what):
    from test_gpu_bwd import _check
    _check(got[rows], ref[rows], what)


@pytest.mark.parametrize("d", [64, 128, 96, 136, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_bwd_parity(d, causal):
    """Packed backward against the per-sequence oracle: empty, single-row and
    ragged sequences, GQA 4:1; rows outside every sequence never written."""
    q, k, v, cu_q, cu_k = make_varlen_inputs(LENS, LENS, 8, 2, d, seed=870 + d, extra_rows=20)
    do = _dout_packed(q.shape, 871 + d)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = gpu_bwd_varlen(q, k, v, do, cu_q, cu_k, causal, scale)
    rq, rk, rv = oracle.attention_bwd_varlen(q, k, v, do, cu_q, cu_k, causal=causal, scale=scale)
    nq, nk = int(cu_q[-1]), int(cu_k[-1])
    _bwd_close(dq, rq, slice(0, nq), f"dQ d={d} causal={causal}")
    _bwd_close(dk, rk, slice(0, nk), f"dK d={d} causal={causal}")
    _bwd_close(dv, rv, slice(0, nk), f"dV d={d} causal={causal}")
    assert np.isnan(dq[nq:]).all() and np.isnan(dk[nk:]).all() and np.isnan(dv[nk:]).all()


@pytest.mark.parametrize("d", [128, 256])
def test_varlen_bwd_cross_lengths(d):
    """Queries and keys of different lengths per sequence (bottom-right causal),
    a sequence without queries (its keys get zero gradients), bf16 gradients."""
    lq = [100, 0, 300, 1, 129]
    lk = [400, 50, 300, 700, 1000]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lq, lk, 4, 4, d, seed=872)
    do = _dout_packed(q.shape, 873)
    for causal in (False, True):
        dq, dk, dv = gpu_bwd_varlen(q, k, v, do, cu_q, cu_k, causal)
        rq, rk, rv = oracle.attention_bwd_varlen(q, k, v, do, cu_q, cu_k, causal=causal)
        _bwd_close(dq, rq, slice(None), f"dQ causal={causal}")
        _bwd_close(dk, rk, slice(None), f"dK causal={causal}")
        _bwd_close(dv, rv, slice(None), f"dV causal={causal}")
        assert (dk[400:450] == 0).all() and (dv[400:450] == 0).all()
    gq, gk, gv = gpu_bwd_varlen(q, k, v, do, cu_q, cu_k, True, grad_dtype=torch.bfloat16)
    rq, rk, rv = oracle.attention_bwd_varlen(q, k, v, do, cu_q, cu_k, causal=True)
    from test_gpu_bwd import _check
    _check(gq, rq, "dQ bf16", bf16=True)
    _check(gk, rk, "dK bf16", bf16=True)
    _check(gv, rv, "dV bf16", bf16=True)


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_varlen_bwd_many_sequences(d, causal):
    """Sixty sequences of 1..700 tokens: far more items than SMs, most of
    them past their sequence's end (no work), mixed with short and long ones
    on the same persistent CTAs."""
    rng = np.random.default_rng(957)
    lens = [int(x) for x in rng.integers(1, 701, 60)]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lens, lens, 4, 2, d, seed=958)
    do = _dout_packed(q.shape, 959)
    scale = 1 / math.sqrt(d)
    dq, dk, dv = gpu_bwd_varlen(q, k, v, do, cu_q, cu_k, causal, scale)
    rq, rk, rv = oracle.attention_bwd_varlen(q, k, v, do, cu_q, cu_k, causal=causal, scale=scale)
    _bwd_close(dq, rq, slice(None), f"dQ d={d} causal={causal}")
    _bwd_close(dk, rk, slice(None), f"dK d={d} causal={causal}")
    _bwd_close(dv, rv, slice(None), f"dV d={d} causal={causal}")


@pytest.mark.parametrize("d", [128, 256])
def test_varlen_bwd_equal_lengths_bit_identical_to_dense(d):
    """All sequences of one length: the dense backward's tiles and arithmetic
    in the packed layout (both fed the same forward outputs)."""
    B, H, N = 3, 4, 700
    q, k, v, cu_q, cu_k = make_varlen_inputs([N] * B, [N] * B, H, H, d, seed=874)
    do = _dout_packed(q.shape, 875)
    dense = lambda t: t.reshape(B, N, H, d).permute(0, 2, 1, 3).contiguous().cuda()  # noqa: E731
    packed = lambda t: t.permute(0, 2, 1, 3).reshape(B * N, H, d).contiguous()  # noqa: E731
    for causal in (False, True):
        od, ld = ea.forward(dense(q), dense(k), dense(v), causal=causal, out_dtype=torch.float32)
        rq, rk, rv = ea.backward(dense(q), dense(k), dense(v), od, dense(do), ld, causal=causal,
                                 grad_dtype=torch.float32)
        grads = [torch.empty(t.shape, dtype=torch.float32, device="cuda") for t in (q, k, v)]
        ea.attn_bwd_varlen(q.cuda(), k.cuda(), v.cuda(), packed(od), do.cuda(),
                           ld.permute(1, 0, 2).reshape(H, B * N).contiguous(), *grads,
                           cu_q.cuda(), cu_k.cuda(), N, N, causal=causal)
        torch.cuda.synchronize()
        assert ea.attn_last_device_error() == 0
        for got, ref in zip(grads, (rq, rk, rv)):
            assert torch.equal(got, packed(ref)), f"causal={causal}"


def test_varlen_bwd_bad_offsets_reported_and_skipped():
    """A sequence longer than max_seqlen is not computed (its gradient rows are
    left as they were), the device error word reports it, the other sequences
    are exact."""
    lens = [64, 236, 64]
    q, k, v, cu_q, cu_k = make_varlen_inputs(lens, lens, 2, 2, 64, seed=876)
    do = _dout_packed(q.shape, 877)
    qd, kd, vd, dod, cq, ck = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu_q.cuda(), cu_k.cuda()
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty((2, q.shape[0]), dtype=torch.float32, device="cuda")
    ea.attn_fwd_varlen(qd, kd, vd, o, cq, ck, 236, 236, lse)
    dq = torch.full(q.shape, 7.0, dtype=torch.float32, device="cuda")
    dk = torch.full(k.shape, 7.0, dtype=torch.float32, device="cuda")
    dv = torch.full(v.shape, 7.0, dtype=torch.float32, device="cuda")
    ea.attn_bwd_varlen(qd, kd, vd, o, dod, lse, dq, dk, dv, cq, ck, 200, 236)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == ea.ATTN_ERR_INVALID_ARG
    dq, dk, dv = (t.cpu().double().numpy() for t in (dq, dk, dv))
    assert (dq[64:300] == 7.0).all() and (dk[64:300] == 7.0).all() and (dv[64:300] == 7.0).all()
    rq, rk, rv = oracle.attention_bwd_varlen(q, k, v, do, cu_q, cu_k)
    for rows in (slice(0, 64), slice(300, 364)):
        _bwd_close(dq, rq, rows, "dQ")
        _bwd_close(dk, rk, rows, "dK")
        _bwd_close(dv, rv, rows, "dV")


def test_varlen_bwd_repeatable_and_graph_capture():
    q, k, v, cu_q, cu_k = make_varlen_inputs(LENS, LENS, 8, 2, 128, seed=878)
    do = _dout_packed(q.shape, 879)
    qd, kd, vd, dod, cq, ck = q.cuda(), k.cuda(), v.cuda(), do.cuda(), cu_q.cuda(), cu_k.cuda()
    o = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((8, q.shape[0]), dtype=torch.float32, device="cuda")
    ea.attn_fwd_varlen(qd, kd, vd, o, cq, ck, 600, 600, lse, causal=True)
    grads = [torch.empty(t.shape, dtype=torch.bfloat16, device="cuda") for t in (q, k, v)]
    ws = torch.empty(ea.attn_bwd_varlen_workspace_size(len(LENS), 8, 2, q.shape[0], 128),
                     dtype=torch.uint8, device="cuda")
    ea.attn_bwd_varlen(qd, kd, vd, o, dod, lse, *grads, cq, ck, 600, 600, causal=True, workspace=ws)
    torch.cuda.synchronize()
    ref = [t.clone() for t in grads]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for t in grads:
            t.zero_()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            ea.attn_bwd_varlen(qd, kd, vd, o, dod, lse, *grads, cq, ck, 600, 600, causal=True,
                               workspace=ws, stream=s)
    for _ in range(3):
        for t in grads:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(grads, ref))
    assert ea.attn_last_device_error() == 0
