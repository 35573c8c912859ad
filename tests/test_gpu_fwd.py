"""GPU parity of attn_fwd against the fp64 oracle, through the C ABI.

Tolerances (fp32 output): max |dO| <= 1e-2, relative L2(O) <= 5e-3,
max |dLSE| <= 1e-3.  bf16 output is compared with the oracle rounded to bf16
(round-to-nearest-even) and a bound of 1e-2 plus half a bf16 ulp of the
reference value.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import exact_attention_14_gb300 as ea
import oracle
from exact_attention_14_gb300.inputs import (GQA, LONG, PREFILL, TINY, make_config_inputs,
                                             make_fwd_inputs)

pytestmark = pytest.mark.gpu

MAX_ABS_O = 1e-2
REL_L2_O = 5e-3
MAX_ABS_LSE = 1e-3


def gpu_fwd(q, k, v, causal, scale=None, out_dtype=torch.float32, with_lse=True):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = ea.forward(qd, kd, vd, causal=causal, scale=scale, out_dtype=out_dtype,
                        return_lse=with_lse)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    o = o.float().cpu().double().numpy()
    lse = None if lse is None else lse.cpu().double().numpy()
    return o, lse


def assert_close(o, lse, o_ref, lse_ref, what=""):
    d_o = np.abs(o - o_ref)
    rel = np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    assert d_o.max() <= MAX_ABS_O, f"{what}: max|dO| = {d_o.max():.3e}"
    assert rel <= REL_L2_O, f"{what}: relL2(O) = {rel:.3e}"
    if lse is not None:
        d_l = np.abs(lse - lse_ref)
        assert d_l.max() <= MAX_ABS_LSE, f"{what}: max|dLSE| = {d_l.max():.3e}"


def bf16_round(x):
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


def assert_close_bf16(o, o_ref, what=""):
    ref = bf16_round(o_ref)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 8)
    err = np.abs(o - ref)
    assert (err <= MAX_ABS_O + half_ulp).all(), f"{what}: bf16 O off by {err.max():.3e}"


# ------------------------------- the configs --------------------------------
def test_tiny_config_full():
    q, k, v = make_config_inputs(TINY)
    o, lse = gpu_fwd(q, k, v, False, TINY.scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=False, scale=TINY.scale)
    assert_close(o, lse, o_ref, lse_ref, "tiny")


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_config_full(causal):
    q, k, v = make_config_inputs(PREFILL)
    o, lse = gpu_fwd(q, k, v, causal, PREFILL.scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=PREFILL.scale)
    assert_close(o, lse, o_ref, lse_ref, f"prefill causal={causal}")


def sampled_rows(cfg, full_heads, n_random, seed):
    rng = np.random.default_rng(seed)
    rows = [(b, h, i) for (b, h) in full_heads for i in range(cfg.N)]
    rows += [(int(rng.integers(cfg.B)), int(rng.integers(cfg.Hq)), int(rng.integers(cfg.N)))
             for _ in range(n_random)]
    # the first and last rows of a few heads (diagonal tiles, longest rows)
    for h in range(0, cfg.Hq, max(1, cfg.Hq // 4)):
        rows += [(cfg.B - 1, h, 0), (cfg.B - 1, h, cfg.N - 1), (0, h, 127), (0, h, 128)]
    return np.array(rows, np.int32)


@pytest.mark.parametrize("cfg,full_heads", [
    (LONG, [(0, 0), (0, 31)]),
    (GQA, [(0, 0), (7, 31), (3, 13)]),
])
def test_large_configs_sampled(cfg, full_heads):
    """Full-size launch; the oracle computes whole heads plus random rows."""
    q, k, v = make_config_inputs(cfg)
    o, lse = gpu_fwd(q, k, v, True, cfg.scale)
    rows = sampled_rows(cfg, full_heads, 2048, cfg.seed)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, rows, causal=True, scale=cfg.scale)
    o_s = o[rows[:, 0], rows[:, 1], rows[:, 2]]
    lse_s = lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(o_s, lse_s, o_ref, lse_ref, cfg.name)
    # properties that hold for every row: finite, LSE >= max possible lower bound
    assert np.isfinite(o).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("cfg", [LONG, GQA], ids=["long", "gqa"])
def test_large_configs_full(cfg):
    """Full-size launch of the long-context (B1 H32 N16384, outlier channels)
    and GQA (B8 Hq32 Hkv8 N4096) causal workloads, every row of O and LSE
    against the fp64 oracle (about a minute of oracle time on 16 cores)."""
    q, k, v = make_config_inputs(cfg)
    o, lse = gpu_fwd(q, k, v, True, cfg.scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True, scale=cfg.scale)
    assert_close(o, lse, o_ref, lse_ref, f"{cfg.name} (all rows)")


# ------------------------------- edge cases ---------------------------------
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 1, 1, 1, 1, 64, False),
    (1, 1, 1, 1, 1, 128, True),
    (1, 2, 1, 17, 17, 64, True),
    (2, 2, 2, 128, 128, 128, True),
    (1, 1, 1, 129, 129, 128, False),
    (1, 3, 1, 255, 255, 64, True),
    (1, 1, 1, 256, 256, 128, True),
    (1, 2, 2, 257, 257, 128, False),
    (1, 4, 2, 300, 300, 128, True),
    (2, 8, 1, 1000, 1000, 64, True),
    (1, 2, 2, 100, 333, 128, False),   # Nq < Nk
    (1, 2, 2, 100, 333, 128, True),    # bottom-right causal, mid-tile diagonal
    (1, 2, 1, 384, 1000, 64, True),
    (1, 1, 1, 700, 90, 128, False),    # Nq > Nk
    (3, 16, 2, 520, 520, 128, True),   # GQA 8:1
])
def test_edge_shapes(B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=100 + Nq + Nk + d)
    scale = 1 / math.sqrt(d)
    o, lse = gpu_fwd(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=scale)
    assert_close(o, lse, o_ref, lse_ref, f"{(B, Hq, Hkv, Nq, Nk, d, causal)}")


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_output_and_no_lse(d):
    q, k, v = make_fwd_inputs(2, 4, 2, 333, 333, d, seed=7)
    o, lse = gpu_fwd(q, k, v, True, None, out_dtype=torch.bfloat16, with_lse=False)
    assert lse is None
    o_ref, _ = oracle.attention(q, k, v, causal=True)
    assert_close_bf16(o, o_ref, "bf16 out")


def test_zero_scale_gives_uniform_average():
    q, k, v = make_fwd_inputs(1, 2, 2, 200, 200, 128, seed=9)
    o, lse = gpu_fwd(q, k, v, True, 0.0)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True, scale=0.0)
    assert_close(o, lse, o_ref, lse_ref, "scale 0")


def test_outlier_channels_large_logits():
    """Long-context style outliers (|s| up to ~100) on a small shape."""
    q, k, v = make_fwd_inputs(1, 4, 4, 1024, 1024, 128, seed=21, outlier_channels=4)
    o, lse = gpu_fwd(q, k, v, True, 1 / math.sqrt(128))
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    assert_close(o, lse, o_ref, lse_ref, "outliers")


# ------------------------------- tail split ----------------------------------
# Non-causal launches whose unit count is not a multiple of the SM count cut
# their last units along the KV range; the last piece to finish merges them.

def _num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,out_f32,outliers", [
    (1, 1, 1, 256, 4000, 64, True, 0),      # one unit in 8 pieces, ragged last KV tile
    (1, 8, 8, 100, 2048, 128, True, 0),     # Q tile 1 of every unit is empty
    (5, 7, 7, 1500, 1500, 128, True, 0),    # whole units, then a split tail
    (1, 3, 1, 300, 5000, 64, False, 0),     # GQA 3:1, bf16 output
    (1, 4, 4, 1024, 1024, 128, True, 4),    # outlier channels: piece maxima far apart
])
def test_tail_split_parity(B, Hq, Hkv, Nq, Nk, d, out_f32, outliers):
    n_full, n_split, parts = ea.attn_fwd_split_plan(B, Hq, Hkv, Nq, Nk, d, False, _num_sms())
    assert n_split > 0 and parts > 1
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=200 + Nq + d,
                              outlier_channels=outliers)
    scale = 1 / math.sqrt(d)
    o, lse = gpu_fwd(q, k, v, False, scale,
                     out_dtype=torch.float32 if out_f32 else torch.bfloat16)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=False, scale=scale)
    what = f"split {(B, Hq, Hkv, Nq, Nk, d)} into {n_split} x {parts}"
    if out_f32:
        assert_close(o, lse, o_ref, lse_ref, what)
    else:
        assert_close_bf16(o, o_ref, what)
        assert np.abs(lse - lse_ref).max() <= MAX_ABS_LSE


def test_repeatable_and_stream_ordered():
    """Same inputs twice on a side stream give bit-identical results."""
    q, k, v = (t.cuda() for t in make_fwd_inputs(2, 4, 4, 640, 640, 128, seed=3))
    s = torch.cuda.Stream()
    outs = []
    with torch.cuda.stream(s):
        for _ in range(2):
            o, lse = ea.forward(q, k, v, causal=True, out_dtype=torch.float32, stream=s)
            outs.append((o.clone(), lse.clone()))
    s.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


# ------------------------------ the work queue -------------------------------
# The kernel's CTAs take units from a device-side queue that the last CTA
# returns to zero.  A unit's result does not depend on which CTA computes it,
# so every launch below must match its eager reference bit for bit.

@pytest.mark.parametrize("causal", [True, False])
def test_graph_replays_reuse_the_work_queue(causal):
    """A captured launch replays on the same queue slot: each replay must see a
    reset queue and compute every unit.  Non-causal, the shape's 64 units are
    split in pieces, whose partials go to the caller's workspace."""
    B, H, N, d = 2, 8, 1024, 128
    q, k, v = (t.cuda() for t in make_fwd_inputs(B, H, H, N, N, d, seed=21))
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    need = ea.attn_fwd_workspace_size(B, H, H, N, N, d, causal)
    assert (need > 0) == (not causal)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    ea.attn_fwd(q, k, v, o, lse, causal=causal, workspace=ws)  # first call outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ea.attn_fwd(q, k, v, o, lse, causal=causal, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for seed in (22, 23, 24):
        q2, k2, v2 = (t.cuda() for t in make_fwd_inputs(B, H, H, N, N, d, seed=seed))
        q.copy_(q2); k.copy_(k2); v.copy_(v2)
        o.fill_(float("nan"))
        g.replay()
        o_ref, l_ref = ea.forward(q, k, v, causal=causal, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert ea.attn_last_device_error() == 0
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref), f"replay with seed {seed}"


def test_workspace_size_and_checks():
    """The workspace holds the split tail units' partials: (d' + 3) x 32 fp32
    values per piece and per 32 query rows (d' = 64 or 128).  A missing,
    short or misaligned workspace is refused with ATTN_ERR_WORKSPACE before
    anything is enqueued; shapes without a split need none."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lib = ea.load()
    for (B, H, N, d) in ((4, 16, 2048, 128), (3, 19, 2048, 64), (2, 8, 1024, 128)):
        n_full, n_split, parts = ea.attn_fwd_split_plan(B, H, H, N, N, d, False, sms)
        want = n_split * parts * 8 * ((64 if d <= 64 else 128) + 3) * 32 * 4
        assert ea.attn_fwd_workspace_size(B, H, H, N, N, d, False) == want
        assert ea.attn_fwd_workspace_size(B, H, H, N, N, d, True) == 0
    B, H, N, d = 4, 16, 2048, 128
    need = ea.attn_fwd_workspace_size(B, H, H, N, N, d, False)
    assert need > 0
    q, k, v = (t.cuda() for t in make_fwd_inputs(B, H, H, N, N, d, seed=1))
    o = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(need + 16, dtype=torch.uint8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    call = lambda c, w, nb: lib.attn_fwd(p(q), p(k), p(v), p(o), None, B, H, H, N, N, d, c,
                                         ctypes.c_float(d ** -0.5), ea.ATTN_OUT_F32, w, nb, None)
    assert call(0, None, 0) == ea.ATTN_ERR_WORKSPACE
    assert call(0, p(ws), need - 1) == ea.ATTN_ERR_WORKSPACE
    assert call(0, ctypes.c_void_p(ws.data_ptr() + 8), need) == ea.ATTN_ERR_WORKSPACE
    assert call(1, None, 0) == ea.ATTN_OK          # causal: nothing is split
    assert call(0, p(ws), need) == ea.ATTN_OK
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    o_ref, _ = ea.forward(q, k, v, causal=False, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)


@pytest.mark.parametrize("causal", [True, False])
def test_concurrent_launches_on_two_streams(causal):
    """Launches in flight together on two streams use different queue slots
    (and, split, different partial buffers)."""
    cases = [make_fwd_inputs(4, 8, 2, 1536, 1536, 128, seed=31),
             make_fwd_inputs(3, 8, 8, 1000, 1000, 64, seed=32)]
    cases = [tuple(t.cuda() for t in c) for c in cases]
    refs = [ea.forward(*c, causal=causal, out_dtype=torch.float32) for c in cases]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    outs = [[], []]
    for _ in range(4):
        for i, (st, c) in enumerate(zip(streams, cases)):
            with torch.cuda.stream(st):
                outs[i].append(ea.forward(*c, causal=causal, out_dtype=torch.float32, stream=st))
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    for i in range(2):
        for o, lse in outs[i]:
            assert torch.equal(o, refs[i][0]) and torch.equal(lse, refs[i][1])


@pytest.mark.parametrize("causal", [False, True])
def test_row_max_jumps_late(causal):
    """Keys late in each row score far higher than the early ones, so the row
    max rises by more than tau after the first KV tiles and the softmax must
    rescale O and redo the tile's exponentials (the rare path)."""
    q, k, v = make_fwd_inputs(2, 4, 4, 1000, 1000, 128, seed=41)
    k = k.clone()
    k[:, :, 600:, :] *= 8.0   # a power of two: exact in bf16
    k[:, :, 900:, :] *= 4.0
    o, lse = gpu_fwd(q, k, v, causal, 1 / math.sqrt(128))
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    assert_close(o, lse, o_ref, lse_ref, f"late max, causal={causal}")


# ------------------------------ other head dims ------------------------------
@pytest.mark.parametrize("d,causal", [(32, True), (48, False), (80, True), (96, False),
                                      (96, True), (120, True)])
def test_head_dims_padded(d, causal):
    """Head dims below 64 / 128 run on those kernels: the loads zero-fill the
    columns past d and the stores skip them."""
    q, k, v = make_fwd_inputs(2, 4, 2, 300, 300, d, seed=500 + d)
    scale = 1 / math.sqrt(d)
    o, lse = gpu_fwd(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=scale)
    assert_close(o, lse, o_ref, lse_ref, f"d={d} causal={causal}")
    ob, _ = gpu_fwd(q, k, v, causal, scale, out_dtype=torch.bfloat16, with_lse=False)
    assert_close_bf16(ob, o_ref, f"bf16 out d={d}")


def test_head_dim_96_split_tail():
    """d = 96 through the tail split (the merge's stores also stop at d)."""
    q, k, v = make_fwd_inputs(1, 8, 8, 100, 2048, 96, seed=601)
    n_full, n_split, parts = ea.attn_fwd_split_plan(1, 8, 8, 100, 2048, 96, False, _num_sms())
    assert n_split > 0
    o, lse = gpu_fwd(q, k, v, False, 1 / math.sqrt(96))
    o_ref, lse_ref = oracle.attention(q, k, v, causal=False)
    assert_close(o, lse, o_ref, lse_ref, "d=96 split")


# ---------------------- head dims above 128 (wide kernel) --------------------
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 1, 1, 128, 128, 256, False),
    (2, 4, 2, 300, 300, 256, True),      # GQA, ragged tails
    (2, 4, 2, 300, 300, 192, False),
    (1, 4, 1, 200, 520, 192, True),      # MQA, bottom-right causal, Nq < Nk
    (1, 2, 2, 700, 90, 256, False),      # Nq > Nk
    (1, 2, 2, 257, 257, 136, True),      # padded to 192
    (1, 2, 2, 333, 333, 160, False),
    (1, 2, 2, 129, 400, 248, True),      # padded to 256
])
def test_wide_head_dims(B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=1000 + d + Nq)
    scale = 1 / math.sqrt(d)
    o, lse = gpu_fwd(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=scale)
    assert_close(o, lse, o_ref, lse_ref, f"{(B, Hq, Hkv, Nq, Nk, d, causal)}")
    ob, _ = gpu_fwd(q, k, v, causal, scale, out_dtype=torch.bfloat16, with_lse=False)
    assert_close_bf16(ob, o_ref, f"bf16 out d={d}")


def test_wide_sampled_heads_long():
    """B2 H8 N4096 d256, causal and not; the oracle checks two whole heads."""
    q, k, v = make_fwd_inputs(2, 8, 8, 4096, 4096, 256, seed=1100)
    for causal in (False, True):
        o, lse = gpu_fwd(q, k, v, causal, 1 / 16)
        for (b, h) in ((0, 0), (1, 7)):
            sl = (slice(b, b + 1), slice(h, h + 1))
            o_ref, lse_ref = oracle.attention(q[sl], k[sl], v[sl], causal=causal, scale=1 / 16)
            assert_close(o[sl], lse[sl], o_ref, lse_ref, f"head {(b, h)} causal={causal}")


def test_wide_repeatable_and_graph():
    q, k, v = make_fwd_inputs(2, 4, 2, 640, 640, 256, seed=1200)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    ea.attn_fwd(qd, kd, vd, o, lse, causal=True)
    torch.cuda.synchronize()
    ref_o, ref_l = o.clone(), lse.clone()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            ea.attn_fwd(qd, kd, vd, o, lse, causal=True, stream=s)
    for _ in range(3):
        o.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)
    assert ea.attn_last_device_error() == 0


# ------------------------------- edge shapes ---------------------------------
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (1, 1, 1, 1, 1, 128, False),        # one query, one key
    (1, 2, 1, 1, 1, 64, True),
    (2, 2, 2, 5, 7, 64, False),         # fewer keys than a row of 8
    (1, 4, 4, 1, 2049, 128, True),      # a single query row over a ragged key range
    (1, 2, 2, 2, 129, 128, False),
    (64, 32, 8, 128, 128, 64, True),    # 2048 heads, one unit each
    (2, 32, 1, 200, 300, 128, False),   # MQA group of 32
    (3, 19, 19, 2048, 2048, 64, False), # tail split at d = 64
])
def test_small_and_many_head_shapes(B, Hq, Hkv, Nq, Nk, d, causal):
    q, k, v = make_fwd_inputs(B, Hq, Hkv, Nq, Nk, d, seed=1300 + Nq + Nk)
    scale = 1 / math.sqrt(d)
    o, lse = gpu_fwd(q, k, v, causal, scale)
    if B * Hq * Nq > 4096:
        rng = np.random.default_rng(Nq + Nk)
        rows = np.stack([rng.integers(0, B, 256), rng.integers(0, Hq, 256), rng.integers(0, Nq, 256)], 1)
        ro, rl = oracle.attention_rows(q, k, v, rows, causal=causal, scale=scale)
        got = np.stack([o[b, h, i] for b, h, i in rows])
        gl = np.array([lse[b, h, i] for b, h, i in rows])
        assert_close(got, gl, ro, rl, f"{(B, Hq, Hkv, Nq, Nk, d, causal)} sampled")
    else:
        o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=scale)
        assert_close(o, lse, o_ref, lse_ref, f"{(B, Hq, Hkv, Nq, Nk, d, causal)}")
