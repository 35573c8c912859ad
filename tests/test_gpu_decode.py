"""GPU parity of attn_decode (split-KV + log-sum-exp combine) against the fp64
oracle, through the C ABI; same tolerances as the forward."""
import numpy as np
import pytest
import torch

import exact_attention_14_gb300 as ea
import oracle
from exact_attention_14_gb300.inputs import DECODE, make_decode_config_inputs, make_decode_inputs

pytestmark = pytest.mark.gpu

MAX_ABS_O = 1e-2
REL_L2_O = 5e-3
MAX_ABS_LSE = 1e-3


def gpu_decode(q, kc, vc, sl, num_splits=0, out_dtype=torch.float32, scale=None):
    o, lse = ea.decode(q.cuda(), kc.cuda(), vc.cuda(), sl.cuda(), num_splits=num_splits,
                       out_dtype=out_dtype, scale=scale)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def assert_close(o, lse, o_ref, lse_ref, what=""):
    assert np.isfinite(o).all() and np.isfinite(lse).all(), what
    d_o = np.abs(o - o_ref).max()
    rel = np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref)
    d_l = np.abs(lse - lse_ref).max()
    assert d_o <= MAX_ABS_O, f"{what}: max|dO| {d_o:.3e}"
    assert rel <= REL_L2_O, f"{what}: relL2 {rel:.3e}"
    assert d_l <= MAX_ABS_LSE, f"{what}: max|dLSE| {d_l:.3e}"


@pytest.fixture(scope="module")
def decode_config():
    q, kc, vc, sl = make_decode_config_inputs(DECODE)
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl, scale=DECODE.scale)
    return q, kc, vc, sl, o_ref, lse_ref


def test_decode_config_full(decode_config):
    q, kc, vc, sl, o_ref, lse_ref = decode_config
    o, lse = gpu_decode(q, kc, vc, sl, scale=DECODE.scale)
    assert_close(o, lse, o_ref, lse_ref, "decode config")


@pytest.mark.parametrize("num_splits", [1, 3, 8, 32, 64])
def test_decode_config_any_split_count(decode_config, num_splits):
    """Exactness of the merge for any split count (notes 6.1, exercise 3)."""
    q, kc, vc, sl, o_ref, lse_ref = decode_config
    o, lse = gpu_decode(q, kc, vc, sl, num_splits=num_splits, scale=DECODE.scale)
    assert_close(o, lse, o_ref, lse_ref, f"splits={num_splits}")


def test_nan_tail_never_leaks():
    q, kc, vc, sl = make_decode_inputs(4, 8, 2, 3000, 128, seed=31, len_lo=1, len_hi=3000)
    sl[0] = 1
    sl[1] = 3000
    sl[2] = 65
    sl[3] = 2  # two keys: the LSE must use the unrounded softmax sum
    for b in range(4):  # NaN past the final lengths
        kc[b, :, int(sl[b]):] = float("nan")
        vc[b, :, int(sl[b]):] = float("nan")
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
    for ns in (0, 1, 7):
        o, lse = gpu_decode(q, kc, vc, sl, num_splits=ns)
        assert_close(o, lse, o_ref, lse_ref, f"nan tail splits={ns}")


@pytest.mark.parametrize("B,Hq,Hkv,Nmax,d,lo,hi", [
    (1, 1, 1, 1, 128, 1, 1),
    (2, 8, 8, 100, 64, 1, 100),
    (3, 16, 1, 777, 128, 300, 777),    # MQA, 16 heads packed
    (2, 12, 4, 4100, 64, 4000, 4100),  # group 3
    (5, 32, 4, 2048, 128, 1, 2048),    # group 8
])
def test_decode_shapes(B, Hq, Hkv, Nmax, d, lo, hi):
    q, kc, vc, sl = make_decode_inputs(B, Hq, Hkv, Nmax, d, seed=B + Nmax, len_lo=lo, len_hi=hi)
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
    o, lse = gpu_decode(q, kc, vc, sl)
    assert_close(o, lse, o_ref, lse_ref, f"{(B, Hq, Hkv, Nmax, d)}")


@pytest.mark.parametrize("d", [192, 256])
def test_decode_wide_head_dims_gqa_and_many_splits(d):
    """The 256-column kernel on a GQA group of 8 heads with lengths up to 8192
    (NaN past each length), one split and many, merged inside the split
    kernel, against the oracle."""
    q, kc, vc, sl = make_decode_inputs(4, 32, 4, 8192, d, seed=90 + d, len_lo=1, len_hi=8192,
                                       tail="nan")
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
    for ns in (0, 1, 16):
        o, lse = gpu_decode(q, kc, vc, sl, num_splits=ns)
        assert_close(o, lse, o_ref, lse_ref, f"d={d} splits={ns}")


def test_decode_wide_head_dim_combine_kernel():
    """d = 256 with more (sequence, KV head) groups than the in-kernel merge's
    counter table holds: the splits are merged by the combine kernel."""
    B, Hq, Hkv, Nmax, d = 520, 8, 8, 192, 256
    assert ea.attn_decode_kernel_launches(B, Hq, Hkv, Nmax, d, 3) == 2
    q, kc, vc, sl = make_decode_inputs(B, Hq, Hkv, Nmax, d, seed=97, len_lo=1, len_hi=Nmax)
    o, lse = gpu_decode(q, kc, vc, sl, num_splits=3)
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
    assert_close(o, lse, o_ref, lse_ref, "d=256 combine kernel")


def test_decode_bf16_output():
    q, kc, vc, sl = make_decode_inputs(2, 8, 2, 1500, 128, seed=5, len_lo=700, len_hi=1500)
    o_ref, _ = oracle.decode(q, kc, vc, sl)
    o, _ = gpu_decode(q, kc, vc, sl, out_dtype=torch.bfloat16)
    ref = torch.from_numpy(o_ref).to(torch.bfloat16).double().numpy()
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 8)
    assert (np.abs(o - ref) <= MAX_ABS_O + half_ulp).all()


def test_out_of_range_seqlen_is_reported():
    q, kc, vc, sl = make_decode_inputs(2, 4, 1, 256, 64, seed=8, len_lo=10, len_hi=200)
    sl[1] = 1000  # > Nmax: clamped to Nmax and flagged
    o, lse = ea.decode(q.cuda(), kc.cuda(), vc.cuda(), sl.cuda())
    assert ea.attn_last_device_error() == ea.ATTN_ERR_INVALID_ARG
    assert ea.attn_last_device_error() == 0  # cleared by the read
    sl2 = sl.clone()
    sl2[1] = 256
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl2)
    assert_close(o.float().cpu().double().numpy(), lse.cpu().double().numpy(), o_ref, lse_ref,
                 "clamped")


def test_workspace_too_small_is_rejected():
    q, kc, vc, sl = (t.cuda() for t in make_decode_inputs(1, 4, 1, 512, 64, seed=2, len_lo=512,
                                                          len_hi=512))
    need = ea.attn_decode_workspace_size(1, 4, 1, 512, 64, 0)
    assert need > 0
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    o = torch.empty(1, 4, 1, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(ea.AttnError) as ei:
        ea.attn_decode(q, kc, vc, sl, o, None, workspace=ws)
    assert ei.value.code == ea.ATTN_ERR_WORKSPACE


def test_empty_sequence_gives_zero_output_and_minus_inf_lse():
    """A length of 0 is out of range (reported) and clamps to an empty key set:
    O = 0 and LSE = -inf, the empty-row convention of the oracle."""
    q, kc, vc, sl = make_decode_inputs(3, 8, 2, 2048, 128, seed=12, len_lo=500, len_hi=2048)
    sl[1] = 0
    o, lse = ea.decode(q.cuda(), kc.cuda(), vc.cuda(), sl.cuda(), out_dtype=torch.float32)
    assert ea.attn_last_device_error() == ea.ATTN_ERR_INVALID_ARG
    o = o.cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    assert (o[1] == 0).all() and np.isneginf(lse[1]).all()
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
    keep = [0, 2]
    assert_close(o[keep], lse[keep], o_ref[keep], lse_ref[keep], "other sequences")


def test_many_groups_use_the_combine_kernel():
    """More (sequence, KV head) groups than the in-kernel merge's counter table
    (4096): the merge runs as a second kernel, with the same results."""
    B, Hq, Hkv, Nmax, d = 1100, 8, 4, 192, 64
    assert ea.attn_decode_kernel_launches(B, Hq, Hkv, Nmax, d, 3) == 2
    assert ea.attn_decode_kernel_launches(DECODE.B, DECODE.Hq, DECODE.Hkv, DECODE.Nmax,
                                          DECODE.d) == 1
    q, kc, vc, sl = make_decode_inputs(B, Hq, Hkv, Nmax, d, seed=13, len_lo=1, len_hi=Nmax)
    o, lse = gpu_decode(q, kc, vc, sl, num_splits=3)
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
    assert_close(o, lse, o_ref, lse_ref, "combine kernel")


def test_split_merge_is_repeatable():
    q, kc, vc, sl = (t.cuda() for t in make_decode_inputs(4, 32, 8, 8192, 128, seed=14,
                                                          len_lo=1000, len_hi=8192))
    outs = [ea.decode(q, kc, vc, sl, out_dtype=torch.float32) for _ in range(3)]
    torch.cuda.synchronize()
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


@pytest.mark.parametrize("d", [32, 80, 96, 136, 192, 256])
def test_decode_head_dims_padded(d):
    """Head dims up to 256: d <= 128 on the 64- or 128-column kernel, above on
    the 256-column one (the columns past d read as zeros and are not written)."""
    q, kc, vc, sl = make_decode_inputs(3, 8, 2, 2000, d, seed=70 + d, len_lo=1, len_hi=2000)
    for ns in (0, 5):
        o, lse = gpu_decode(q, kc, vc, sl, num_splits=ns)
        o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
        assert_close(o, lse, o_ref, lse_ref, f"d={d} splits={ns}")
    pad = 64 if d <= 64 else (128 if d <= 128 else 256)
    assert ea.attn_decode_workspace_size(3, 8, 2, 2000, d, 5) == \
        ea.attn_decode_workspace_size(3, 8, 2, 2000, pad, 5)
