"""attn_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (for example a plugin whose host framework owns all GPU memory
through its own pool, or a loop that cannot afford an allocation's implicit
synchronisation).  It keeps its split partials in the library's fixed per-device
scratch array instead of a caller workspace.

Checked through the C ABI against attn_decode with a caller workspace and
against the fp64 oracle, within the parity tolerances used by the other decode
tests, on two calls in a row with different inputs (the second call sees the
first call's leftovers in the shared array).  This file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_14_gb300 as ea
import oracle
from exact_attention_14_gb300.inputs import make_decode_inputs

pytestmark = pytest.mark.gpu

MAX_ABS_O = 1e-2
MAX_ABS_LSE = 1e-3


def _c_call(lib, name, q, kc, vc, sl, o, lse, num_splits, ws=None):
    B, Hq, _, d = q.shape
    Hkv, Nmax = kc.shape[1], kc.shape[2]
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    common = (p(q), p(kc), p(vc), p(sl), p(o), p(lse), B, Hq, Hkv, Nmax, d,
              ctypes.c_float(d ** -0.5), num_splits)
    if name == "attn_decode":
        return lib.attn_decode(*common, p(ws), ws.numel(), ea.ATTN_OUT_F32, stream)
    return lib.attn_decode_noalloc(*common, ea.ATTN_OUT_F32, stream)


def test_noalloc_matches_workspace_decode_on_two_calls_in_a_row(cuda_ok):
    lib = ea.load()
    dev = torch.device("cuda")
    cases = [
        make_decode_inputs(8, 32, 8, 8192, 128, seed=41, len_lo=1, len_hi=8192),
        make_decode_inputs(4, 16, 2, 3000, 64, seed=42, len_lo=500, len_hi=3000),
    ]
    refs = [oracle.decode(*c) for c in cases]
    for num_splits in (0, 5):
        for (q, kc, vc, sl), (o_or, l_or) in zip(cases, refs):
            q, kc, vc, sl = q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev)
            B, Hq, _, d = q.shape
            need = ea.attn_decode_workspace_size(B, Hq, kc.shape[1], kc.shape[2], d, num_splits)
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
            o_ref = torch.empty(B, Hq, 1, d, dtype=torch.float32, device=dev)
            l_ref = torch.empty(B, Hq, 1, dtype=torch.float32, device=dev)
            assert _c_call(lib, "attn_decode", q, kc, vc, sl, o_ref, l_ref, num_splits, ws) == 0
            o = torch.full_like(o_ref, float("nan"))
            lse = torch.full_like(l_ref, float("nan"))
            assert _c_call(lib, "attn_decode_noalloc", q, kc, vc, sl, o, lse, num_splits) == 0
            torch.cuda.synchronize()
            assert ea.attn_last_device_error() == 0
            assert torch.isfinite(o).all() and torch.isfinite(lse).all()
            assert (o - o_ref).abs().max().item() <= MAX_ABS_O
            assert (lse - l_ref).abs().max().item() <= MAX_ABS_LSE
            # and against the fp64 oracle directly
            assert np.abs(o.cpu().double().numpy() - o_or).max() <= MAX_ABS_O
            assert np.abs(lse.cpu().double().numpy() - l_or).max() <= MAX_ABS_LSE


def test_noalloc_through_the_binding(cuda_ok):
    q, kc, vc, sl = make_decode_inputs(2, 8, 2, 3000, 128, seed=43, len_lo=1, len_hi=3000)
    o_or, l_or = oracle.decode(q, kc, vc, sl)
    dev = torch.device("cuda")
    o = torch.empty(2, 8, 1, 128, dtype=torch.float32, device=dev)
    lse = torch.empty(2, 8, 1, dtype=torch.float32, device=dev)
    ea.attn_decode_noalloc(q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), o, lse)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    assert np.abs(o.cpu().double().numpy() - o_or).max() <= MAX_ABS_O
    assert np.abs(lse.cpu().double().numpy() - l_or).max() <= MAX_ABS_LSE


def test_noalloc_rejects_requests_beyond_its_scratch(cuda_ok):
    """A shape whose partials need more than the 16 MiB array is refused with
    ATTN_ERR_WORKSPACE before anything is enqueued.  The operands are real
    device tensors of that shape, so the call stays in bounds whatever the
    order of the checks; attn_decode takes the same shape with a workspace."""
    lib = ea.load()
    # 16 sequences x 64 query heads x 128 splits x 129 floats = 67.6 MB
    B, Hq, Hkv, Nmax, d, splits = 16, 64, 8, 8192, 128, 128
    need = ea.attn_decode_workspace_size(B, Hq, Hkv, Nmax, d, splits)
    assert need > 16 << 20
    dev = torch.device("cuda")
    q = torch.zeros(B, Hq, 1, d, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(B, Hkv, Nmax, d, dtype=torch.bfloat16, device=dev)
    sl = torch.full((B,), Nmax, dtype=torch.int32, device=dev)
    o = torch.empty(B, Hq, 1, d, dtype=torch.float32, device=dev)
    lse = torch.empty(B, Hq, 1, dtype=torch.float32, device=dev)
    assert _c_call(lib, "attn_decode_noalloc", q, kc, kc, sl, o, lse, splits) == \
        ea.ATTN_ERR_WORKSPACE
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    assert _c_call(lib, "attn_decode", q, kc, kc, sl, o, lse, splits, ws) == 0
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0


def test_noalloc_rejects_bad_arguments_like_attn_decode(cuda_ok):
    """Null pointers give ATTN_ERR_INVALID_ARG from both entry points, even for
    a shape beyond the scratch array (the argument checks come first)."""
    lib = ea.load()
    for B, Hq, Nmax, splits in ((2, 8, 64, 0), (16, 64, 8192, 128)):
        rc = lib.attn_decode_noalloc(None, None, None, None, None, None, B, Hq, 8, Nmax, 128,
                                     ctypes.c_float(0.1), splits, ea.ATTN_OUT_F32, None)
        assert rc == ea.ATTN_ERR_INVALID_ARG
        rc = lib.attn_decode(None, None, None, None, None, None, B, Hq, 8, Nmax, 128,
                             ctypes.c_float(0.1), splits, None, 0, ea.ATTN_OUT_F32, None)
        assert rc == ea.ATTN_ERR_INVALID_ARG
