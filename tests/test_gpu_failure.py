"""Failure detection on the GPU without a fault: the kernels' bounded waits.

Every spin-wait in the library's kernels gives up after 2 s, records
ATTN_ERR_TIMEOUT in the device error word and returns, so the context stays
usable.  attn_selftest_bounded_wait runs that same wait on an mbarrier that
nothing ever arrives on (the flag that nothing sets)."""
import math
import time

import numpy as np
import pytest
import torch

import exact_attention_14_gb300 as ea
import oracle
from exact_attention_14_gb300.inputs import make_fwd_inputs

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_context_stays_usable():
    assert ea.attn_last_device_error() == 0
    res = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    ea.attn_selftest_bounded_wait(0, res)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert res.item() == 2                      # ran out of time
    assert 1.9 < waited < 30.0
    assert ea.attn_last_device_error() == ea.ATTN_ERR_TIMEOUT
    assert ea.attn_last_device_error() == 0     # read and cleared
    # the context is still usable: a forward runs and matches the oracle
    q, k, v = make_fwd_inputs(1, 2, 2, 200, 200, 64, seed=1400)
    o, lse = ea.forward(q.cuda(), k.cuda(), v.cuda(), causal=True, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    ro, rl = oracle.attention(q, k, v, causal=True, scale=1 / math.sqrt(64))
    assert np.abs(o.cpu().double().numpy() - ro).max() <= 1e-2


def test_abort_flag_ends_the_wait_early():
    res = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    ea.attn_selftest_bounded_wait(1, res)
    torch.cuda.synchronize()
    assert res.item() == 1                      # left through the abort flag
    assert time.perf_counter() - t0 < 1.5
    assert ea.attn_last_device_error() == 0
