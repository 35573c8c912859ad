"""attn_decode_paged: decode over a block-table KV cache, through the C ABI.

The same keys stored contiguously and scattered over pages give bit-identical
results (the kernel does the same arithmetic; only the copy addresses
differ), and the results match the fp64 oracle; pages no block-table entry
points at, and keys past each length, hold NaN and must not leak.
"""
import numpy as np
import pytest
import torch

import exact_attention_14_gb300 as ea
import oracle
from exact_attention_14_gb300.inputs import make_decode_inputs

pytestmark = pytest.mark.gpu

MAX_ABS_O = 1e-2
MAX_ABS_LSE = 1e-3


def _to_pages(cache, page_size, seed, extra_pages=3):
    """[B, Hkv, Nmax, d] -> pages [num_blocks, page_size, Hkv, d] in a random
    order, plus the block table [B, Nmax / page_size].  Unused pages hold NaN."""
    B, Hkv, Nmax, d = cache.shape
    nb = Nmax // page_size
    total = B * nb + extra_pages
    perm = torch.randperm(total, generator=torch.Generator().manual_seed(seed))[: B * nb]
    pages = torch.full((total, page_size, Hkv, d), float("nan"), dtype=cache.dtype)
    blocks = cache.reshape(B, Hkv, nb, page_size, d).permute(0, 2, 3, 1, 4)  # B, nb, ps, Hkv, d
    pages[perm] = blocks.reshape(B * nb, page_size, Hkv, d)
    table = perm.reshape(B, nb).to(torch.int32)
    return pages, table


@pytest.mark.parametrize("page_size,d,num_splits", [(64, 128, 0), (256, 128, 0), (64, 64, 3),
                                                    (128, 128, 7), (64, 256, 0), (128, 192, 5)])
def test_paged_equals_contiguous_bit_for_bit(page_size, d, num_splits):
    q, kc, vc, sl = make_decode_inputs(4, 16, 4, 2048, d, seed=51, len_lo=1, len_hi=2048)
    kp, table = _to_pages(kc, page_size, seed=52)
    vp, _ = _to_pages(vc, page_size, seed=52)
    dev = "cuda"
    o1, l1 = ea.decode(q.to(dev), kc.to(dev), vc.to(dev), sl.to(dev), num_splits=num_splits,
                       out_dtype=torch.float32)
    o2, l2 = ea.decode_paged(q.to(dev), kp.to(dev), vp.to(dev), table.to(dev), sl.to(dev),
                             num_splits=num_splits, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_paged_matches_oracle_and_ignores_nan():
    q, kc, vc, sl = make_decode_inputs(8, 32, 8, 4096, 128, seed=53, len_lo=100, len_hi=4096,
                                       tail="nan")
    kp, table = _to_pages(kc, 256, seed=54, extra_pages=8)
    vp, _ = _to_pages(vc, 256, seed=54, extra_pages=8)
    o, lse = ea.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), sl.cuda(),
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ea.attn_last_device_error() == 0
    o = o.cpu().double().numpy()
    lse = lse.cpu().double().numpy()
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
    assert np.abs(o - o_ref).max() <= MAX_ABS_O
    assert np.abs(lse - lse_ref).max() <= MAX_ABS_LSE


@pytest.mark.parametrize("d", [96, 256])
def test_paged_head_dims(d):
    q, kc, vc, sl = make_decode_inputs(2, 8, 2, 1024, d, seed=55, len_lo=1, len_hi=1024)
    kp, table = _to_pages(kc, 128, seed=56)
    vp, _ = _to_pages(vc, 128, seed=56)
    o1, l1 = ea.decode(q.cuda(), kc.cuda(), vc.cuda(), sl.cuda(), out_dtype=torch.float32)
    o2, l2 = ea.decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), sl.cuda(),
                             out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    o_ref, lse_ref = oracle.decode(q, kc, vc, sl)
    assert np.abs(o2.cpu().double().numpy() - o_ref).max() <= MAX_ABS_O
