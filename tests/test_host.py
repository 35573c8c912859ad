"""CPU tests of the C-ABI library: it loads, exports every symbol the header
declares, rejects bad arguments before touching CUDA, and its host-side
scheduling logic reproduces the worked examples printed in the lecture notes
(tests/golden/scheduling.json, each entry cited)."""
import ctypes
import json
import math
import os
import re

import pytest

import exact_attention_14_gb300 as ea

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = json.load(open(os.path.join(ROOT, "tests", "golden", "scheduling.json")))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_14_gb300 import _build
    _build.build()
    return ea.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_header_symbol(lib):
    names = header_functions()
    assert "attn_fwd" in names and "attn_decode" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in ea.SIGNATURES, f"binding lacks a signature for {n}"


def test_status_strings(lib):
    assert ea.attn_status_string(0) == "ATTN_OK"
    assert ea.attn_status_string(4) == "ATTN_ERR_TIMEOUT"
    assert ea.attn_status_string(99) == "ATTN_ERR_UNKNOWN"


FAKE = 0x10000  # aligned, never dereferenced: every case fails validation first


def fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=2, Hkv=1, Nq=8, Nk=8, d=64,
             causal=0, scale=0.125, odt=0, ws=None, wsb=0)
    a.update(kw)
    return lib.attn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"],
                        a["Nq"], a["Nk"], a["d"], a["causal"], a["scale"], a["odt"], a["ws"],
                        a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(o=None), 1), (dict(k=FAKE + 8), 1), (dict(lse=FAKE + 2), 1),
    (dict(B=0), 1), (dict(Hq=3, Hkv=2), 1), (dict(Nq=0), 1), (dict(Nk=0), 1),
    (dict(Nq=(1 << 24) + 1), 1), (dict(causal=2), 1), (dict(causal=1, Nq=9, Nk=8), 1),
    (dict(scale=-1.0), 1), (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1),
    (dict(odt=7), 1), (dict(d=100), 2), (dict(d=264), 2), (dict(d=4), 2), (dict(d=0), 1),
])
def test_fwd_argument_checks(lib, kw, code):
    assert fwd(lib, **kw) == code


def dec(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, sl=FAKE, o=FAKE, lse=None, B=2, Hq=8, Hkv=2, Nmax=64, d=128,
             scale=0.1, ns=0, ws=FAKE, wsb=1 << 20, odt=1)
    a.update(kw)
    return lib.attn_decode(a["q"], a["k"], a["v"], a["sl"], a["o"], a["lse"], a["B"], a["Hq"],
                           a["Hkv"], a["Nmax"], a["d"], a["scale"], a["ns"], a["ws"], a["wsb"],
                           a["odt"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(sl=None), 1), (dict(sl=FAKE + 2), 1), (dict(v=FAKE + 4), 1),
    (dict(Hq=9), 1), (dict(Nmax=0), 1), (dict(ns=-1), 1), (dict(scale=-0.5), 1),
    (dict(d=84), 2), (dict(d=264), 2), (dict(d=4), 2), (dict(Hq=34, Hkv=2), 2),
])
def test_decode_argument_checks(lib, kw, code):
    assert dec(lib, **kw) == code


def test_workspace_size_rejects_bad_shapes(lib):
    assert ea.attn_decode_workspace_size(0, 8, 2, 64, 128) == 0
    assert ea.attn_decode_workspace_size(1, 8, 3, 64, 128) == 0
    assert ea.attn_decode_workspace_size(1, 8, 2, 64, 96) == 0
    for args in [(0, 8, 8, 64, 64, 128, 0), (1, 8, 3, 64, 64, 128, 0), (1, 8, 8, 64, 64, 100, 0),
                 (1, 8, 8, 64, 32, 128, 1), (1, 8, 8, 64, 64, 128, 2), (1, 8, 8, 0, 64, 128, 0)]:
        assert ea.attn_fwd_workspace_size(*args) == 0, args


def test_fwd_workspace_size_without_a_device(lib):
    """The size depends on the device's SM count: with no device to ask, the
    query returns 0 and attn_fwd stops at the device query."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device answers here (the GPU tests check the size)")
    assert ea.attn_fwd_workspace_size(4, 16, 16, 2048, 2048, 128, 0) == 0
    assert fwd(lib, B=4, Hq=16, Hkv=16, Nq=2048, Nk=2048, d=128) == ea.ATTN_ERR_CUDA


# ------------------------------ scheduling pins ------------------------------
def test_lpt_toy_from_the_notes(lib):
    g = GOLDEN["lpt_toy"]
    mk, loads = ea.attn_list_schedule(g["costs"], g["workers"], lpt=False)
    assert loads == g["natural_loads"] and mk == max(g["natural_loads"])
    mk, loads = ea.attn_list_schedule(g["costs"], g["workers"], lpt=True)
    assert loads == g["lpt_loads"] and mk == g["lower_bound"]


def test_exercise_10_from_the_notes(lib):
    g = GOLDEN["exercise_10"]
    assert ea.attn_list_schedule(g["costs"], g["workers"], lpt=False)[0] == g["natural_makespan"]
    assert ea.attn_list_schedule(g["costs"], g["workers"], lpt=True)[0] == g["lpt_makespan"]
    assert math.ceil(sum(g["costs"]) / g["workers"]) == g["lower_bound"]


def test_split_heuristic_from_the_notes(lib):
    for c in GOLDEN["split_heuristic"]["cases"]:
        s = ea.attn_decode_num_splits(c["units"], c["num_sms"], 128)
        assert s == c["splits"]
        w = c["units"] * s / c["num_sms"]
        assert abs(w / math.ceil(w) - c["efficiency"]) < 0.005


def test_split_heuristic_bad_args(lib):
    assert ea.attn_decode_num_splits(0, 132, 8) == 0
    assert ea.attn_decode_num_splits(4, 0, 8) == 0


def test_causal_block_count_from_the_notes(lib):
    g = GOLDEN["causal_blocks"]
    nb = g["N"] // g["block"]
    full = sum(ea.attn_kv_tiles(i * g["block"], g["block"], g["N"], g["N"], False, g["block"])
               for i in range(nb))
    causal = sum(ea.attn_kv_tiles(i * g["block"], g["block"], g["N"], g["N"], True, g["block"])
                 for i in range(nb))
    assert full == g["blocks_total"] and causal == g["blocks_causal"]
    per_block = 4 * g["block"] * g["block"] * g["d"]  # QK^T and PV, 2 flops per MAC
    assert round(full * per_block / 1e6, 1) == g["mflop_full"]
    assert round(causal * per_block / 1e6, 1) == g["mflop_causal"]


def test_kv_tiles_edge_cases(lib):
    assert ea.attn_kv_tiles(0, 0, 10, 10, True, 128) == 0          # no rows
    assert ea.attn_kv_tiles(0, 1, 1, 1, True, 128) == 1
    assert ea.attn_kv_tiles(0, 128, 128, 300, False, 128) == 3     # ragged Nk
    # bottom-right causal with Nq < Nk: row 0 sees keys 0..Nk-Nq
    assert ea.attn_kv_tiles(0, 1, 100, 300, True, 128) == 2
    assert ea.attn_kv_tiles(0, 128, 128, 128, True, 128) == 1


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [
    (4, 16, 16, 2048, 128, True), (4, 16, 16, 2048, 128, False), (1, 32, 32, 16384, 128, True),
    (8, 32, 8, 4096, 128, True), (1, 3, 1, 300, 64, True), (2, 4, 2, 129, 64, False),
])
@pytest.mark.parametrize("sms", [0, 152])
def test_forward_schedule_covers_every_unit_once(lib, B, Hq, Hkv, N, d, causal, sms):
    order, costs = ea.attn_fwd_schedule(B, Hq, Hkv, N, N, d, causal, num_sms=sms)
    nmb = -(-N // 256)
    assert len(order) == B * Hq * nmb == ea.attn_fwd_num_units(B, Hq, Hkv, N, N, d, causal)
    assert sorted(order) == sorted((b, h, m) for b in range(B) for h in range(Hq)
                                   for m in range(nmb))
    # cost = KV tiles of the unit's two Q tiles; totals match the causal count
    total = sum(costs)
    nt = -(-N // 128)
    if causal:
        assert total == sum(ea.attn_kv_tiles(i * 128, min(128, N - i * 128), N, N, True, 128)
                            for i in range(nt)) * B * Hq
    else:
        assert total == nt * nt * B * Hq


def test_forward_schedule_is_longest_first_within_sections(lib):
    # long-context shape: 8 KB... K/V per head = 8 MiB, so 8 heads per section
    B, Hq, Hkv, N, d = 1, 32, 32, 16384, 128
    order, costs = ea.attn_fwd_schedule(B, Hq, Hkv, N, N, d, True)
    per_sec = 8 * (N // 256)
    for s in range(0, len(order), per_sec):
        sec = costs[s:s + per_sec]
        assert sec == sorted(sec, reverse=True)
        heads = {h for _, h, _ in order[s:s + per_sec]}
        assert len(heads) == 8


def test_dense_schedule_uses_narrow_sections(lib):
    # non-causal prefill: K/V per head = 1 MiB, 16 MiB sections -> 16 heads each,
    # walked m-block rank by rank (all units cost the same)
    B, Hq, Hkv, N, d = 4, 16, 16, 2048, 128
    order, costs = ea.attn_fwd_schedule(B, Hq, Hkv, N, N, d, False)
    per_sec = 16 * (N // 256)
    assert len(set(costs)) == 1
    for s in range(0, len(order), per_sec):
        chunk = order[s:s + per_sec]
        assert len({(b, h) for b, h, _ in chunk}) == 16
        assert [m for _, _, m in chunk] == sorted(m for _, _, m in chunk)


@pytest.mark.parametrize("shape,causal,sms,expect", [
    ((4, 16, 16, 2048, 2048, 128), False, 152, (456, 56, 2)),   # prefill: 512 units
    ((4, 16, 16, 2048, 2048, 128), True, 152, (512, 0, 1)),     # causal: never split
    ((3, 19, 19, 2048, 2048, 128), False, 152, (456, 0, 1)),    # 3 full rounds
    ((1, 8, 8, 2048, 2048, 128), False, 152, (0, 64, 2)),       # 64 units, 152 SMs
    ((1, 2, 2, 4096, 4096, 64), False, 152, (0, 32, 4)),        # 32 units: 4 pieces
    ((1, 1, 1, 256, 128, 64), False, 152, (1, 0, 1)),           # 1 KV tile: cannot split
    ((1, 1, 1, 256, 256, 64), False, 152, (0, 1, 2)),
    ((1, 1, 1, 256, 100000, 64), False, 152, (0, 1, 8)),        # at most 8 pieces
    ((2, 100, 100, 256, 2048, 128), False, 152, (152, 48, 3)),
])
def test_tail_split_plan(lib, shape, causal, sms, expect):
    assert ea.attn_fwd_split_plan(*shape, causal, sms) == expect


def _split_items(shape, causal, sms):
    """(cost in (Q tile, KV tile) pairs) of every work item in queue order."""
    B, Hq, Hkv, Nq, Nk, d = shape
    order, costs = ea.attn_fwd_schedule(B, Hq, Hkv, Nq, Nk, d, causal)
    n_full, n_split, parts = ea.attn_fwd_split_plan(*shape, causal, sms)
    items = list(costs[:n_full])
    for u in range(n_full, n_full + n_split):
        n = -(-Nk // 128)
        tiles = 2 if Nq - order[u][2] * 256 > 128 else 1
        bounds = [p * n // parts for p in range(parts + 1)]
        assert bounds[0] == 0 and bounds[-1] == n and all(b1 > b0 for b0, b1 in zip(bounds, bounds[1:]))
        items += [tiles * (b1 - b0) for b0, b1 in zip(bounds, bounds[1:])]
    return costs, items


@pytest.mark.parametrize("B,H,N", [(4, 16, 2048), (1, 8, 2048), (2, 12, 3000), (5, 7, 1500),
                                   (1, 40, 8192), (8, 16, 1024)])
def test_tail_split_never_lengthens_the_modelled_makespan(lib, B, H, N):
    shape = (B, H, H, N, N, 128)
    costs, items = _split_items(shape, False, 152)
    assert sum(items) == sum(costs)  # the pieces cover every unit's KV tiles once
    whole = ea.attn_list_schedule(costs, 152, lpt=False)[0]
    split = ea.attn_list_schedule(items, 152, lpt=False)[0]
    assert split <= whole
    if (B, H, N) == (4, 16, 2048):
        assert (whole, split) == (4 * 32, 3 * 32 + 16)


def _section_order(B, Hq, Hkv, N, hps, causal):
    """The unit list for sections of hps query heads: sections in order; in a
    section, m-block ranks longest-first (causal), heads in index order."""
    nmb = -(-N // 256)
    order = []
    for h0 in range(0, B * Hq, hps):
        heads = range(h0, min(h0 + hps, B * Hq))
        for rank in range(nmb):
            mb = nmb - 1 - rank if causal else rank
            order += [(bh // Hq, bh % Hq, mb) for bh in heads]
    return order


@pytest.mark.parametrize("B,Hq,Hkv,N", [(4, 16, 16, 2048), (1, 32, 32, 16384), (8, 32, 8, 4096),
                                        (3, 19, 19, 2048), (1, 16, 16, 8192), (8, 8, 8, 1024)])
def test_causal_section_width_minimises_the_modelled_makespan(lib, B, Hq, Hkv, N):
    """With the SM count given, a causal launch takes the narrowest candidate
    section width (8..128 MiB of K/V) whose greedy-list makespan, each unit
    costing the KV steps of its longer Q tile plus 2, is within 1 % of the
    best candidate's (lecture notes 4.5).  The lists are rebuilt here."""
    d, sms = 128, 152
    kv_head = 2 * N * d * 2
    nt = -(-N // 128)

    def steps(order):
        return [max(min(2 * m + 1, nt), min(2 * m + 2, nt)) + 2 for _, _, m in order]

    cands = []
    for mib in (8, 16, 32, 64, 128):
        hps = min(max(1, (mib << 20) // kv_head) * (Hq // Hkv), B * Hq)
        if cands and cands[-1][0] == hps:
            continue
        order = _section_order(B, Hq, Hkv, N, hps, True)
        cands.append((hps, order, ea.attn_list_schedule(steps(order), sms, lpt=False)[0]))
    best = min(c[2] for c in cands)
    want = next(c for c in cands if c[2] <= best * 1.01)
    got, _ = ea.attn_fwd_schedule(B, Hq, Hkv, N, N, d, True, num_sms=sms)
    assert got == want[1], [(c[0], c[2]) for c in cands]
    if (B, Hq, N) == (4, 16, 2048):
        assert want[0] == 16          # prefill: 16 MiB sections (64 MiB models no better)
    # without an SM count the fixed 64 MiB width stays
    fixed, _ = ea.attn_fwd_schedule(B, Hq, Hkv, N, N, d, True)
    hps64 = min(max(1, (64 << 20) // kv_head) * (Hq // Hkv), B * Hq)
    assert fixed == _section_order(B, Hq, Hkv, N, hps64, True)


def test_gqa_siblings_are_adjacent(lib):
    order, _ = ea.attn_fwd_schedule(2, 8, 2, 512, 512, 64, True)
    # consecutive units of one m-block rank share a KV head in groups of 4
    for i in range(0, len(order), 4):
        kv = {(b, h // 4) for b, h, _ in order[i:i + 4]}
        assert len(kv) == 1


def test_wave_quantisation_model_from_the_notes():
    for c in GOLDEN["wave_quantisation"]["cases"]:
        waves = math.ceil(c["blocks"] / c["num_sms"])
        assert waves == c["waves"]
        assert abs(c["blocks"] / (waves * c["num_sms"]) - c["utilisation"]) < 0.005


def test_tau_bound_from_the_notes():
    g = GOLDEN["tau_bound"]
    bound = 128 - math.log2(g["N"])
    assert bound == g["tau_max_exclusive"] and g["tau_used"] < bound


def test_bwd_workspace_size_and_argument_checks(lib):
    # two fp32 row vectors (D, lse2) over rows padded to 128
    assert ea.attn_bwd_workspace_size(2, 8, 2, 300, 300, 128) == 8 * 2 * 8 * 384
    assert ea.attn_bwd_workspace_size(1, 4, 3, 128, 128, 64) == 0      # Hq % Hkv
    assert ea.attn_bwd_workspace_size(1, 4, 4, 128, 128, 100) == 0     # unsupported d
    assert ea.attn_bwd_workspace_size(1, 4, 4, 128, 128, 96) > 0       # padded to 128
    fake = ctypes.c_void_p(0x10000)
    args = [fake] * 9 + [1, 2, 2, 128, 128, 128, 0, ctypes.c_float(0.1), 0, 0, fake, 1 << 30, None]
    bad = list(args)
    bad[4] = None                                                      # no dout
    assert lib.attn_bwd(*bad) == ea.ATTN_ERR_INVALID_ARG
    bad = list(args)
    bad[20] = 16                                                       # workspace too small
    assert lib.attn_bwd(*bad) == ea.ATTN_ERR_WORKSPACE
    bad = list(args)
    bad[14] = 100                                                      # d (not a multiple of 8)
    assert lib.attn_bwd(*bad) == ea.ATTN_ERR_UNSUPPORTED
    bad = list(args)
    bad[15] = 1
    bad[12], bad[13] = 256, 128                                        # causal with Nq > Nk
    assert lib.attn_bwd(*bad) == ea.ATTN_ERR_INVALID_ARG


def test_decode_paged_argument_checks(lib):
    fake = ctypes.c_void_p(0x10000)
    args = [fake] * 7 + [2, 8, 2, 100, 64, 16, 128, ctypes.c_float(0.1), 0, fake, 1 << 30, 0, None]
    bad = list(args)
    bad[3] = None                                                      # no block table
    assert lib.attn_decode_paged(*bad) == ea.ATTN_ERR_INVALID_ARG
    bad = list(args)
    bad[11] = 96                                                       # page size not a multiple of 64
    assert lib.attn_decode_paged(*bad) == ea.ATTN_ERR_UNSUPPORTED
    bad = list(args)
    bad[11] = 32                                                       # page size below 64
    assert lib.attn_decode_paged(*bad) == ea.ATTN_ERR_INVALID_ARG
    bad = list(args)
    bad[10] = 0                                                        # no blocks
    assert lib.attn_decode_paged(*bad) == ea.ATTN_ERR_INVALID_ARG
    bad = list(args)
    bad[13] = 264                                                      # d above 256
    assert lib.attn_decode_paged(*bad) == ea.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("d,fwd_ok,bwd_ok", [
    (8, True, True), (32, True, True), (48, True, True), (80, True, True), (96, True, True),
    (120, True, True), (128, True, True), (4, False, False), (100, False, False),
    (130, False, False), (136, True, True), (192, True, True), (200, True, True),
    (256, True, True), (264, False, False)])
def test_supported_head_dims(lib, d, fwd_ok, bwd_ok):
    """The forward, the backward (workspace size 0 when unsupported) and decode
    take d in [8, 256] (multiples of 8): up to 128 on the 64- or 128-column
    kernels, above on the wider ones (zero-filled columns)."""
    import torch
    assert (ea.attn_bwd_workspace_size(2, 8, 2, 1000, 1000, d) > 0) == bwd_ok
    # decode takes the forward's head dims (its size query needs a device)
    if not torch.cuda.is_available():
        rc = lib.attn_decode(FAKE, FAKE, FAKE, FAKE, FAKE, None, 2, 8, 2, 64, d, 0.1, 0, FAKE,
                             1 << 20, 1, None)
        assert rc == (ea.ATTN_ERR_CUDA if fwd_ok else ea.ATTN_ERR_UNSUPPORTED)
    # FAKE is not device memory: a call whose arguments pass every check is
    # made only where no device can run it (it then stops at the device query)
    if not fwd_ok:
        assert fwd(lib, d=d) == ea.ATTN_ERR_UNSUPPORTED
    elif not torch.cuda.is_available():
        assert fwd(lib, d=d) == ea.ATTN_ERR_CUDA
    if not bwd_ok:
        bwd_rc = lib.attn_bwd(*([FAKE] * 9), 1, 2, 1, 8, 8, d, 0, 0.125, 0, 0, FAKE, 1 << 30, None)
        assert bwd_rc == ea.ATTN_ERR_UNSUPPORTED


def fwd_varlen(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, cq=FAKE, ck=FAKE, B=2, Hq=2, Hkv=1,
             tq=300, tk=300, mq=200, mk=200, d=128, causal=1, scale=0.1, odt=1)
    a.update(kw)
    return lib.attn_fwd_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cq"], a["ck"],
                               a["B"], a["Hq"], a["Hkv"], a["tq"], a["tk"], a["mq"], a["mk"],
                               a["d"], a["causal"], a["scale"], a["odt"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(cq=None), 1), (dict(ck=FAKE + 2), 1), (dict(o=FAKE + 4), 1),
    (dict(tq=0), 1), (dict(tk=0), 1), (dict(tq=(1 << 30) + 1), 1), (dict(mq=301), 1),
    (dict(mk=301), 1), (dict(mq=0), 1), (dict(B=0), 1), (dict(Hq=3, Hkv=2), 1),
    (dict(causal=2), 1), (dict(scale=-1.0), 1), (dict(odt=5), 1), (dict(d=100), 2),
    (dict(d=264), 2), (dict(d=252), 2),
])
def test_fwd_varlen_argument_checks(lib, kw, code):
    assert fwd_varlen(lib, **kw) == code


def bwd_varlen(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             cq=FAKE, ck=FAKE, B=2, Hq=2, Hkv=1, tq=300, tk=300, mq=200, mk=200, d=128, causal=1,
             scale=0.1, odt=1, gdt=1, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    return lib.attn_bwd_varlen(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"],
                               a["dv"], a["cq"], a["ck"], a["B"], a["Hq"], a["Hkv"], a["tq"], a["tk"],
                               a["mq"], a["mk"], a["d"], a["causal"], a["scale"], a["odt"], a["gdt"],
                               a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(do=None), 1), (dict(lse=None), 1), (dict(dq=None), 1),
    (dict(cq=None), 1), (dict(ck=FAKE + 2), 1), (dict(dk=FAKE + 4), 1), (dict(tq=0), 1),
    (dict(mq=301), 1), (dict(B=0), 1), (dict(Hq=3, Hkv=2), 1), (dict(causal=2), 1),
    (dict(gdt=7), 1), (dict(d=100), 2), (dict(d=264), 2), (dict(d=252), 2),
    (dict(ws=None), 5), (dict(wsb=16), 5), (dict(ws=FAKE + 4), 5),
])
def test_bwd_varlen_argument_checks(lib, kw, code):
    """Every rejection happens on the host, before a device is touched."""
    assert bwd_varlen(lib, **kw) == code


def test_bwd_varlen_workspace_size():
    # 2 vectors x Hq x (total_q + 132 B, rounded up to 4) floats
    assert ea.attn_bwd_varlen_workspace_size(3, 4, 2, 1000, 128) == 2 * 4 * ((1000 + 396 + 3) // 4 * 4) * 4
    assert ea.attn_bwd_varlen_workspace_size(3, 4, 2, 1000, 256) == 2 * 4 * ((1000 + 396 + 3) // 4 * 4) * 4
    assert ea.attn_bwd_varlen_workspace_size(3, 4, 2, 1000, 264) == 0   # d > 256: not supported
    assert ea.attn_bwd_varlen_workspace_size(3, 4, 3, 1000, 128) == 0   # Hq % Hkv
    assert ea.attn_bwd_varlen_workspace_size(0, 4, 2, 1000, 128) == 0


def test_fp8_sizes_and_argument_checks(lib):
    assert ea.attn_fp8_codes_bytes(2, 3, 300, 128) == 2 * 3 * 300 * 128
    assert ea.attn_fp8_codes_bytes(2, 3, 300, 128, transpose=True) == 2 * 3 * 128 * 304
    assert ea.attn_fp8_codes_bytes(1, 1, 10, 64) == 0
    assert ea.attn_fp8_descale_count(2, 3, 300) == 18
    q = lib.attn_fp8_quantize
    assert q(None, FAKE, FAKE, None, 1, 1, 8, 128, 0, None) == 1
    assert q(FAKE, FAKE + 8, FAKE, None, 1, 1, 8, 128, 0, None) == 1
    assert q(FAKE, FAKE, FAKE + 2, None, 1, 1, 8, 128, 0, None) == 1
    assert q(FAKE, FAKE, FAKE, None, 1, 1, 0, 128, 0, None) == 1
    assert q(FAKE, FAKE, FAKE, None, 1, 1, 8, 128, 2, None) == 1
    assert q(FAKE, FAKE, FAKE, None, 1, 1, 8, 64, 0, None) == 2
    f = lib.attn_fwd_fp8
    args = [FAKE] * 6 + [FAKE, None, 1, 2, 1, 8, 8, 128, 0, 0.1, 0, 0, None]
    bad_d = list(args); bad_d[13] = 64
    assert f(*bad_d) == 2
    bad_s = list(args); bad_s[3] = None
    assert f(*bad_s) == 1
    bad_c = list(args); bad_c[14] = 1; bad_c[11] = 9
    assert f(*bad_c) == 1
    bad_r = list(args); bad_r[16] = 2       # rotated is 0 or 1
    assert f(*bad_r) == 1


def test_no_test_function_defined_twice():
    """A second definition of a test function would silently replace the first
    (and its parametrised cases) when pytest collects the module."""
    import ast
    import glob
    for path in glob.glob(os.path.join(ROOT, "tests", "test_*.py")):
        tree = ast.parse(open(path).read())
        names = [n.name for n in tree.body if isinstance(n, ast.FunctionDef) and n.name.startswith("test_")]
        dup = {n for n in names if names.count(n) > 1}
        assert not dup, f"{os.path.basename(path)} defines {sorted(dup)} more than once"


def test_operands_must_share_one_device():
    """The binding makes the operands' device current for each call and
    refuses operands spread over devices (checked here with host and meta
    tensors, no GPU needed)."""
    import torch
    a, b = torch.empty(2), torch.empty(2)
    assert ea._one_device(a, None, b) == a.device
    with pytest.raises(ValueError, match="different devices"):
        ea._one_device(a, torch.empty(2, device="meta"))


@pytest.mark.parametrize("fn", ["attn_decode", "attn_decode_noalloc"])
def test_decode_binding_checks_shapes_before_the_library(fn):
    """The decode wrappers reject wrong types and shapes (an o, lse, cache or
    length vector the kernels would index out of bounds) before any pointer
    reaches the library; host tensors are refused as well."""
    import torch
    call = getattr(ea, fn)
    B, Hq, Hkv, N, d = 2, 8, 2, 64, 128
    q = torch.zeros(B, Hq, 1, d, dtype=torch.bfloat16)
    kc = torch.zeros(B, Hkv, N, d, dtype=torch.bfloat16)
    sl = torch.full((B,), N, dtype=torch.int32)
    o = torch.zeros(B, Hq, 1, d, dtype=torch.float32)
    lse = torch.zeros(B, Hq, 1, dtype=torch.float32)
    bad = [
        (dict(o=torch.zeros(B, Hq - 1, 1, d)), ValueError),
        (dict(o=torch.zeros(B, Hq, 1, d, dtype=torch.float64)), TypeError),
        (dict(o=torch.zeros(B, Hq, 1, d, dtype=torch.float16)), TypeError),
        (dict(lse=torch.zeros(B, Hq - 2, 1)), ValueError),
        (dict(lse=torch.zeros(B, Hq, 1, dtype=torch.float64)), TypeError),
        (dict(v_cache=torch.zeros(B, Hkv, N - 1, d, dtype=torch.bfloat16)), ValueError),
        (dict(k_cache=torch.zeros(B, Hkv, N, d, dtype=torch.float32)), TypeError),
        (dict(seqlens=torch.zeros(B + 1, dtype=torch.int32)), ValueError),
        (dict(seqlens=torch.zeros(B, dtype=torch.int64)), TypeError),
        (dict(q=torch.zeros(B, Hq, 2, d, dtype=torch.bfloat16)), ValueError),
        (dict(), ValueError),   # all well formed, but host tensors: "must be a CUDA tensor"
    ]
    for kw, exc in bad:
        a = dict(q=q, k_cache=kc, v_cache=kc.clone(), seqlens=sl, o=o, lse=lse)
        a.update(kw)
        with pytest.raises(exc, match="CUDA" if not kw else "tensor|mismatch|4-D"):
            call(a["q"], a["k_cache"], a["v_cache"], a["seqlens"], a["o"], a["lse"])


def test_decode_paged_binding_checks_output_shapes():
    import torch
    B, Hq, Hkv, d = 2, 8, 2, 128
    q = torch.zeros(B, Hq, 1, d, dtype=torch.bfloat16)
    pages = torch.zeros(4, 64, Hkv, d, dtype=torch.bfloat16)
    bt = torch.zeros(B, 2, dtype=torch.int32)
    sl = torch.full((B,), 128, dtype=torch.int32)
    with pytest.raises(ValueError, match="o shape"):
        ea.attn_decode_paged(q, pages, pages, bt, sl, torch.zeros(B, Hq, 1, d - 8),
                             torch.zeros(B, Hq, 1))
    with pytest.raises(ValueError, match="lse shape"):
        ea.attn_decode_paged(q, pages, pages, bt, sl, torch.zeros(B, Hq, 1, d),
                             torch.zeros(B, Hq))
    with pytest.raises(ValueError, match="CUDA"):
        ea.attn_decode_paged(q, pages, pages, bt, sl, torch.zeros(B, Hq, 1, d),
                             torch.zeros(B, Hq, 1))
