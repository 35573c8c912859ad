"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows);
this module only compiles it with gcc and marshals numpy arrays through ctypes.
See the header of ``attn_oracle.c`` for the definition it follows and the
readings it takes where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc (-O2 -fopenmp); return its path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            u16 = ctypes.POINTER(ctypes.c_uint16)
            i32 = ctypes.POINTER(ctypes.c_int32)
            lib.oracle_attention_rows.argtypes = [
                u16, u16, u16, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, i32, ctypes.c_int, ctypes.c_int, ctypes.c_long,
                i32, dp, dp, ctypes.c_int]
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_attention.argtypes = [
                u16, u16, u16, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, i32, ctypes.c_int, ctypes.c_int, dp, dp,
                ctypes.c_int]
            lib.oracle_attention.restype = ctypes.c_int
            lib.oracle_lse_merge.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp,
                                             dp, dp]
            lib.oracle_lse_merge.restype = None
            lib.oracle_attention_bwd.argtypes = [
                u16, u16, u16, u16, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                dp, dp, dp, ctypes.c_int]
            lib.oracle_attention_bwd.restype = ctypes.c_int
            _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    """bf16 data as a contiguous uint16 numpy array of its bit patterns."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            if a.dtype != torch.bfloat16:
                raise TypeError("oracle inputs must be bfloat16 tensors")
            return np.ascontiguousarray(
                a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs must be bf16 bit patterns (uint16)")
    return np.ascontiguousarray(a)


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if Bk != B or dk != d or tuple(v.shape) != tuple(k.shape):
        raise ValueError("inconsistent q/k/v shapes")
    return B, Hq, Hkv, Nq, Nk, d


def attention(q, k, v, *, causal: bool = False, scale: float | None = None,
              kv_len=None, window=(0, 0), n_threads: int = 0):
    """Full attention in fp64.  Returns (O [B,Hq,Nq,d] float64, LSE [B,Hq,Nq] float64)."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hq, Hkv, Nq, Nk, d = _shapes(qb, kb, vb)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.empty((B, Hq, Nq, d), np.float64)
    lse = np.empty((B, Hq, Nq), np.float64)
    kl = None if kv_len is None else np.ascontiguousarray(np.asarray(kv_len, np.int32))
    rc = _load().oracle_attention(
        _ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
        B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale),
        None if kl is None else _ptr(kl, ctypes.c_int32),
        int(window[0]), int(window[1]), _ptr(o, ctypes.c_double),
        _ptr(lse, ctypes.c_double), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return o, lse


def attention_rows(q, k, v, rows, *, causal: bool = False, scale: float | None = None,
                   kv_len=None, window=(0, 0), n_threads: int = 0):
    """Selected rows only.  rows: int array [n, 3] of (b, hq, i).

    Returns (O [n, d] float64, LSE [n] float64)."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hq, Hkv, Nq, Nk, d = _shapes(qb, kb, vb)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.ascontiguousarray(np.asarray(rows, np.int32).reshape(-1, 3))
    n = rows.shape[0]
    o = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    kl = None if kv_len is None else np.ascontiguousarray(np.asarray(kv_len, np.int32))
    rc = _load().oracle_attention_rows(
        _ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
        B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale),
        None if kl is None else _ptr(kl, ctypes.c_int32),
        int(window[0]), int(window[1]), n, _ptr(rows, ctypes.c_int32),
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_attention_rows rejected its arguments")
    return o, lse


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, *, causal: bool = False,
                     scale: float | None = None, n_threads: int = 0):
    """Packed batch of independent sequences: sequence b is query rows
    cu_q[b]..cu_q[b+1] of q [total_q, Hq, d] and key rows cu_k[b]..cu_k[b+1]
    of k, v [total_k, Hkv, d]; it is its own attention problem (causal
    bottom-right aligned within it), computed by attention() above.

    Returns (O [total_q, Hq, d], LSE [Hq, total_q]) float64; rows that belong
    to no sequence are NaN."""
    cu_q = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    total_q, Hq, d = q.shape
    o = np.full((total_q, Hq, d), np.nan)
    lse = np.full((Hq, total_q), np.nan)
    for b in range(len(cu_q) - 1):
        qs, qe, ks, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if qe == qs:
            continue
        qb = q[qs:qe].permute(1, 0, 2).unsqueeze(0)
        kb = k[ks:ke].permute(1, 0, 2).unsqueeze(0)
        vb = v[ks:ke].permute(1, 0, 2).unsqueeze(0)
        ob, lb = attention(qb, kb, vb, causal=causal, scale=scale, n_threads=n_threads)
        o[qs:qe] = ob[0].transpose(1, 0, 2)
        lse[:, qs:qe] = lb[0]
    return o, lse


def attention_bwd_varlen(q, k, v, dout, cu_seqlens_q, cu_seqlens_k, *, causal: bool = False,
                         scale: float | None = None, n_threads: int = 0):
    """Gradients for a packed batch (layouts as attention_varlen, dout shaped
    like q): each sequence is its own problem, so its gradients are
    attention_bwd() of its rows; key rows of a sequence without queries get
    zero dK and dV.  Returns (dQ, dK, dV) float64 shaped like q, k, v; rows
    that belong to no sequence are NaN."""
    cu_q = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    dq = np.full(tuple(q.shape), np.nan)
    dk = np.full(tuple(k.shape), np.nan)
    dv = np.full(tuple(v.shape), np.nan)
    for b in range(len(cu_q) - 1):
        qs, qe, ks, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if qe == qs:
            dk[ks:ke] = 0.0
            dv[ks:ke] = 0.0
            continue
        seq = lambda t, s0, s1: t[s0:s1].permute(1, 0, 2).unsqueeze(0)  # noqa: E731
        gq, gk, gv = attention_bwd(seq(q, qs, qe), seq(k, ks, ke), seq(v, ks, ke),
                                   seq(dout, qs, qe), causal=causal, scale=scale,
                                   n_threads=n_threads)
        dq[qs:qe] = gq[0].transpose(1, 0, 2)
        dk[ks:ke] = gk[0].transpose(1, 0, 2)
        dv[ks:ke] = gv[0].transpose(1, 0, 2)
    return dq, dk, dv


def decode(q, k_cache, v_cache, seqlens, *, scale: float | None = None,
           n_threads: int = 0):
    """Single-query decode over the valid prefix of each sequence's KV cache.

    q: [B, Hq, 1, d]; caches: [B, Hkv, Nmax, d]; seqlens: [B].
    Returns (O [B, Hq, 1, d], LSE [B, Hq, 1])."""
    return attention(q, k_cache, v_cache, causal=False, scale=scale,
                     kv_len=seqlens, n_threads=n_threads)


def lse_merge(lse_parts, o_parts):
    """Merge partial (LSE_s, O_s) of disjoint key sets.  Returns (LSE, O[d])."""
    lse_parts = np.ascontiguousarray(np.asarray(lse_parts, np.float64).reshape(-1))
    o_parts = np.ascontiguousarray(np.asarray(o_parts, np.float64))
    n = lse_parts.shape[0]
    d = o_parts.shape[-1]
    o_parts = o_parts.reshape(n, d)
    lse = np.empty((1,), np.float64)
    o = np.empty((d,), np.float64)
    _load().oracle_lse_merge(n, d, _ptr(lse_parts, ctypes.c_double),
                             _ptr(o_parts, ctypes.c_double),
                             _ptr(lse, ctypes.c_double), _ptr(o, ctypes.c_double))
    return float(lse[0]), o


def attention_bwd(q, k, v, dout, *, causal: bool = False, scale: float | None = None,
                  n_threads: int = 0):
    """Gradients of O = attention(q, k, v) for the upstream gradient dout
    (bf16, shaped like q), in fp64.  Returns (dQ, dK, dV) as float64 arrays
    shaped like q, k, v."""
    qb, kb, vb, ob = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, Hq, Hkv, Nq, Nk, d = _shapes(qb, kb, vb)
    if tuple(ob.shape) != tuple(qb.shape):
        raise ValueError("dout must be shaped like q")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.empty(qb.shape, np.float64)
    dk = np.empty(kb.shape, np.float64)
    dv = np.empty(vb.shape, np.float64)
    rc = _load().oracle_attention_bwd(
        _ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16), _ptr(vb, ctypes.c_uint16),
        _ptr(ob, ctypes.c_uint16), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale),
        _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double),
        int(n_threads))
    if rc != 0:
        raise ValueError("oracle_attention_bwd rejected its arguments")
    return dq, dk, dv
