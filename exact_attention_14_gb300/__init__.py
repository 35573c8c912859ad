"""GB300 (sm_103a) exact attention: fused forward (dense and packed
variable-length), backward, and split-KV decode (contiguous or paged cache).

Thin ctypes binding over the C ABI in ``include/attn.h`` (library
``libgb300_attn.so`` built in-tree by ``_build.build()``).  The functions here
only marshal arguments -- shapes, data pointers and the CUDA stream -- and turn
status codes into exceptions; every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.

There is no fallback: if the library is missing or was not built for this GPU,
the first call raises.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "ATTN_OUT_BF16", "ATTN_OUT_F32", "AttnError", "attn_fwd", "attn_fwd_workspace_size",
    "attn_fwd_varlen", "forward_varlen",
    "attn_fp8_quantize", "fp8_quantize", "attn_fwd_fp8", "forward_fp8", "attn_fp8_codes_bytes",
    "attn_fp8_descale_count",
    "attn_decode",
    "attn_decode_workspace_size", "attn_decode_noalloc", "attn_status_string", "attn_last_device_error",
    "attn_decode_num_splits", "attn_list_schedule", "attn_kv_tiles",
    "attn_fwd_num_units", "attn_fwd_schedule", "attn_fwd_split_plan", "attn_decode_kernel_launches",
    "attn_bwd", "attn_bwd_workspace_size", "backward", "attn_bwd_varlen",
    "attn_bwd_varlen_workspace_size", "backward_varlen", "attn_decode_paged", "decode_paged", "forward", "decode", "library_path", "load",
]

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_WORKSPACE = 5
ATTN_OUT_BF16 = 0
ATTN_OUT_F32 = 1

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgb300_attn.so")
_lib = None

# Every symbol the header declares, with its ctypes signature.
_c_int, _c_ll, _c_sz, _c_f, _vp = (ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t,
                                   ctypes.c_float, ctypes.c_void_p)
SIGNATURES = {
    "attn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int,
                          _c_int, _c_int, _c_f, _c_int, _vp, _c_sz, _vp]),
    "attn_fwd_workspace_size": (_c_sz, [_c_int] * 7),
    "attn_fwd_varlen": (_c_int, [_vp] * 7 + [_c_int] * 9 + [_c_f, _c_int, _vp]),
    "attn_fp8_codes_bytes": (_c_sz, [_c_int] * 5),
    "attn_fp8_descale_count": (_c_sz, [_c_int] * 3),
    "attn_fp8_quantize": (_c_int, [_vp] * 4 + [_c_int] * 5 + [_vp]),
    "attn_fwd_fp8": (_c_int, [_vp] * 8 + [_c_int] * 7 + [_c_f, _c_int, _c_int, _vp]),
    "attn_selftest_bounded_wait": (_c_int, [_c_int, _vp, _vp]),
    "attn_decode_workspace_size": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "attn_decode": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                             _c_int, _c_f, _c_int, _vp, _c_sz, _c_int, _vp]),
    "attn_decode_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int,
                                     _c_int, _c_int, _c_f, _c_int, _c_int, _vp]),
    "attn_status_string": (ctypes.c_char_p, [_c_int]),
    "attn_last_device_error": (_c_int, [_vp]),
    "attn_decode_num_splits": (_c_int, [_c_int, _c_int, _c_int]),
    "attn_list_schedule": (_c_ll, [ctypes.POINTER(ctypes.c_int), _c_int, _c_int, _c_int,
                                   ctypes.POINTER(ctypes.c_longlong)]),
    "attn_kv_tiles": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "attn_fwd_num_units": (_c_ll, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int]),
    "attn_fwd_schedule": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                   _c_int, _c_ll, ctypes.POINTER(ctypes.c_int),
                                   ctypes.POINTER(ctypes.c_int)]),
    "attn_decode_kernel_launches": (_c_int, [_c_int] * 6),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [_c_int] * 6),
    "attn_bwd_varlen_workspace_size": (ctypes.c_size_t, [_c_int] * 5),
    "attn_bwd_varlen": (_c_int, [ctypes.c_void_p] * 11 + [_c_int] * 9 + [ctypes.c_float, _c_int, _c_int,
                                                                          ctypes.c_void_p, ctypes.c_size_t,
                                                                          ctypes.c_void_p]),
    "attn_decode_paged": (_c_int, [ctypes.c_void_p] * 7 + [_c_int, _c_int, _c_int, _c_ll, _c_int,
                                                            _c_int, _c_int, ctypes.c_float, _c_int,
                                                            ctypes.c_void_p, ctypes.c_size_t, _c_int,
                                                            ctypes.c_void_p]),
    "attn_bwd": (_c_int, [ctypes.c_void_p] * 9 + [_c_int] * 7 + [ctypes.c_float, _c_int, _c_int,
                                                                 ctypes.c_void_p, ctypes.c_size_t,
                                                                 ctypes.c_void_p]),
    "attn_fwd_split_plan": (_c_int, [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                     _c_int, ctypes.POINTER(ctypes.c_int),
                                     ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
}


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {attn_status_string(code)} ({code})")


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def attn_status_string(code: int) -> str:
    return load().attn_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != ATTN_OK:
        raise AttnError(code, where)


def _stream_ptr(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _workspace(ws):
    """(pointer, bytes) of an optional workspace tensor."""
    if ws is None:
        return None, 0
    _need(ws, ws.dtype, "workspace")
    return _ptr(ws), ws.numel() * ws.element_size()


def _one_device(*tensors):
    """The device of the given tensors (None entries skipped): the library
    launches on the current CUDA device, so every operand must live on one
    device, which the call then makes current."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"operands on different devices: {dev} and {t.device}")
    return dev


def _on(dev):
    import torch
    return torch.cuda.device(dev)


def attn_fwd_workspace_size(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int,
                            causal: bool) -> int:
    """Bytes of workspace attn_fwd needs for this shape on the current device
    (0 when it splits no unit)."""
    return int(load().attn_fwd_workspace_size(B, Hq, Hkv, Nq, Nk, d, int(bool(causal))))


def attn_fwd(q, k, v, o, lse=None, *, causal: bool = False, scale: float | None = None,
             workspace=None, stream=None):
    """Fused forward into caller-provided outputs.

    q [B,Hq,Nq,d] bf16; k, v [B,Hkv,Nk,d] bf16; o [B,Hq,Nq,d] bf16 or fp32;
    lse [B,Hq,Nq] fp32 or None; workspace: a CUDA tensor of at least
    attn_fwd_workspace_size(...) bytes, or None (then one is allocated with
    torch when the shape needs it).  Asynchronous on ``stream`` (default: the
    current torch stream)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be bfloat16 or float32")
    _need(o, o.dtype, "o")
    if lse is not None:
        _need(lse, torch.float32, "lse")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, Hkv, Nk, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k/v shape mismatch")
    if tuple(o.shape) != (B, Hq, Nq, d):
        raise ValueError("o shape mismatch")
    if lse is not None and tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("lse shape mismatch")
    if scale is None:
        scale = d ** -0.5
    odt = ATTN_OUT_F32 if o.dtype == torch.float32 else ATTN_OUT_BF16
    dev = _one_device(q, k, v, o, lse, workspace)
    with _on(dev):
        if workspace is None:
            need = attn_fwd_workspace_size(B, Hq, Hkv, Nq, Nk, d, causal)
            if need > 0:
                workspace = torch.empty(need, dtype=torch.uint8, device=dev)
                if isinstance(stream, torch.cuda.Stream):
                    workspace.record_stream(stream)   # freed only after that stream's use
        ws_ptr, ws_bytes = _workspace(workspace)
        rc = load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                             int(bool(causal)), float(scale), odt, ws_ptr, ws_bytes,
                             _stream_ptr(stream))
    _check(rc, "attn_fwd")
    return o, lse


def attn_fwd_varlen(q, k, v, o, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                    max_seqlen_k: int, lse=None, *, causal: bool = False,
                    scale: float | None = None, stream=None):
    """Packed variable-length forward into caller-provided outputs.

    q [total_q,Hq,d] bf16; k, v [total_k,Hkv,d] bf16; o [total_q,Hq,d] bf16 or
    fp32; cu_seqlens_q / cu_seqlens_k int32 [B+1] on the device (sequence b is
    rows cu[b]..cu[b+1]); lse [Hq,total_q] fp32 or None.  Asynchronous."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, n)
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _need(t, torch.int32, n)
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be bfloat16 or float32")
    _need(o, o.dtype, "o")
    if lse is not None:
        _need(lse, torch.float32, "lse")
    total_q, Hq, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    if tuple(k.shape) != (total_k, Hkv, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k/v shape mismatch")
    if tuple(o.shape) != tuple(q.shape):
        raise ValueError("o shape mismatch")
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1 or B < 1:
        raise ValueError("cu_seqlens_q / cu_seqlens_k must both have B + 1 entries")
    if lse is not None and tuple(lse.shape) != (Hq, total_q):
        raise ValueError("lse shape mismatch")
    if scale is None:
        scale = d ** -0.5
    odt = ATTN_OUT_F32 if o.dtype == torch.float32 else ATTN_OUT_BF16
    with _on(_one_device(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k)):
        rc = load().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                    _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, Hq, Hkv, total_q,
                                    total_k, int(max_seqlen_q), int(max_seqlen_k), d,
                                    int(bool(causal)), float(scale), odt, _stream_ptr(stream))
    _check(rc, "attn_fwd_varlen")
    return o, lse


def forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
                   *, causal: bool = False, scale: float | None = None, out_dtype=None,
                   return_lse: bool = True, stream=None):
    """Allocate O (and LSE [Hq, total_q]) with torch and run attn_fwd_varlen."""
    import torch
    out_dtype = out_dtype or torch.bfloat16
    o = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    lse = (torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
           if return_lse else None)
    return attn_fwd_varlen(q, k, v, o, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k,
                           lse, causal=causal, scale=scale, stream=stream)


def attn_fp8_codes_bytes(B: int, H: int, N: int, d: int, transpose: bool = False) -> int:
    return int(load().attn_fp8_codes_bytes(B, H, N, d, int(bool(transpose))))


def attn_fp8_descale_count(B: int, H: int, N: int) -> int:
    return int(load().attn_fp8_descale_count(B, H, N))


def attn_fp8_quantize(x, codes, descale, signs=None, *, transpose: bool = False, stream=None):
    """Block-quantize x [B,H,N,d] bf16 into caller-provided E4M3 codes (uint8
    [B,H,N,d], or [B,H,d,Np] when transpose) and descale [B,H,ceil(N/128)]
    fp32; signs: None or an int8 tensor of d values +-1 (rotate first)."""
    import torch
    _need(x, torch.bfloat16, "x")
    _need(codes, torch.uint8, "codes")
    _need(descale, torch.float32, "descale")
    if signs is not None:
        _need(signs, torch.int8, "signs")
    B, H, N, d = x.shape
    if signs is not None and signs.numel() != d:
        raise ValueError("signs must hold d values")
    npad = (N + 15) // 16 * 16
    want = (B, H, d, npad) if transpose else (B, H, N, d)
    if tuple(codes.shape) != want:
        raise ValueError(f"codes must be {want}")
    if tuple(descale.shape) != (B, H, (N + 127) // 128):
        raise ValueError("descale shape mismatch")
    with _on(_one_device(x, codes, descale, signs)):
        rc = load().attn_fp8_quantize(_ptr(x), _ptr(codes), _ptr(descale), _ptr(signs), B, H, N, d,
                                      int(bool(transpose)), _stream_ptr(stream))
    _check(rc, "attn_fp8_quantize")
    return codes, descale


def fp8_quantize(x, signs=None, *, transpose: bool = False, stream=None):
    """Allocate the codes and scales with torch and run attn_fp8_quantize."""
    import torch
    B, H, N, d = x.shape
    npad = (N + 15) // 16 * 16
    shape = (B, H, d, npad) if transpose else (B, H, N, d)
    codes = (torch.zeros if transpose else torch.empty)(shape, dtype=torch.uint8, device=x.device)
    descale = torch.empty((B, H, (N + 127) // 128), dtype=torch.float32, device=x.device)
    return attn_fp8_quantize(x, codes, descale, signs, transpose=transpose, stream=stream)


def attn_fwd_fp8(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse=None, *,
                 causal: bool = False, scale: float | None = None, rotated: bool = False,
                 stream=None):
    """Forward on E4M3 operands into caller-provided outputs: q8 [B,Hq,Nq,128],
    k8 [B,Hkv,Nk,128], vt8 [B,Hkv,128,Np] (uint8 codes), descales fp32
    [B,H,ceil(N/128)]; o [B,Hq,Nq,128] bf16/fp32; lse [B,Hq,Nq] or None.
    scale is the original problem's softmax scale; rotated: Q and K were
    quantized with the same Hadamard signs (the library then divides the
    scale by d)."""
    import torch
    for t, n in ((q8, "q8"), (k8, "k8"), (vt8, "vt8")):
        _need(t, torch.uint8, n)
    for t, n in ((q_descale, "q_descale"), (k_descale, "k_descale"), (v_descale, "v_descale")):
        _need(t, torch.float32, n)
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be bfloat16 or float32")
    _need(o, o.dtype, "o")
    if lse is not None:
        _need(lse, torch.float32, "lse")
    B, Hq, Nq, d = q8.shape
    Hkv, Nk = k8.shape[1], k8.shape[2]
    if tuple(k8.shape) != (B, Hkv, Nk, d) or tuple(vt8.shape) != (B, Hkv, d, (Nk + 15) // 16 * 16):
        raise ValueError("k8 / vt8 shape mismatch")
    if tuple(o.shape) != (B, Hq, Nq, d):
        raise ValueError("o shape mismatch")
    if lse is not None and tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("lse shape mismatch")
    nbq, nbk = (Nq + 127) // 128, (Nk + 127) // 128
    if (tuple(q_descale.shape) != (B, Hq, nbq) or tuple(k_descale.shape) != (B, Hkv, nbk)
            or tuple(v_descale.shape) != (B, Hkv, nbk)):
        raise ValueError("descale shape mismatch")
    if scale is None:
        scale = d ** -0.5
    odt = ATTN_OUT_F32 if o.dtype == torch.float32 else ATTN_OUT_BF16
    with _on(_one_device(q8, k8, vt8, q_descale, k_descale, v_descale, o, lse)):
        rc = load().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(q_descale), _ptr(k_descale),
                                 _ptr(v_descale), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, d,
                                 int(bool(causal)), float(scale), int(bool(rotated)), odt,
                                 _stream_ptr(stream))
    _check(rc, "attn_fwd_fp8")
    return o, lse


def forward_fp8(q, k, v, *, causal: bool = False, scale: float | None = None, signs=None,
                out_dtype=None, return_lse: bool = True, stream=None):
    """bf16 q, k, v -> E4M3 (Q and K rotated by diag(signs) H when signs is
    given: an int8 tensor of d values +-1) -> attn_fwd_fp8.  Returns (O, LSE)."""
    import torch
    d = q.shape[-1]
    if scale is None:
        scale = d ** -0.5
    q8, qd = fp8_quantize(q, signs, stream=stream)
    k8, kd = fp8_quantize(k, signs, stream=stream)
    vt8, vd = fp8_quantize(v, None, transpose=True, stream=stream)
    out_dtype = out_dtype or torch.bfloat16
    o = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    lse = (torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
           if return_lse else None)
    return attn_fwd_fp8(q8, k8, vt8, qd, kd, vd, o, lse, causal=causal, scale=scale,
                        rotated=signs is not None, stream=stream)


def attn_bwd_workspace_size(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int) -> int:
    return int(load().attn_bwd_workspace_size(B, Hq, Hkv, Nq, Nk, d))


def attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, *, causal: bool = False,
             scale: float | None = None, workspace=None, stream=None):
    """Backward into caller-provided gradients.

    q, dout [B,Hq,Nq,d] bf16; k, v [B,Hkv,Nk,d] bf16; o [B,Hq,Nq,d] bf16 or
    fp32 (the forward's output); lse [B,Hq,Nq] fp32 (the forward's natural-log
    logsumexp); dq [B,Hq,Nq,d] and dk, dv [B,Hkv,Nk,d], all bf16 or all fp32;
    workspace: uint8 of attn_bwd_workspace_size bytes.  Asynchronous."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be bfloat16 or float32")
    _need(o, o.dtype, "o")
    _need(lse, torch.float32, "lse")
    gdt = dq.dtype
    if gdt not in (torch.bfloat16, torch.float32) or dk.dtype != gdt or dv.dtype != gdt:
        raise TypeError("dq, dk, dv must all be bfloat16 or all float32")
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, gdt, n)
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if (tuple(k.shape) != (B, Hkv, Nk, d) or tuple(v.shape) != tuple(k.shape)
            or tuple(dk.shape) != tuple(k.shape) or tuple(dv.shape) != tuple(k.shape)):
        raise ValueError("k/v/dk/dv shape mismatch")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape) \
            or tuple(dq.shape) != tuple(q.shape):
        raise ValueError("o/dout/dq shape mismatch")
    if tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("lse shape mismatch")
    if scale is None:
        scale = d ** -0.5
    need = attn_bwd_workspace_size(B, Hq, Hkv, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        if isinstance(stream, torch.cuda.Stream):
            workspace.record_stream(stream)   # freed only after that stream's use
    odt = ATTN_OUT_F32 if o.dtype == torch.float32 else ATTN_OUT_BF16
    g32 = ATTN_OUT_F32 if gdt == torch.float32 else ATTN_OUT_BF16
    with _on(_one_device(q, k, v, o, dout, lse, dq, dk, dv, workspace)):
        rc = load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                             _ptr(dk), _ptr(dv), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)),
                             float(scale), odt, g32, _ptr(workspace), workspace.numel(),
                             _stream_ptr(stream))
    _check(rc, "attn_bwd")
    return dq, dk, dv


def backward(q, k, v, o, dout, lse, *, causal: bool = False, scale: float | None = None,
             grad_dtype=None, stream=None):
    """Allocate dQ, dK, dV (and the workspace) with torch and run attn_bwd."""
    import torch
    grad_dtype = grad_dtype or torch.bfloat16
    dq = torch.empty(q.shape, dtype=grad_dtype, device=q.device)
    dk = torch.empty(k.shape, dtype=grad_dtype, device=q.device)
    dv = torch.empty(v.shape, dtype=grad_dtype, device=q.device)
    return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, causal=causal, scale=scale,
                    stream=stream)


def attn_bwd_varlen_workspace_size(B: int, Hq: int, Hkv: int, total_q: int, d: int) -> int:
    return int(load().attn_bwd_varlen_workspace_size(B, Hq, Hkv, total_q, d))


def attn_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k,
                    max_seqlen_q: int, max_seqlen_k: int, *, causal: bool = False,
                    scale: float | None = None, workspace=None, stream=None):
    """Packed variable-length backward into caller-provided gradients.

    q, dout [total_q,Hq,d] bf16; k, v [total_k,Hkv,d] bf16; o [total_q,Hq,d]
    bf16 or fp32 and lse [Hq,total_q] fp32 from attn_fwd_varlen; dq
    [total_q,Hq,d] and dk, dv [total_k,Hkv,d], all bf16 or all fp32;
    cu_seqlens_q / cu_seqlens_k int32 [B+1] on the device; workspace: uint8 of
    attn_bwd_varlen_workspace_size bytes.  Asynchronous."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, torch.bfloat16, n)
    for t, n in ((cu_seqlens_q, "cu_seqlens_q"), (cu_seqlens_k, "cu_seqlens_k")):
        _need(t, torch.int32, n)
    if o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be bfloat16 or float32")
    _need(o, o.dtype, "o")
    _need(lse, torch.float32, "lse")
    gdt = dq.dtype
    if gdt not in (torch.bfloat16, torch.float32) or dk.dtype != gdt or dv.dtype != gdt:
        raise TypeError("dq, dk, dv must all be bfloat16 or all float32")
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, gdt, n)
    total_q, Hq, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    if (tuple(k.shape) != (total_k, Hkv, d) or tuple(v.shape) != tuple(k.shape)
            or tuple(dk.shape) != tuple(k.shape) or tuple(dv.shape) != tuple(k.shape)):
        raise ValueError("k/v/dk/dv shape mismatch")
    if tuple(o.shape) != tuple(q.shape) or tuple(dout.shape) != tuple(q.shape) \
            or tuple(dq.shape) != tuple(q.shape):
        raise ValueError("o/dout/dq shape mismatch")
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1 or B < 1:
        raise ValueError("cu_seqlens_q / cu_seqlens_k must both have B + 1 entries")
    if tuple(lse.shape) != (Hq, total_q):
        raise ValueError("lse shape mismatch")
    if scale is None:
        scale = d ** -0.5
    dev = _one_device(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, workspace)
    with _on(dev):
        if workspace is None:
            workspace = torch.empty(attn_bwd_varlen_workspace_size(B, Hq, Hkv, total_q, d),
                                    dtype=torch.uint8, device=dev)
            if isinstance(stream, torch.cuda.Stream):
                workspace.record_stream(stream)   # freed only after that stream's use
        ws_ptr, ws_bytes = _workspace(workspace)
        odt = ATTN_OUT_F32 if o.dtype == torch.float32 else ATTN_OUT_BF16
        g32 = ATTN_OUT_F32 if gdt == torch.float32 else ATTN_OUT_BF16
        rc = load().attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                    _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q),
                                    _ptr(cu_seqlens_k), B, Hq, Hkv, total_q, total_k,
                                    int(max_seqlen_q), int(max_seqlen_k), d, int(bool(causal)),
                                    float(scale), odt, g32, ws_ptr, ws_bytes, _stream_ptr(stream))
    _check(rc, "attn_bwd_varlen")
    return dq, dk, dv


def backward_varlen(q, k, v, o, dout, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                    max_seqlen_k: int, *, causal: bool = False, scale: float | None = None,
                    grad_dtype=None, stream=None):
    """Allocate dQ, dK, dV (and the workspace) with torch and run attn_bwd_varlen."""
    import torch
    grad_dtype = grad_dtype or torch.bfloat16
    dq = torch.empty(q.shape, dtype=grad_dtype, device=q.device)
    dk = torch.empty(k.shape, dtype=grad_dtype, device=q.device)
    dv = torch.empty(v.shape, dtype=grad_dtype, device=q.device)
    return attn_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens_q, cu_seqlens_k,
                           max_seqlen_q, max_seqlen_k, causal=causal, scale=scale, stream=stream)


def forward(q, k, v, *, causal: bool = False, scale: float | None = None,
            out_dtype=None, return_lse: bool = True, stream=None):
    """Allocate O (and LSE) with torch and run attn_fwd."""
    import torch
    out_dtype = out_dtype or torch.bfloat16
    o = torch.empty(q.shape, dtype=out_dtype, device=q.device)
    lse = (torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
           if return_lse else None)
    return attn_fwd(q, k, v, o, lse, causal=causal, scale=scale, stream=stream)


def attn_decode_workspace_size(B: int, Hq: int, Hkv: int, Nmax: int, d: int,
                               num_splits: int = 0) -> int:
    return int(load().attn_decode_workspace_size(B, Hq, Hkv, Nmax, d, num_splits))


def _check_decode_args(q, k_cache, v_cache, seqlens, o, lse):
    """Types and shapes of a contiguous-cache decode call (everything the
    kernels index by): q [B,Hq,1,d] bf16, caches [B,Hkv,Nmax,d] bf16, seqlens
    [B] int32, o [B,Hq,1,d] bf16/fp32, lse [B,Hq,1] fp32 or None.  Returns
    (B, Hq, Hkv, Nmax, d)."""
    import torch
    named = [(q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
             (v_cache, "v_cache", torch.bfloat16), (seqlens, "seqlens", torch.int32)]
    if lse is not None:
        named.append((lse, "lse", torch.float32))
    # types, then shapes, then placement: each is checked before any pointer
    # reaches the library
    for t, n, dt in named:
        if not isinstance(t, torch.Tensor) or t.dtype != dt:
            raise TypeError(f"{n} must be a {dt} tensor")
    if not isinstance(o, torch.Tensor) or o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be a bfloat16 or float32 tensor")
    if q.ndim != 4 or k_cache.ndim != 4:
        raise ValueError("q and the caches must be 4-D")
    B, Hq, one, d = q.shape
    Hkv, Nmax = k_cache.shape[1], k_cache.shape[2]
    if one != 1 or tuple(k_cache.shape) != (B, Hkv, Nmax, d) or v_cache.shape != k_cache.shape:
        raise ValueError("decode shape mismatch")
    if tuple(o.shape) != (B, Hq, 1, d) or tuple(seqlens.shape) != (B,):
        raise ValueError("decode output/seqlens shape mismatch")
    if lse is not None and tuple(lse.shape) != (B, Hq, 1):
        raise ValueError("lse shape mismatch")
    for t, n, dt in named + [(o, "o", o.dtype)]:
        _need(t, dt, n)
    return B, Hq, Hkv, Nmax, d


def attn_decode(q, k_cache, v_cache, seqlens, o, lse=None, *, scale: float | None = None,
                num_splits: int = 0, workspace=None, stream=None):
    """Split-KV decode into caller-provided outputs.

    q [B,Hq,1,d] bf16; caches [B,Hkv,Nmax,d] bf16; seqlens [B] int32 (device);
    o [B,Hq,1,d] bf16/fp32; lse [B,Hq,1] fp32 or None; workspace: a uint8
    CUDA tensor of at least attn_decode_workspace_size(...) bytes."""
    import torch
    B, Hq, Hkv, Nmax, d = _check_decode_args(q, k_cache, v_cache, seqlens, o, lse)
    if scale is None:
        scale = d ** -0.5
    ws_ptr, ws_bytes = _workspace(workspace)
    odt = ATTN_OUT_F32 if o.dtype == torch.float32 else ATTN_OUT_BF16
    with _on(_one_device(q, k_cache, v_cache, seqlens, o, lse)):
        rc = load().attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(o),
                                _ptr(lse), B, Hq, Hkv, Nmax, d, float(scale), int(num_splits),
                                ws_ptr, ws_bytes, odt, _stream_ptr(stream))
    _check(rc, "attn_decode")
    return o, lse


def decode(q, k_cache, v_cache, seqlens, *, scale=None, num_splits: int = 0,
           out_dtype=None, stream=None):
    """Allocate O, LSE and the workspace with torch and run attn_decode."""
    import torch
    out_dtype = out_dtype or torch.bfloat16
    B, Hq, _, d = q.shape
    Hkv, Nmax = k_cache.shape[1], k_cache.shape[2]
    ws = torch.empty(attn_decode_workspace_size(B, Hq, Hkv, Nmax, d, num_splits),
                     dtype=torch.uint8, device=q.device)
    o = torch.empty((B, Hq, 1, d), dtype=out_dtype, device=q.device)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    return attn_decode(q, k_cache, v_cache, seqlens, o, lse, scale=scale,
                       num_splits=num_splits, workspace=ws, stream=stream)


def attn_decode_noalloc(q, k_cache, v_cache, seqlens, o, lse=None, *,
                        scale: float | None = None, num_splits: int = 0, stream=None):
    """attn_decode without a workspace argument, for callers that cannot
    allocate device memory: the library's fixed 16 MiB per-device scratch array
    holds the split partials.  Calls that overlap on the GPU share that array
    and race; calls ordered on one stream do not.  The first call on a device
    must come before any stream capture."""
    import torch
    B, Hq, Hkv, Nmax, d = _check_decode_args(q, k_cache, v_cache, seqlens, o, lse)
    if scale is None:
        scale = d ** -0.5
    odt = ATTN_OUT_F32 if o.dtype == torch.float32 else ATTN_OUT_BF16
    with _on(_one_device(q, k_cache, v_cache, seqlens, o, lse)):
        rc = load().attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(o),
                                        _ptr(lse), B, Hq, Hkv, Nmax, d, float(scale),
                                        int(num_splits), odt, _stream_ptr(stream))
    _check(rc, "attn_decode_noalloc")
    return o, lse


def attn_selftest_bounded_wait(mode: int, result, stream=None) -> None:
    """Run the bounded-wait diagnostic (mode 0: time out; mode 1: abort flag)
    writing its outcome into `result` (an int32 CUDA tensor of one element)."""
    import torch
    _need(result, torch.int32, "result")
    with _on(_one_device(result)):
        _check(load().attn_selftest_bounded_wait(int(mode), _ptr(result), _stream_ptr(stream)),
               "attn_selftest_bounded_wait")


def attn_last_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(load().attn_last_device_error(_stream_ptr(stream)))


# ------------------------- host-side scheduling logic -------------------------
def attn_decode_num_splits(units: int, num_sms: int, max_splits: int = 128) -> int:
    return int(load().attn_decode_num_splits(units, num_sms, max_splits))


def attn_list_schedule(costs, workers: int, lpt: bool):
    """Returns (makespan, per-worker loads)."""
    n = len(costs)
    arr = (ctypes.c_int * max(n, 1))(*[int(c) for c in costs])
    loads = (ctypes.c_longlong * workers)()
    mk = load().attn_list_schedule(arr, n, workers, int(bool(lpt)), loads)
    if mk < 0:
        raise ValueError("attn_list_schedule rejected its arguments")
    return int(mk), [int(x) for x in loads]


def attn_kv_tiles(row0: int, rows: int, Nq: int, Nk: int, causal: bool, block: int) -> int:
    return int(load().attn_kv_tiles(row0, rows, Nq, Nk, int(bool(causal)), block))


def attn_fwd_num_units(B, Hq, Hkv, Nq, Nk, d, causal) -> int:
    return int(load().attn_fwd_num_units(B, Hq, Hkv, Nq, Nk, d, int(bool(causal))))


def attn_fwd_schedule(B, Hq, Hkv, Nq, Nk, d, causal, num_sms: int = 0):
    """Returns ([(b, hq, m_block), ...] in walk order, [cost, ...]) for a GPU
    with num_sms SMs (0: the fixed section widths)."""
    n = attn_fwd_num_units(B, Hq, Hkv, Nq, Nk, d, causal)
    units = (ctypes.c_int * (3 * n))()
    costs = (ctypes.c_int * n)()
    rc = load().attn_fwd_schedule(B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), int(num_sms), n,
                                  units, costs)
    if rc != 0:
        raise ValueError("attn_fwd_schedule rejected its arguments")
    return [tuple(units[3 * i:3 * i + 3]) for i in range(n)], list(costs)


def attn_fwd_split_plan(B, Hq, Hkv, Nq, Nk, d, causal, num_sms):
    """Returns (n_full, n_split, parts): the tail split attn_fwd applies on a
    GPU with num_sms SMs."""
    out = [ctypes.c_int() for _ in range(3)]
    rc = load().attn_fwd_split_plan(B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), num_sms,
                                    *(ctypes.byref(o) for o in out))
    if rc != 0:
        raise ValueError("attn_fwd_split_plan rejected its arguments")
    return tuple(o.value for o in out)


def attn_decode_kernel_launches(B, Hq, Hkv, Nmax, d, num_splits=0) -> int:
    """Kernels attn_decode launches for this shape: 1 (the split kernel merges)
    or 2 (split + combine)."""
    n = int(load().attn_decode_kernel_launches(B, Hq, Hkv, Nmax, d, num_splits))
    if n < 0:
        raise ValueError("attn_decode_kernel_launches rejected its arguments")
    return n


def attn_decode_paged(q, k_pages, v_pages, block_table, seqlens, o, lse=None, *,
                      scale: float | None = None, num_splits: int = 0, workspace=None,
                      stream=None):
    """Decode over a paged KV cache into caller-provided outputs.

    q [B,Hq,1,d] bf16; k_pages, v_pages [num_blocks, page_size, Hkv, d] bf16;
    block_table [B, max_blocks] int32; seqlens [B] int32; o [B,Hq,1,d] bf16
    or fp32; lse [B,Hq,1] fp32 or None.  Asynchronous."""
    import torch
    named = [(q, "q", torch.bfloat16), (k_pages, "k_pages", torch.bfloat16),
             (v_pages, "v_pages", torch.bfloat16), (block_table, "block_table", torch.int32),
             (seqlens, "seqlens", torch.int32)]
    if lse is not None:
        named.append((lse, "lse", torch.float32))
    for t, n, dt in named:   # types, then shapes, then placement
        if not isinstance(t, torch.Tensor) or t.dtype != dt:
            raise TypeError(f"{n} must be a {dt} tensor")
    if not isinstance(o, torch.Tensor) or o.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("o must be a bfloat16 or float32 tensor")
    if q.ndim != 4 or k_pages.ndim != 4:
        raise ValueError("q and the pages must be 4-D")
    B, Hq, one, d = q.shape
    num_blocks, page_size, Hkv, dk = k_pages.shape
    if one != 1 or dk != d or tuple(v_pages.shape) != tuple(k_pages.shape):
        raise ValueError("q / page shapes mismatch")
    if block_table.ndim != 2 or block_table.shape[0] != B or tuple(seqlens.shape) != (B,):
        raise ValueError("block_table must be [B, max_blocks] and seqlens [B]")
    if tuple(o.shape) != (B, Hq, 1, d):
        raise ValueError("o shape mismatch")
    if lse is not None and tuple(lse.shape) != (B, Hq, 1):
        raise ValueError("lse shape mismatch")
    for t, n, dt in named + [(o, "o", o.dtype)]:
        _need(t, dt, n)
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = d ** -0.5
    need = attn_decode_workspace_size(B, Hq, Hkv, max_blocks * page_size, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    odt = ATTN_OUT_F32 if o.dtype == torch.float32 else ATTN_OUT_BF16
    with _on(_one_device(q, k_pages, v_pages, block_table, seqlens, o, lse, workspace)):
        rc = load().attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                      _ptr(seqlens), _ptr(o), _ptr(lse), B, Hq, Hkv, num_blocks,
                                      page_size, max_blocks, d, float(scale), num_splits,
                                      _ptr(workspace), workspace.numel(), odt, _stream_ptr(stream))
    _check(rc, "attn_decode_paged")
    return o, lse


def decode_paged(q, k_pages, v_pages, block_table, seqlens, *, scale: float | None = None,
                 num_splits: int = 0, out_dtype=None, stream=None):
    """Allocate O and LSE with torch and run attn_decode_paged."""
    import torch
    out_dtype = out_dtype or torch.bfloat16
    B, Hq, _, d = q.shape
    o = torch.empty((B, Hq, 1, d), dtype=out_dtype, device=q.device)
    lse = torch.empty((B, Hq, 1), dtype=torch.float32, device=q.device)
    return attn_decode_paged(q, k_pages, v_pages, block_table, seqlens, o, lse, scale=scale,
                             num_splits=num_splits, stream=stream)
