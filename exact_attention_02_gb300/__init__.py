"""Exact tiled attention (forward + backward) for GB300 — thin Python binding.

Every function here marshals torch tensors into the C ABI of ``libfa_gb300.so``
(declared in ``include/fa.h``) and calls it on the current CUDA stream. All arithmetic
runs in the library's CUDA kernels; PyTorch only provides device memory and streams.
The library must be built (``exact_attention_02_gb300.build.build()``); if it is
missing, every call raises instead of computing anything another way.
"""
from __future__ import annotations

import ctypes
import math
import os

from .workloads import HEADLINE, WORKLOADS, Workload, make_inputs  # noqa: F401

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT, FA_ERR_WORKSPACE = range(6)
FA_DTYPE_BF16, FA_DTYPE_FP32 = 0, 1

# Which execution unit bounds each entry point's main kernel for bf16 inputs
# ("tensor": tcgen05 MMAs, "alu": FFMA pipes, "hbm": memory bandwidth). fp32 is all FFMA.
BF16_KERNEL_BOUND = {"fa_fwd": "tensor", "fa_bwd": "tensor", "fa_bwd_preprocess": "hbm"}
# Kernels each entry point launches, in order (the dQ accumulator clear in fa_bwd is a
# cudaMemsetAsync, not a library kernel).
BF16_KERNELS = {"fa_fwd": ["fa_fwd_tc_kernel"], "fa_bwd_preprocess": ["preprocess_kernel"],
                "fa_bwd": ["fa_bwd_wide_kernel", "dq_convert_kernel"]}
SPLITKV_KERNELS = ["splitkv_tc_kernel", "splitkv_merge_kernel"]
FP8_KERNELS = ["fa_fwd_tc_kernel"]  # the e4m3 instance of the forward kernel
FP32_KERNELS = {"fa_fwd": ["simt_fwd_kernel"], "fa_bwd_preprocess": ["preprocess_kernel"],
                "fa_bwd": ["simt_bwd_dkdv_kernel", "simt_bwd_dq_kernel"]}

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {error_string(status)}")


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"the CUDA library {LIB_PATH} is not built; run exact_attention_02_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, i, vp]
    L.fa_fwd.restype = i
    L.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
    L.fa_bwd_preprocess.restype = i
    L.fa_bwd_workspace_size.argtypes = [i, i, i, i, i]
    L.fa_bwd_workspace_size.restype = sz
    L.fa_bwd.argtypes = [vp] * 11 + [sz, i, i, i, i, f, i, i, vp]
    L.fa_bwd.restype = i
    L.fa_fwd_rect.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    L.fa_fwd_rect.restype = i
    L.fa_bwd_rect_workspace_size.argtypes = [i, i, i, i, i, i]
    L.fa_bwd_rect_workspace_size.restype = sz
    L.fa_bwd_rect.argtypes = [vp] * 11 + [sz, i, i, i, i, i, f, i, i, vp]
    L.fa_bwd_rect.restype = i
    L.fa_fwd_splitkv_workspace_size.argtypes = [i, i, i, i, i, i]
    L.fa_fwd_splitkv_workspace_size.restype = sz
    L.fa_fwd_splitkv.argtypes = [vp] * 5 + [i, i, i, i, i, f, i, i, vp, sz, vp]
    L.fa_fwd_splitkv.restype = i
    ll = ctypes.c_longlong
    L.fa_fwd_masked.argtypes = [vp] * 6 + [ll, ll, ll, i, i, i, i, f, i, i, vp]
    L.fa_fwd_masked.restype = i
    L.fa_bwd_masked.argtypes = [vp] * 11 + [ll, ll, ll, vp, sz, i, i, i, i, f, i, i, vp]
    L.fa_bwd_masked.restype = i
    L.fa_fwd_bitmask.argtypes = [vp] * 6 + [ll, ll, ll, i, i, i, i, f, i, i, vp]
    L.fa_fwd_bitmask.restype = i
    L.fa_bwd_bitmask.argtypes = [vp] * 11 + [ll, ll, ll, vp, sz, i, i, i, i, f, i, i, vp]
    L.fa_bwd_bitmask.restype = i
    ull = ctypes.c_ulonglong
    L.fa_fwd_dropout.argtypes = [vp] * 5 + [i, i, i, i, f, i, f, ull, i, vp]
    L.fa_fwd_dropout.restype = i
    L.fa_bwd_dropout.argtypes = [vp] * 11 + [sz, i, i, i, i, f, i, f, ull, i, vp]
    L.fa_bwd_dropout.restype = i
    L.fa_fwd_bwd_host_workspace_size.argtypes = [i, i, i, i, i, i]
    L.fa_fwd_bwd_host_workspace_size.restype = sz
    L.fa_fwd_bwd_host.argtypes = [vp] * 10 + [sz, i, i, i, i, f, i, i, i, vp]
    L.fa_fwd_bwd_host.restype = i
    L.fa_fwd_fp8.argtypes = [vp] * 5 + [i, i, i, i, f, i, f, f, f, vp]
    L.fa_fwd_fp8.restype = i
    L.fa_get_error_string.argtypes = [i]
    L.fa_get_error_string.restype = ctypes.c_char_p
    L.fa_get_last_device_status.argtypes = []
    L.fa_get_last_device_status.restype = i
    L.fa_test_inject_timeout.argtypes = [i, ctypes.c_ulonglong]
    L.fa_test_inject_timeout.restype = i
    L.fa_set_bwd_dq_mode.argtypes = [i]
    L.fa_set_bwd_dq_mode.restype = i
    L.fa_get_bwd_dq_mode.argtypes = []
    L.fa_get_bwd_dq_mode.restype = i
    _lib = L
    return L


def lib():
    """The loaded ctypes library (raises if it is not built)."""
    return _load()


def error_string(status: int) -> str:
    return _load().fa_get_error_string(int(status)).decode()


def _check(status: int, where: str):
    if status != FA_OK:
        raise FAError(status, where)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return FA_DTYPE_BF16
    if t.dtype == torch.float32:
        return FA_DTYPE_FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream_ptr(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(x) for x in q.shape)


def _same(ref, *ts):
    for t in ts:
        if t is None:
            continue
        if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device:
            raise ValueError("Q/K/V/O/dO/dQ/dK/dV must share shape, dtype and device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def padded_mask(mask):
    """A copy of a [B|1, H|1, N, N] bf16 mask whose rows are padded to a multiple of 8
    elements (the layout ``fa_fwd_masked`` reads); returns a view of the first N columns."""
    import torch
    n = int(mask.shape[-1])
    cols = (n + 7) // 8 * 8
    out = torch.zeros(tuple(mask.shape[:-1]) + (cols,), dtype=torch.bfloat16, device=mask.device)
    out[..., :n] = mask
    return out[..., :n]


def _mask_args(mask, q):
    """Pointer and element strides (batch, head, row) of an additive mask for q's shape."""
    import torch
    B, H, N, _ = _shape(q)
    if mask.dim() != 4 or mask.dtype != torch.bfloat16 or mask.device != q.device:
        raise ValueError("mask must be a bf16 [B or 1, H or 1, N, N] tensor on q's device")
    mb, mh, mn, mc = (int(x) for x in mask.shape)
    if mb not in (1, B) or mh not in (1, H) or mn != N or mc != N or mask.stride(3) != 1:
        raise ValueError("mask must be [B or 1, H or 1, N, N] with contiguous rows")
    srow = int(mask.stride(2))
    sb = 0 if mb == 1 else int(mask.stride(0))
    sh = 0 if mh == 1 else int(mask.stride(1))
    if srow % 8 or sb % 8 or sh % 8 or srow < (N + 7) // 8 * 8:
        raise ValueError("mask rows must start 16-byte aligned: use padded_mask(mask)")
    return _p(mask), sb, sh, srow


def pack_mask_bits(visible):
    """The int32 words ``fa_fwd_bitmask`` reads for a boolean [B|1, H|1, N, N] tensor
    (True: the key is visible): bit j % 32 of word j / 32 of each row, each row padded to
    4 words per 128 keys. Returns [B|1, H|1, N, 4 * ceil(N / 128)] on visible's device."""
    import torch
    n = int(visible.shape[-1])
    words = (n + 127) // 128 * 4
    lead = tuple(visible.shape[:-1])
    v = torch.zeros(lead + (words * 32,), dtype=torch.uint8, device=visible.device)
    v[..., :n] = visible.to(torch.uint8)
    # one byte per 8 keys (bit k = key 8i + k); read as little-endian words, byte i of a
    # word holds keys 8i .. 8i+7 of its 32, so bit j % 32 of word j / 32 is key j
    shifts = torch.arange(8, dtype=torch.uint8, device=visible.device)
    b = (v.view(lead + (words * 4, 8)) << shifts).sum(-1, dtype=torch.uint8)
    return b.view(torch.int32)


def _bits_args(bits, q):
    """Pointer and word strides (batch, head, row) of packed mask bits for q's shape."""
    import torch
    B, H, N, _ = _shape(q)
    if bits.dim() != 4 or bits.dtype != torch.int32 or bits.device != q.device:
        raise ValueError("mask_bits must be an int32 [B or 1, H or 1, N, words] tensor on q's device")
    mb, mh, mn, mw = (int(x) for x in bits.shape)
    if mb not in (1, B) or mh not in (1, H) or mn != N or mw < (N + 127) // 128 * 4 or bits.stride(3) != 1:
        raise ValueError("mask_bits must be [B or 1, H or 1, N, >= 4 * ceil(N / 128)] with contiguous rows: "
                         "use pack_mask_bits(visible)")
    srow = int(bits.stride(2))
    sb = 0 if mb == 1 else int(bits.stride(0))
    sh = 0 if mh == 1 else int(bits.stride(1))
    if srow % 4 or sb % 4 or sh % 4:
        raise ValueError("mask_bits strides must be multiples of 4 words")
    return _p(bits), sb, sh, srow


def fa_fwd(q, k, v, causal: bool, scale: float | None = None, o=None, lse=None, stream=None, mask=None,
           dropout: tuple[float, int] | None = None, mask_bits=None):
    """O, LSE = attention forward of [B, H, N, d] CUDA tensors (see ``fa_fwd`` in fa.h).
    With ``mask`` (bf16 [B|1, H|1, N, N], added to the scaled scores) it calls
    ``fa_fwd_masked``; with ``mask_bits`` (a boolean mask packed by ``pack_mask_bits``)
    ``fa_fwd_bitmask``; with ``dropout = (p, seed)`` it calls ``fa_fwd_dropout``."""
    import torch
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _same(q, k, v, o)
    if sum(x is not None for x in (mask, mask_bits, dropout)) > 1:
        raise ValueError("only one of mask, mask_bits and dropout per call is supported")
    if mask_bits is not None:
        bp, sb, sh, srow = _bits_args(mask_bits, q)
        _check(_load().fa_fwd_bitmask(_p(q), _p(k), _p(v), _p(o), _p(lse), bp, sb, sh, srow, B, H, N, d, scale,
                                      int(bool(causal)), _dtype_code(q), _stream_ptr(stream)), "fa_fwd_bitmask")
        return o, lse
    if dropout is not None:
        pd, seed = float(dropout[0]), int(dropout[1]) & 0xFFFFFFFFFFFFFFFF
        _check(_load().fa_fwd_dropout(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d, scale, int(bool(causal)), pd,
                                      seed, _dtype_code(q), _stream_ptr(stream)), "fa_fwd_dropout")
        return o, lse
    if mask is not None:
        mp, sb, sh, srow = _mask_args(mask, q)
        _check(_load().fa_fwd_masked(_p(q), _p(k), _p(v), _p(o), _p(lse), mp, sb, sh, srow, B, H, N, d, scale,
                                     int(bool(causal)), _dtype_code(q), _stream_ptr(stream)), "fa_fwd_masked")
        return o, lse
    _check(_load().fa_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, d, scale, int(bool(causal)),
                          _dtype_code(q), _stream_ptr(stream)), "fa_fwd")
    return o, lse


def fa_bwd_preprocess(o, do, D=None, stream=None):
    """D = rowsum(dO * O) as float32 [B, H, N] (see ``fa_bwd_preprocess`` in fa.h)."""
    import torch
    B, H, N, d = _shape(o)
    _same(o, do)
    D = torch.empty((B, H, N), dtype=torch.float32, device=o.device) if D is None else D
    _check(_load().fa_bwd_preprocess(_p(o), _p(do), _p(D), B, H, N, d, _dtype_code(o),
                                     _stream_ptr(stream)), "fa_bwd_preprocess")
    return D


def fa_bwd_workspace_size(B: int, H: int, N: int, d: int, dtype) -> int:
    import torch
    code = dtype if isinstance(dtype, int) else (FA_DTYPE_BF16 if dtype == torch.bfloat16 else FA_DTYPE_FP32)
    return int(_load().fa_bwd_workspace_size(B, H, N, d, code))


def fa_bwd(q, k, v, o, do, lse, causal: bool, scale: float | None = None, D=None,
           dq=None, dk=None, dv=None, workspace=None, stream=None, mask=None,
           dropout: tuple[float, int] | None = None, mask_bits=None):
    """dQ, dK, dV of attention from the forward's O and LSE (see ``fa_bwd`` in fa.h);
    with ``mask`` (the forward's additive mask) it calls ``fa_bwd_masked``, with
    ``mask_bits`` (the forward's packed boolean mask) ``fa_bwd_bitmask``, with
    ``dropout`` (the forward's (p, seed)) ``fa_bwd_dropout``."""
    import torch
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _same(q, k, v, o, do, dq, dk, dv)
    need = fa_bwd_workspace_size(B, H, N, d, q.dtype) + (0 if D is not None else 4 * B * H * N)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if sum(x is not None for x in (mask, mask_bits, dropout)) > 1:
        raise ValueError("only one of mask, mask_bits and dropout per call is supported")
    if mask_bits is not None:
        bp, sb, sh, srow = _bits_args(mask_bits, q)
        _check(_load().fa_bwd_bitmask(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(D), _p(dq), _p(dk), _p(dv),
                                      bp, sb, sh, srow, _p(workspace), wbytes, B, H, N, d, scale, int(bool(causal)),
                                      _dtype_code(q), _stream_ptr(stream)), "fa_bwd_bitmask")
        return dq, dk, dv
    if dropout is not None:
        pd, seed = float(dropout[0]), int(dropout[1]) & 0xFFFFFFFFFFFFFFFF
        _check(_load().fa_bwd_dropout(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(D), _p(dq), _p(dk), _p(dv),
                                      _p(workspace), wbytes, B, H, N, d, scale, int(bool(causal)), pd, seed,
                                      _dtype_code(q), _stream_ptr(stream)), "fa_bwd_dropout")
        return dq, dk, dv
    if mask is not None:
        mp, sb, sh, srow = _mask_args(mask, q)
        _check(_load().fa_bwd_masked(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(D), _p(dq), _p(dk), _p(dv),
                                     mp, sb, sh, srow, _p(workspace), wbytes, B, H, N, d, scale, int(bool(causal)),
                                     _dtype_code(q), _stream_ptr(stream)), "fa_bwd_masked")
        return dq, dk, dv
    _check(_load().fa_bwd(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(D), _p(dq), _p(dk), _p(dv),
                          _p(workspace), wbytes, B, H, N, d, scale, int(bool(causal)), _dtype_code(q),
                          _stream_ptr(stream)), "fa_bwd")
    return dq, dk, dv


def _rect_shapes(q, k, v, *others_q):
    """(B, H, Nq, Nk, d) of q [B,H,Nq,d] against k, v [B,H,Nk,d]; checks contiguity, dtype
    and device, and that the tensors in ``others_q`` have q's shape."""
    B, H, Nq, d = _shape(q)
    if k.dim() != 4 or k.shape != v.shape or tuple(k.shape[:2]) != (B, H) or int(k.shape[3]) != d:
        raise ValueError("k and v must be [B, H, Nk, d] with the batch, heads and d of q")
    for t in (q, k, v) + tuple(t for t in others_q if t is not None):
        if not t.is_contiguous() or t.dtype != q.dtype or t.device != q.device:
            raise ValueError("tensors must be contiguous and share dtype and device")
    for t in others_q:
        if t is not None and t.shape != q.shape:
            raise ValueError("O, dO and dQ must have q's shape")
    return B, H, Nq, int(k.shape[2]), d


def fa_fwd_rect(q, k, v, causal: bool, scale: float | None = None, o=None, lse=None, stream=None):
    """O, LSE for q [B,H,Nq,d] against k, v [B,H,Nk,d] (see ``fa_fwd_rect`` in fa.h; causal
    is bottom-right aligned: query i hides keys j > i + Nk - Nq)."""
    import torch
    B, H, Nq, Nk, d = _rect_shapes(q, k, v, o)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(_load().fa_fwd_rect(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, Nq, Nk, d, scale, int(bool(causal)),
                               _dtype_code(q), _stream_ptr(stream)), "fa_fwd_rect")
    return o, lse


def fa_bwd_rect(q, k, v, o, do, lse, causal: bool, scale: float | None = None, D=None, dq=None, dk=None, dv=None,
                workspace=None, stream=None):
    """dQ [B,H,Nq,d], dK, dV [B,H,Nk,d] from the outputs of ``fa_fwd_rect`` (see
    ``fa_bwd_rect`` in fa.h)."""
    import torch
    B, H, Nq, Nk, d = _rect_shapes(q, k, v, o, do, dq)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if dk.shape != k.shape or dv.shape != v.shape or not dk.is_contiguous() or not dv.is_contiguous():
        raise ValueError("dK and dV must be contiguous with k's shape")
    code = _dtype_code(q)
    need = int(_load().fa_bwd_rect_workspace_size(B, H, Nq, Nk, d, code)) + (0 if D is not None else 4 * B * H * Nq)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_load().fa_bwd_rect(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(D), _p(dq), _p(dk), _p(dv),
                               _p(workspace), wbytes, B, H, Nq, Nk, d, scale, int(bool(causal)), code,
                               _stream_ptr(stream)), "fa_bwd_rect")
    return dq, dk, dv


def fa_fwd_splitkv(q, k, v, causal: bool, scale: float | None = None, o=None, lse=None, workspace=None,
                   stream=None):
    """O, LSE for a few queries q [B,H,Nq,d] against k, v [B,H,Nk,d] (see ``fa_fwd_splitkv`` in fa.h)."""
    import torch
    B, H, Nq, d = _shape(q)
    Nk = int(k.shape[2])
    if k.shape != v.shape or tuple(k.shape[:2]) != (B, H) or int(k.shape[3]) != d:
        raise ValueError("k and v must be [B, H, Nk, d] with the batch, heads and d of q")
    for t in (q, k, v):
        if not t.is_contiguous() or t.dtype != q.dtype or t.device != q.device:
            raise ValueError("q, k, v must be contiguous and share dtype and device")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    code = _dtype_code(q)
    need = int(_load().fa_fwd_splitkv_workspace_size(B, H, Nq, Nk, d, code))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    wbytes = workspace.numel() * workspace.element_size()
    _check(_load().fa_fwd_splitkv(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, Nq, Nk, d, scale,
                                  int(bool(causal)), code, _p(workspace), wbytes, _stream_ptr(stream)),
           "fa_fwd_splitkv")
    return o, lse


def fa_fwd_fp8(q8, k8, v8, descale, causal: bool, scale: float | None = None, o=None, lse=None, stream=None):
    """O (bf16), LSE for e4m3 q8, k8, v8 [B,H,N,d] with dequantisation factors
    descale = (q, k, v) (see ``fa_fwd_fp8`` in fa.h). The byte tensors may be uint8 or
    float8_e4m3fn; only their bytes are passed."""
    import torch
    B, H, N, d = _shape(q8)
    for t in (q8, k8, v8):
        if t.shape != q8.shape or t.element_size() != 1 or not t.is_contiguous() or t.device != q8.device:
            raise ValueError("q8, k8, v8 must be contiguous one-byte [B, H, N, d] tensors on one device")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    qd, kd, vd = (float(x) for x in descale)
    _check(_load().fa_fwd_fp8(_p(q8), _p(k8), _p(v8), _p(o), _p(lse), B, H, N, d, scale, int(bool(causal)),
                              qd, kd, vd, _stream_ptr(stream)), "fa_fwd_fp8")
    return o, lse


def fa_fwd_bwd_host_workspace_size(B: int, H: int, N: int, d: int, chunks: int = 0) -> int:
    return int(_load().fa_fwd_bwd_host_workspace_size(B, H, N, d, FA_DTYPE_BF16, chunks))


def fa_fwd_bwd_host(q, k, v, do, causal: bool, scale: float | None = None, out=None, chunks: int = 0,
                    workspace=None, stream=None):
    """Forward + backward of host-resident bf16 tensors q, k, v, do [B,H,N,d] (page-locked
    for overlap; see ``fa_fwd_bwd_host`` in fa.h). Returns host (o, lse, dq, dk, dv); they
    hold the results once ``stream`` (default: the current stream) has been synchronised.
    ``out`` may pass preallocated host tensors in that order."""
    import torch
    B, H, N, d = _shape(q)
    for t in (q, k, v, do):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("q, k, v, do must be contiguous bf16 host tensors of one shape")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        pin = torch.cuda.is_available()
        out = (torch.empty_like(q, pin_memory=pin), torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin),
               torch.empty_like(q, pin_memory=pin), torch.empty_like(q, pin_memory=pin),
               torch.empty_like(q, pin_memory=pin))
    need = fa_fwd_bwd_host_workspace_size(B, H, N, d, chunks)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
    wbytes = workspace.numel() * workspace.element_size()
    o, lse, dq, dk, dv = out
    _check(_load().fa_fwd_bwd_host(_p(q), _p(k), _p(v), _p(do), _p(o), _p(lse), _p(dq), _p(dk), _p(dv), _p(workspace),
                                   wbytes, B, H, N, d, scale, int(bool(causal)), FA_DTYPE_BF16, int(chunks),
                                   _stream_ptr(stream)), "fa_fwd_bwd_host")
    return out


def fa_get_last_device_status() -> int:
    return int(_load().fa_get_last_device_status())


# How the bf16 backward computes dQ (``fa_set_bwd_dq_mode`` in fa.h): chosen by shape,
# atomic fp32 partials, or the separate dQ pass.
FA_BWD_DQ_AUTO, FA_BWD_DQ_ATOMIC, FA_BWD_DQ_SEPARATE = 0, 1, 2


def fa_set_bwd_dq_mode(mode: int) -> None:
    _check(_load().fa_set_bwd_dq_mode(int(mode)), "fa_set_bwd_dq_mode")


def fa_get_bwd_dq_mode() -> int:
    return int(_load().fa_get_bwd_dq_mode())


# Failure-path test hook (see ``fa_test_inject_timeout`` in fa.h): which = 1 makes the
# first CTA of fa_fwd skip one producer arrival, 2 the same in fa_bwd, 0 turns it off.
FA_INJECT_OFF, FA_INJECT_FWD, FA_INJECT_BWD = 0, 1, 2


def fa_test_inject_timeout(which: int, wait_limit_ns: int = 0) -> None:
    _check(_load().fa_test_inject_timeout(int(which), int(wait_limit_ns)), "fa_test_inject_timeout")
