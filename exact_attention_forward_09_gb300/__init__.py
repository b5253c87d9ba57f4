"""Fused exact attention forward for NVIDIA GB300 (sm_103a).

The product is the C library ``libfa.so`` (C ABI declared in
``include/fa.h``; hand-written CUDA kernels under ``csrc/``).  This package is
a thin ctypes binding with the same entry-point names: it checks tensor
shapes, allocates outputs with torch, passes raw device pointers and the
current CUDA stream, and turns status codes into exceptions.  Every step of
the computation runs in the library's kernels; there is no other code path.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from .build import LIB as _LIB_PATH

__all__ = ["fwd_host", "fwd_host_workspace_bytes", "bwd", "bwd_workspace_bytes", "fwd_splitkv", "splitkv_workspace_bytes", "fwd", "fwd_gqa", "fwd_fp8", "fwd_fp8_gqa", "quant_fp8", "quant_fp8_per_tensor_noalloc", "check_device_error", "lib",
           "FaError", "FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT",
           "FA_ERR_SCRATCH_LIMIT", "FA_DTYPE_BF16", "FA_DTYPE_FP16", "FP8_BLOCK_ROWS",
           "FA_ROPE_INTERLEAVED", "FA_ROPE_HALF",
           "QUANT_NOALLOC_MAX_BLOCKS"]

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, 1, 2, 3, 4
FA_ERR_SCRATCH_LIMIT = 5
QUANT_NOALLOC_MAX_BLOCKS = 65536
FA_DTYPE_BF16, FA_DTYPE_FP16 = 0, 1
FA_ROPE_INTERLEAVED, FA_ROPE_HALF = 1, 2
FP8_BLOCK_ROWS = 128


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib().fa_status_string(status).decode()}")


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libfa.so has not been built ({_LIB_PATH}); run "
                              "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, f32, i32, vp]
        lib.fa_fwd.restype = i32
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, f32, vp, vp, vp, vp]
        lib.fa_fwd_fp8.restype = i32
        lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, f32, i32, vp]
        lib.fa_fwd_gqa.restype = i32
        lib.fa_fwd_fp8_gqa.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, f32, vp, vp, vp,
                                       vp]
        lib.fa_fwd_fp8_gqa.restype = i32
        lib.fa_quant_fp8.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, i32, vp, vp]
        lib.fa_quant_fp8.restype = i32
        lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, f32, i32, i32, vp,
                                       ctypes.c_size_t, vp]
        lib.fa_fwd_splitkv.restype = i32
        lib.fa_splitkv_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i64, i32, ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_splitkv_workspace_bytes.restype = i32
        lib.fa_quant_fp8_rope.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp, i32, vp, i32, vp, vp]
        lib.fa_quant_fp8_rope.restype = i32
        lib.fa_quant_fp8_qkv.argtypes = [vp] * 9 + [i64] * 6 + [vp, vp]
        lib.fa_quant_fp8_qkv.restype = i32
        lib.fa_quant_fp8_per_tensor_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp]
        lib.fa_quant_fp8_per_tensor_noalloc.restype = i32
        lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, f32, i32, vp,
                                    ctypes.c_size_t, vp]
        lib.fa_fwd_host.restype = i32
        lib.fa_fwd_host_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, i64, ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_fwd_host_workspace_bytes.restype = i32
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, f32, i32,
                               vp, ctypes.c_size_t, vp]
        lib.fa_bwd.restype = i32
        lib.fa_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64, ctypes.POINTER(ctypes.c_size_t)]
        lib.fa_bwd_workspace_bytes.restype = i32
        lib.fa_status_string.argtypes = [i32]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_check_device_error.argtypes = [vp]
        lib.fa_check_device_error.restype = i32
        lib.fa_debug_inject.argtypes = [i32]
        lib.fa_debug_inject.restype = i32
        lib.fa_debug_exp2.argtypes = [vp, vp, i64, i32, vp]
        lib.fa_debug_exp2.restype = i32
        lib.fa_version.argtypes = []
        lib.fa_version.restype = i32
        _LIB = lib
    return _LIB


def lib():
    """The loaded ctypes library (raw C entry points)."""
    return _lib()


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _check(status: int, where: str):
    if status != FA_OK:
        raise FaError(status, where)


def _check_qkv(q, k, v, allowed):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
        if t.dtype not in allowed:
            raise ValueError(f"{name} has dtype {t.dtype}; expected one of {allowed}")
    if not (q.shape == k.shape == v.shape and q.dtype == k.dtype == v.dtype and
            q.device == k.device == v.device):
        raise ValueError("q, k, v must share shape, dtype and device")


def fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
        scale: float | None = None, out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
    """BF16/FP16 attention forward (``fa_fwd``).  Returns (O, LSE)."""
    _check_qkv(q, k, v, (torch.bfloat16, torch.float16))
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    dt = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
    with torch.cuda.device(q.device):
        st = _lib().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                           B, H, N, d, int(bool(causal)), float(scale), dt, _stream(q))
    _check(st, "fa_fwd")
    return out, lse


def splitkv_workspace_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, num_splits: int = 0) -> int:
    """Device workspace (bytes) ``fwd_splitkv`` needs on the current device."""
    n = ctypes.c_size_t(0)
    _check(_lib().fa_splitkv_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, int(num_splits), ctypes.byref(n)),
           "fa_splitkv_workspace_bytes")
    return int(n.value)


def fwd_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                scale: float | None = None, num_splits: int = 0, out: torch.Tensor | None = None,
                lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """Split-KV forward for decode-like shapes (``fa_fwd_splitkv``): q [B, Hq,
    Nq, d], k/v [B, Hkv, Nk, d]; the query heads of a key/value group are
    packed together and the keys split into ``num_splits`` runs (0: chosen
    for the device).  Returns (O [B, Hq, Nq, d], LSE [B, Hq, Nq])."""
    _check_gqa(q, k, v, (torch.bfloat16, torch.float16))
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    dt = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
    with torch.cuda.device(q.device):
        need = splitkv_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, num_splits)
        if workspace is None and need > 0:
            workspace = torch.empty((need,), dtype=torch.uint8, device=q.device)
        wp = workspace.data_ptr() if workspace is not None else None
        wb = workspace.numel() * workspace.element_size() if workspace is not None else 0
        st = _lib().fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale), dt, int(num_splits),
                                   wp, wb, _stream(q))
    _check(st, "fa_fwd_splitkv")
    return out, lse


def fwd_host_workspace_bytes(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int) -> int:
    """Bytes of device workspace ``fa_fwd_host`` needs for this shape."""
    n = ctypes.c_size_t(0)
    _check(_lib().fa_fwd_host_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, ctypes.byref(n)), "fa_fwd_host_workspace_bytes")
    return int(n.value)


def fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False, scale: float | None = None,
             out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
             workspace: torch.Tensor | None = None, device=None):
    """``fa_fwd_host``: q [B, Hq, Nq, d], k/v [B, Hkv, Nk, d] in HOST memory
    (page-locked for overlapped copies); the call copies them to the device,
    runs the kernel and copies O and LSE back, asynchronously on the current
    stream of ``device`` (default: the current CUDA device).  Returns
    (O, LSE) as host tensors, complete once that stream has synchronised."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D host tensor")
        if t.dtype not in (torch.bfloat16, torch.float16):
            raise ValueError(f"{name} has dtype {t.dtype}; expected bf16 or fp16")
    B, Hq, Nq, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d or q.dtype != k.dtype or k.dtype != v.dtype:
        raise ValueError("k and v must be [B, Hkv, Nk, d] with q's batch, head dimension and dtype")
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=pin)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, pin_memory=pin)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    dt = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
    with torch.cuda.device(dev):
        need = fwd_host_workspace_bytes(B, Hq, Hkv, Nq, Nk, d)
        if workspace is None:
            workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
        st = _lib().fa_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale), dt,
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                torch.cuda.current_stream(dev).cuda_stream)
    _check(st, "fa_fwd_host")
    return out, lse


def bwd_workspace_bytes(B: int, Hq: int, Nq: int, d: int) -> int:
    """Bytes of device workspace ``fa_bwd`` needs for this shape."""
    n = ctypes.c_size_t(0)
    _check(_lib().fa_bwd_workspace_bytes(B, Hq, Nq, d, ctypes.byref(n)), "fa_bwd_workspace_bytes")
    return int(n.value)


def bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
        dout: torch.Tensor, causal: bool = False, scale: float | None = None, dq: torch.Tensor | None = None,
        dk: torch.Tensor | None = None, dv: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """Gradients of sum(dout * O) (``fa_bwd``): q, out, dout [B, Hq, Nq, d],
    k/v [B, Hkv, Nk, d], lse [B, Hq, Nq] fp32 from the forward with the same
    causal flag and scale.  Returns (dq, dk, dv)."""
    _check_gqa(q, k, v, (torch.bfloat16, torch.float16))
    for name, t in (("out", out), ("dout", dout)):
        if not isinstance(t, torch.Tensor) or t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous() \
                or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous tensor with q's shape, dtype and device")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if not isinstance(lse, torch.Tensor) or lse.shape != (B, Hq, Nq) or lse.dtype != torch.float32 \
            or not lse.is_contiguous() or lse.device != q.device:
        raise ValueError("lse must be a contiguous fp32 [B, Hq, Nq] tensor on q's device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    dt = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
    with torch.cuda.device(q.device):
        need = bwd_workspace_bytes(B, Hq, Nq, d)
        if workspace is None:
            workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=q.device)
        st = _lib().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                           dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                           B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale), dt,
                           workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream(q))
    _check(st, "fa_bwd")
    return dq, dk, dv


def _check_gqa(q, k, v, allowed):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor")
        if t.dtype not in allowed:
            raise ValueError(f"{name} has dtype {t.dtype}; expected one of {allowed}")
    B, Hq, Nq, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d or q.dtype != k.dtype or k.dtype != v.dtype:
        raise ValueError("k and v must be [B, Hkv, Nk, d] with q's batch, head dimension and dtype")
    if k.shape[1] == 0 or Hq % k.shape[1] != 0:
        raise ValueError("the number of query heads must be a multiple of the number of key/value heads")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k, v must be on one device")


def fwd_gqa(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
            scale: float | None = None, out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
    """Grouped/multi-query attention with Nq != Nk allowed (``fa_fwd_gqa``):
    q [B, Hq, Nq, d], k/v [B, Hkv, Nk, d]; causal masks are bottom-right
    aligned.  Returns (O [B, Hq, Nq, d], LSE [B, Hq, Nq])."""
    _check_gqa(q, k, v, (torch.bfloat16, torch.float16))
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    dt = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
    with torch.cuda.device(q.device):
        st = _lib().fa_fwd_gqa(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale), dt, _stream(q))
    _check(st, "fa_fwd_gqa")
    return out, lse


def fwd_fp8_gqa(q8, k8, v8, q_descale, k_descale, v_descale, causal: bool = False,
                scale: float | None = None, out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
    """FP8 E4M3 version of ``fwd_gqa`` (``fa_fwd_fp8_gqa``); descales are
    [B, Hq, ceil(Nq/128)] for Q and [B, Hkv, ceil(Nk/128)] for K and V."""
    _check_gqa(q8, k8, v8, (torch.uint8, torch.float8_e4m3fn))
    B, Hq, Nq, d = q8.shape
    Hkv, Nk = k8.shape[1], k8.shape[2]
    nq, nk = (Nq + FP8_BLOCK_ROWS - 1) // FP8_BLOCK_ROWS, (Nk + FP8_BLOCK_ROWS - 1) // FP8_BLOCK_ROWS
    for name, t, shape in (("q_descale", q_descale, (B, Hq, nq)), ("k_descale", k_descale, (B, Hkv, nk)),
                           ("v_descale", v_descale, (B, Hkv, nk))):
        if t.dtype != torch.float32 or tuple(t.shape) != shape or not t.is_contiguous() or t.device != q8.device:
            raise ValueError(f"{name} must be a contiguous fp32 {list(shape)} tensor on {q8.device}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, Nq, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q8.device)
    with torch.cuda.device(q8.device):
        st = _lib().fa_fwd_fp8_gqa(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                   B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale), q_descale.data_ptr(),
                                   k_descale.data_ptr(), v_descale.data_ptr(), _stream(q8))
    _check(st, "fa_fwd_fp8_gqa")
    return out, lse


def fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, v8: torch.Tensor, q_descale: torch.Tensor,
            k_descale: torch.Tensor, v_descale: torch.Tensor, causal: bool = False,
            scale: float | None = None, out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
    """FP8 E4M3 attention forward (``fa_fwd_fp8``).  q8/k8/v8 hold E4M3 codes
    (uint8 or float8_e4m3fn), descales are [B, H, ceil(N/128)] fp32.
    Returns (O bf16, LSE fp32)."""
    _check_qkv(q8, k8, v8, (torch.uint8, torch.float8_e4m3fn))
    B, H, N, d = q8.shape
    nblk = (N + FP8_BLOCK_ROWS - 1) // FP8_BLOCK_ROWS
    for name, t in (("q_descale", q_descale), ("k_descale", k_descale), ("v_descale", v_descale)):
        if t.dtype != torch.float32 or tuple(t.shape) != (B, H, nblk) or not t.is_contiguous() or \
                t.device != q8.device:
            raise ValueError(f"{name} must be a contiguous fp32 [B, H, {nblk}] tensor on {q8.device}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    with torch.cuda.device(q8.device):
        st = _lib().fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               B, H, N, d, int(bool(causal)), float(scale), q_descale.data_ptr(),
                               k_descale.data_ptr(), v_descale.data_ptr(), _stream(q8))
    _check(st, "fa_fwd_fp8")
    return out, lse


def quant_fp8(x: torch.Tensor, signs=None, per_tensor: bool = False, workspace: torch.Tensor | None = None,
              rope=None):
    """fp32 [B, H, N, d] -> (E4M3 codes uint8 [B, H, N, d], descale fp32
    [B, H, ceil(N/128)]) via ``fa_quant_fp8``.  ``signs``: d entries of +-1
    (host sequence / numpy / CPU tensor) for the Hadamard rotation, or None.
    ``rope``: None, or (cos, sin, layout) with cos / sin contiguous fp32 CUDA
    tensors [N, d/2] and layout FA_ROPE_INTERLEAVED or FA_ROPE_HALF: the
    rotary embedding is applied first, in the same pass (``fa_quant_fp8_rope``)."""
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32 or x.dim() != 4 \
            or not x.is_contiguous():
        raise ValueError("x must be a contiguous fp32 [B, H, N, d] CUDA tensor")
    B, H, N, d = x.shape
    nblk = (N + FP8_BLOCK_ROWS - 1) // FP8_BLOCK_ROWS
    x8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
    ds = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device)
    sp = None
    keep = None
    if signs is not None:
        keep = (ctypes.c_int8 * d)(*[int(s) for s in (signs.tolist() if hasattr(signs, "tolist") else signs)])
        sp = ctypes.cast(keep, ctypes.c_void_p)
    ws = None
    if per_tensor:
        if workspace is None:
            workspace = torch.empty((1,), dtype=torch.float32, device=x.device)
        ws = workspace.data_ptr()
    with torch.cuda.device(x.device):
        if rope is None:
            st = _lib().fa_quant_fp8(x.data_ptr(), x8.data_ptr(), ds.data_ptr(), B, H, N, d, sp,
                                     int(bool(per_tensor)), ws, _stream(x))
            name = "fa_quant_fp8"
        else:
            cos, sin, layout = rope
            for nm, t in (("cos", cos), ("sin", sin)):
                if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 \
                        or not t.is_contiguous() or tuple(t.shape) != (N, d // 2) or t.device != x.device:
                    raise ValueError(f"rope {nm} must be a contiguous fp32 [N, d/2] tensor on x's device")
            st = _lib().fa_quant_fp8_rope(x.data_ptr(), x8.data_ptr(), ds.data_ptr(), B, H, N, d,
                                          cos.data_ptr(), sin.data_ptr(), int(layout), sp,
                                          int(bool(per_tensor)), ws, _stream(x))
            name = "fa_quant_fp8_rope"
    _check(st, name)
    del keep
    return x8, ds


def quant_fp8_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, signs=None, out=None):
    """The FP8 inputs of one attention call (``fa_quant_fp8_qkv``): Q and K
    with block scales after the rotation given by ``signs`` (or none), V with
    block scales, the three on internal streams joined back into the current
    stream.  q: fp32 [B, Hq, Nq, d]; k, v: fp32 [B, Hkv, Nk, d].  Returns
    (q8, k8, v8, q_descale, k_descale, v_descale), each as ``quant_fp8``
    would give it; ``out`` may supply those six tensors (written in place)."""
    for nm, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 or t.dim() != 4 \
                or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{nm} must be a contiguous fp32 [B, H, N, d] CUDA tensor on q's device")
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or dk != d:
        raise ValueError("k and v must be [B, Hkv, Nk, d] with q's B and d")
    shapes_ds = [(B, Hq, (Nq + FP8_BLOCK_ROWS - 1) // FP8_BLOCK_ROWS)] + \
                [(B, Hkv, (Nk + FP8_BLOCK_ROWS - 1) // FP8_BLOCK_ROWS)] * 2
    if out is None:
        outs = [torch.empty(t.shape, dtype=torch.uint8, device=q.device) for t in (q, k, v)]
        ds = [torch.empty(sh, dtype=torch.float32, device=q.device) for sh in shapes_ds]
    else:
        outs, ds = list(out[:3]), list(out[3:])
        for t, ref in zip(outs, (q, k, v)):
            if t.dtype != torch.uint8 or tuple(t.shape) != tuple(ref.shape) or not t.is_contiguous() \
                    or t.device != q.device:
                raise ValueError("code outputs must be contiguous uint8 tensors shaped like q, k, v")
        for t, sh in zip(ds, shapes_ds):
            if t.dtype != torch.float32 or tuple(t.shape) != sh or not t.is_contiguous() or t.device != q.device:
                raise ValueError(f"descale outputs must be contiguous fp32 {sh}")
    sp = None
    keep = None
    if signs is not None:
        keep = (ctypes.c_int8 * d)(*[int(s) for s in (signs.tolist() if hasattr(signs, "tolist") else signs)])
        sp = ctypes.cast(keep, ctypes.c_void_p)
    with torch.cuda.device(q.device):
        st = _lib().fa_quant_fp8_qkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), *[t.data_ptr() for t in outs],
                                     *[t.data_ptr() for t in ds], B, Hq, Hkv, Nq, Nk, d, sp, _stream(q))
    _check(st, "fa_quant_fp8_qkv")
    del keep
    return outs[0], outs[1], outs[2], ds[0], ds[1], ds[2]


def quant_fp8_per_tensor_noalloc(x: torch.Tensor, signs=None, x8: torch.Tensor | None = None,
                                 descale: torch.Tensor | None = None):
    """Per-tensor FP8 quantisation through ``fa_quant_fp8_per_tensor_noalloc``:
    the library uses its own static device scratch, so the call itself needs
    no allocation (pass ``x8`` and ``descale`` to avoid torch allocating the
    outputs too).  Same result as ``quant_fp8(x, signs, per_tensor=True)``.
    Calls that overlap on the GPU share the scratch and race."""
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32 or x.dim() != 4 \
            or not x.is_contiguous():
        raise ValueError("x must be a contiguous fp32 [B, H, N, d] CUDA tensor")
    B, H, N, d = x.shape
    nblk = (N + FP8_BLOCK_ROWS - 1) // FP8_BLOCK_ROWS
    if x8 is None:
        x8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
    if descale is None:
        descale = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device)
    keep = None
    sp = None
    if signs is not None:
        keep = (ctypes.c_int8 * d)(*[int(s) for s in (signs.tolist() if hasattr(signs, "tolist") else signs)])
        sp = ctypes.cast(keep, ctypes.c_void_p)
    with torch.cuda.device(x.device):
        st = _lib().fa_quant_fp8_per_tensor_noalloc(x.data_ptr(), x8.data_ptr(), descale.data_ptr(),
                                                    B, H, N, d, sp, _stream(x))
    _check(st, "fa_quant_fp8_per_tensor_noalloc")
    del keep
    return x8, descale


def check_device_error(device=None):
    """Synchronise the current stream and raise FaError if a kernel reported
    a pipeline timeout since the last check."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = _lib().fa_check_device_error(torch.cuda.current_stream(dev).cuda_stream)
    _check(st, "fa_check_device_error")
