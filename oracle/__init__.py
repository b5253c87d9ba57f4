"""Oracle for the exact attention forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product path (the CUDA library in
``exact_attention_forward_09_gb300``) never imports it, and it never imports
the product: the two share no code, header, table or constant.  The one
module both sides use is ``attn_inputs`` (seeded input generators, no
attention arithmetic).

Functions and the passages they follow:

* :func:`attn_fwd` -- plain fp64 scaled dot-product attention (materialised
  row of scores, two-pass softmax) with the row log-sum-exp.  Definition of
  attention: wmrh.cn FlashAttention V3 article, sec. 1.1; the tiled online
  softmax reaches exactly this result: same article sec. 2.1 and
  "FlashAttention-3: async pipelines on Hopper", section "Online Softmax is
  still the core of exact merging".
* :func:`attn_bwd` -- fp64 gradients dQ, dK, dV of sum(dO * O): the
  derivative of the same definition, one query row at a time with its row of
  probabilities materialised.  The pages name the backward pass among the
  paths to test ("FlashAttention-3: async pipelines on Hopper", section
  "correctness validation must cover asynchronous boundaries") but print no
  formula.
* :func:`online_attn_fwd` -- the tiled online-softmax recurrence itself
  (running max m, running sum l, accumulator o, initial m=-inf, l=0, o=0;
  wmrh.cn article sec. 2.1), with an optional lazy-rescale threshold.  Kept
  as a self-check of :func:`attn_fwd`, in fp64.
* :func:`quant_e4m3` -- per-128-row-block FP8 E4M3 quantisation, scale =
  amax/448, optional random-sign Hadamard rotation (sections "why block
  quantization beats a per-tensor scale" and "how incoherent processing
  flattens outliers" of "FlashAttention-3: async pipelines on Hopper"; the
  constant 448 from the wmrh.cn article sec. 3.3).  fp32 arithmetic, as the
  code decision is taken in the kernel's precision.
  With ``rope`` given, each row first gets a rotary position embedding in
  the same fp32 arithmetic as the kernel (the pages let RoPE share that
  pass, same two sections; they give no RoPE formula, so it is the usual
  planar rotation of channel pairs by the caller's angles).
* :func:`rope` -- the same rotary embedding in fp64, written as the
  rotation it is (per pair: [[cos, -sin], [sin, cos]] applied to (a, b)),
  for the attention-level checks.
* :func:`e4m3_encode` / :func:`e4m3_decode` -- the E4M3 format.
* :func:`hadamard_signs` is NOT here: random signs are inputs, drawn by
  ``attn_inputs``.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, f64, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_int
        vp = ctypes.c_void_p
        lib.oracle_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                        i32, f64, vp, i64, i32]
        lib.oracle_attn_fwd.restype = i32
        lib.oracle_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                        i32, f64, i32]
        lib.oracle_attn_bwd.restype = i32
        lib.oracle_quant_e4m3.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, i32, vp, vp, i32]
        lib.oracle_quant_e4m3.restype = i32
        lib.oracle_e4m3_encode_array.argtypes = [vp, vp, i64]
        lib.oracle_e4m3_encode_array.restype = None
        lib.oracle_e4m3_decode_array.argtypes = [vp, vp, i64]
        lib.oracle_e4m3_decode_array.restype = None
        lib.oracle_fwht_f32.argtypes = [vp, vp, i64, vp]
        lib.oracle_fwht_f32.restype = None
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        _LIB = lib
    return _LIB


def _np(x, dtype):
    """Host array of the given dtype, contiguous.  Accepts numpy or CPU torch."""
    if hasattr(x, "detach"):  # torch tensor
        import torch
        t = x.detach().cpu()
        if dtype == np.float64:
            t = t.to(torch.float64)
        elif dtype == np.float32:
            t = t.to(torch.float32)
        x = t.contiguous().numpy()
    return np.ascontiguousarray(x, dtype=dtype)


def max_threads() -> int:
    return int(_lib().oracle_max_threads())


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, rows=None,
             nthreads: int | None = None):
    """fp64 attention forward.

    q: [B, Hq, Nq, d]; k, v: [B, Hkv, Nk, d] (numpy or CPU torch, any float
    dtype; converted exactly to fp64).  Query head h reads K/V head
    h // (Hq // Hkv).  Causal: key j visible to query i iff j <= i + Nk - Nq.
    rows: optional 1-D list of query indices to compute (same for every head).

    Returns (o [B, Hq, R, d] fp64, lse [B, Hq, R] fp64), R = len(rows) or Nq.
    """
    q = _np(q, np.float64)
    k = _np(k, np.float64)
    v = _np(v, np.float64)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    assert v.shape == k.shape and Bk == B and dk == d and Hq % Hkv == 0
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rows_arr = None
    R = Nq
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        assert rows_arr.ndim == 1 and (rows_arr.size == 0 or
                                       (rows_arr.min() >= 0 and rows_arr.max() < Nq))
        R = rows_arr.size
    o = np.zeros((B, Hq, R, d), dtype=np.float64)
    lse = np.zeros((B, Hq, R), dtype=np.float64)
    nt = nthreads if nthreads is not None else max_threads()
    rc = _lib().oracle_attn_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                o.ctypes.data, lse.ctypes.data,
                                B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale),
                                rows_arr.ctypes.data if rows_arr is not None else None,
                                R, int(nt))
    if rc != 0:
        raise RuntimeError("oracle_attn_fwd failed")
    return o, lse


def attn_bwd(q, k, v, dout, causal: bool = False, scale: float | None = None,
             nthreads: int | None = None):
    """fp64 gradients of sum(dout * O) for O = attention(q, k, v).

    Shapes and masking as :func:`attn_fwd`; dout has q's shape.  Returns
    (dq [B, Hq, Nq, d], dk [B, Hkv, Nk, d], dv [B, Hkv, Nk, d]) in fp64;
    dk and dv sum over the query heads of each key/value group.
    """
    q = _np(q, np.float64)
    k = _np(k, np.float64)
    v = _np(v, np.float64)
    dout = _np(dout, np.float64)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk_ = k.shape
    assert v.shape == k.shape and Bk == B and dk_ == d and Hq % Hkv == 0
    assert dout.shape == q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = np.zeros(q.shape, dtype=np.float64)
    dk = np.zeros(k.shape, dtype=np.float64)
    dv = np.zeros(k.shape, dtype=np.float64)
    nt = nthreads if nthreads is not None else max_threads()
    rc = _lib().oracle_attn_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data,
                                dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
                                B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), float(scale), int(nt))
    if rc != 0:
        raise RuntimeError("oracle_attn_bwd failed")
    return dq, dk, dv


def online_attn_fwd(q, k, v, causal: bool = False, scale: float | None = None,
                    tile: int = 128, tau: float = 0.0):
    """The tiled online-softmax recurrence, fp64 (self-check of attn_fwd).

    Keys are visited in tiles of ``tile`` rows.  State per query row: m (the
    reference maximum), l (sum of exp(s - m)), o (sum of exp(s - m) v), with
    m = -inf, l = 0, o = 0 at the start; after the last tile O = o / l.
    With tau > 0 the reference maximum is only moved when the tile maximum
    exceeds it by more than tau (natural-log units); o, l and m stay
    consistent, so the result is the same.
    """
    q = _np(q, np.float64)
    k = _np(k, np.float64)
    v = _np(v, np.float64)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    g = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O = np.zeros((B, Hq, Nq, d))
    L = np.zeros((B, Hq, Nq))
    qi_idx = np.arange(Nq)[:, None]
    for b in range(B):
        for h in range(Hq):
            Q = q[b, h]
            K = k[b, h // g]
            V = v[b, h // g]
            m = np.full(Nq, -np.inf)
            l = np.zeros(Nq)
            o = np.zeros((Nq, d))
            for j0 in range(0, Nk, tile):
                j1 = min(j0 + tile, Nk)
                s = scale * (Q @ K[j0:j1].T)
                if causal:
                    kj = np.arange(j0, j1)[None, :]
                    s = np.where(kj <= qi_idx + (Nk - Nq), s, -np.inf)
                tmax = s.max(axis=1)
                m_new = np.where(tmax > m + tau, np.maximum(m, tmax), m)
                with np.errstate(invalid="ignore"):
                    alpha = np.where(np.isneginf(m_new), 1.0, np.exp(m - m_new))
                    p = np.where(np.isneginf(s), 0.0, np.exp(s - m_new[:, None]))
                l = alpha * l + p.sum(axis=1)
                o = alpha[:, None] * o + p @ V[j0:j1]
                m = m_new
            with np.errstate(invalid="ignore", divide="ignore"):
                O[b, h] = np.where(l[:, None] > 0, o / np.where(l > 0, l, 1.0)[:, None], 0.0)
                L[b, h] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return O, L


def e4m3_encode(x) -> np.ndarray:
    x = _np(x, np.float32)
    c = np.empty(x.shape, dtype=np.uint8)
    _lib().oracle_e4m3_encode_array(x.ctypes.data, c.ctypes.data, x.size)
    return c


def e4m3_decode(c) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(c, dtype=np.uint8))
    x = np.empty(c.shape, dtype=np.float32)
    _lib().oracle_e4m3_decode_array(c.ctypes.data, x.ctypes.data, c.size)
    return x


def fwht_f32(x, signs=None) -> np.ndarray:
    """H_d (signs o x) along the last axis with the fp32 butterfly (no 1/sqrt(d))."""
    x = _np(x, np.float32)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    out = np.empty_like(flat)
    sg = None
    if signs is not None:
        sg = np.ascontiguousarray(np.asarray(signs, dtype=np.int8))
        assert sg.shape == (d,)
    for r in range(flat.shape[0]):
        _lib().oracle_fwht_f32(flat[r].ctypes.data, out[r].ctypes.data, d,
                               sg.ctypes.data if sg is not None else None)
    return out.reshape(x.shape)


ROPE_INTERLEAVED, ROPE_HALF = 1, 2   # channel pairs (2i, 2i+1) / (i, i + d/2)


def rope(x, cos, sin, layout) -> np.ndarray:
    """Rotary embedding of x [..., N, d] in fp64: for every row n and pair
    index i < d/2, the channel pair (a, b) -- (2i, 2i+1) for ROPE_INTERLEAVED,
    (i, i + d/2) for ROPE_HALF -- is multiplied by the 2x2 rotation
    [[cos[n, i], -sin[n, i]], [sin[n, i], cos[n, i]]]."""
    x = _np(x, np.float64)
    cos = _np(cos, np.float64)
    sin = _np(sin, np.float64)
    d = x.shape[-1]
    half = d // 2
    if layout == ROPE_INTERLEAVED:
        ia, ib = np.arange(half) * 2, np.arange(half) * 2 + 1
    elif layout == ROPE_HALF:
        ia, ib = np.arange(half), np.arange(half) + half
    else:
        raise ValueError("unknown rope layout")
    a, b = x[..., ia], x[..., ib]
    out = np.empty_like(x)
    out[..., ia] = cos * a - sin * b
    out[..., ib] = sin * a + cos * b
    return out


def quant_e4m3(x, signs=None, per_tensor: bool = False, block_rows: int = 128, rope=None):
    """Quantise x [B, H, N, d] fp32 to E4M3 codes + descale [B, H, ceil(N/block_rows)].

    dequantised value = decode(code) * descale; with rotation on (signs given)
    that approximates x diag(signs) H_d / sqrt(d).  ``rope``: None or
    (cos, sin, layout) with fp32 tables [N, d/2]: the rotary embedding is
    applied to every row first, in fp32.
    """
    x = _np(x, np.float32)
    B, H, N, d = x.shape
    nblk = (N + block_rows - 1) // block_rows
    codes = np.empty(x.shape, dtype=np.uint8)
    descale = np.empty((B, H, nblk), dtype=np.float32)
    sg = None
    if signs is not None:
        sg = np.ascontiguousarray(np.asarray(signs, dtype=np.int8))
        assert sg.shape == (d,)
    cos_ptr, sin_ptr, layout = None, None, 0
    keep = None
    if rope is not None:
        tcos, tsin, layout = rope
        tcos = np.ascontiguousarray(_np(tcos, np.float32))
        tsin = np.ascontiguousarray(_np(tsin, np.float32))
        assert tcos.shape == (N, d // 2) and tsin.shape == (N, d // 2)
        keep = (tcos, tsin)
        cos_ptr, sin_ptr = tcos.ctypes.data, tsin.ctypes.data
    rc = _lib().oracle_quant_e4m3(x.ctypes.data, codes.ctypes.data, descale.ctypes.data,
                                  B * H, N, d, block_rows,
                                  sg.ctypes.data if sg is not None else None, int(bool(per_tensor)),
                                  cos_ptr, sin_ptr, int(layout))
    del keep
    if rc != 0:
        raise RuntimeError("oracle_quant_e4m3 failed")
    return codes, descale


def dequant_e4m3(codes, descale, block_rows: int = 128) -> np.ndarray:
    """decode(code) * descale of its block, fp64 [B, H, N, d]."""
    vals = e4m3_decode(codes).astype(np.float64)
    B, H, N, d = vals.shape
    ds = np.repeat(np.asarray(descale, dtype=np.float64), block_rows, axis=2)[:, :, :N]
    return vals * ds[..., None]


def rotate(x, signs) -> np.ndarray:
    """x diag(signs) H_d / sqrt(d) along the last axis, fp64, from the dense
    Sylvester matrix (H[i, j] = (-1)^popcount(i & j))."""
    x = _np(x, np.float64)
    d = x.shape[-1]
    idx = np.arange(d)
    Hd = np.array([[(-1.0) ** bin(i & j).count("1") for j in idx] for i in idx])
    M = np.diag(np.asarray(signs, dtype=np.float64)) @ Hd / math.sqrt(d)
    return x @ M
