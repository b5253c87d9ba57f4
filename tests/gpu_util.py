"""Shared helpers for the GPU parity tests: seeded inputs, the oracle on the
exact values the GPU saw, and the error metrics."""
from __future__ import annotations

import math

import numpy as np
import torch

import attn_inputs as gen
import oracle

# tolerances for BF16/FP16 on N(0,1) inputs, against the fp64 oracle
O_MAXABS = 1e-2
O_RMSE = 2e-3
LSE_ABS = 1e-3
# FP8 (vs the oracle on the unquantised fp32 inputs)
FP8_O_RMSE = 3e-2


def make_qkv(B, H, N, d, seed, dtype=torch.bfloat16, device="cuda"):
    """Seeded N(0,1) Q, K, V rounded to `dtype`; returns (host fp64 views, device tensors)."""
    q, k, v = gen.qkv_normal((B, H, N, d), seed)
    host = [torch.from_numpy(a).to(dtype) for a in (q, k, v)]
    dev = [t.to(device) for t in host]
    return host, dev


def oracle_rows(host, causal, scale, rows=None):
    """Oracle on the exact low-precision values (converted to fp64), one head
    at a time to bound memory."""
    q, k, v = host
    B, H, N, d = q.shape
    R = N if rows is None else len(rows)
    O = np.empty((B, H, R, d))
    L = np.empty((B, H, R))
    for b in range(B):
        for h in range(H):
            o, l = oracle.attn_fwd(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1],
                                   causal=causal, scale=scale, rows=rows)
            O[b, h] = o[0, 0]
            L[b, h] = l[0, 0]
    return O, L


def errors(o_gpu, lse_gpu, o_ref, lse_ref, rows=None):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        o = o[:, :, rows]
        lse = lse[:, :, rows]
    diff = o - o_ref
    return dict(o_maxabs=float(np.abs(diff).max()) if diff.size else 0.0,
                o_rmse=float(math.sqrt((diff ** 2).mean())) if diff.size else 0.0,
                lse_maxabs=float(np.abs(lse - lse_ref).max()) if lse.size else 0.0,
                finite=bool(np.isfinite(o).all() and np.isfinite(lse).all()))


def assert_bf16_parity(err, what=""):
    assert err["finite"], f"{what}: non-finite output"
    assert err["o_maxabs"] <= O_MAXABS, f"{what}: O max-abs {err['o_maxabs']:.3e} > {O_MAXABS}"
    assert err["o_rmse"] <= O_RMSE, f"{what}: O RMSE {err['o_rmse']:.3e} > {O_RMSE}"
    assert err["lse_maxabs"] <= LSE_ABS, f"{what}: LSE max-abs {err['lse_maxabs']:.3e} > {LSE_ABS}"


def assert_bf16_bound(o_gpu, o_ref, v_absmax, what=""):
    """Element-wise bound for inputs outside N(0,1), derived from the
    arithmetic: P is rounded to bf16 before P V (relative 2^-9 per weight, at
    most 2^-9 * max|V| on O), O is rounded to bf16 on output (2^-9 * |O|), and
    the fp32 accumulation adds far less.  Twice that, plus 1e-4."""
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -8 * (np.abs(o_ref) + v_absmax) + 1e-4
    bad = np.abs(o - o_ref) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside the derived bound; worst excess " \
                          f"{float((np.abs(o - o_ref) - tol).max()):.3e}"


# unit roundoff of the backward's element types
BWD_UNIT = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


def bwd_check(got, ref, dtype, what):
    """Backward errors normalised by the reference: the largest error within
    2.5 u of the largest |reference| entry, the rms error within 1.25 u of
    the reference's rms (u the element type's unit roundoff)."""
    u = BWD_UNIT[dtype]
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        g = g.float().cpu().numpy().astype(np.float64)
        assert g.shape == r.shape, f"{what} {name}: shape"
        assert np.isfinite(g).all(), f"{what} {name}: non-finite values"
        if r.size == 0:
            continue
        e = g - r
        rmax = np.abs(r).max()
        rrms = math.sqrt((r ** 2).mean())
        if rmax == 0.0:
            # an exactly zero gradient (a single key: dS = 0) comes out as
            # fp32 rounding residue of P (dP - D)
            assert np.abs(g).max() <= 1e-5, f"{what} {name}: expected zeros, got {np.abs(g).max():.3e}"
            continue
        assert np.abs(e).max() <= 2.5 * u * rmax, f"{what} {name}: max error {np.abs(e).max() / rmax:.3e} of max|ref|"
        assert math.sqrt((e ** 2).mean()) <= 1.25 * u * rrms, \
            f"{what} {name}: rms error {math.sqrt((e ** 2).mean()) / rrms:.3e} of rms(ref)"
