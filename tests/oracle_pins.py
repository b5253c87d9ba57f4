"""Pins for the oracle: checks against facts the pages and the mathematics
fix, never against the oracle's own formula.

Each ``pin_*`` function raises AssertionError when the oracle disagrees.  They
are collected by ``test_oracle_pins.py`` and re-run against planted mistakes
by ``test_oracle_mutants.py``.

Sources of truth used here:
  * torch's CPU float64 ``scaled_dot_product_attention`` and ``logsumexp``
    (independent library implementations of the definition);
  * closed forms: Q = 0 gives the mean of the visible V rows and LSE = ln(count);
    a causal row 0 is V[0] with LSE = scale q0.k0; scale 0 gives the mean;
    a single key gives that V row; joint permutations of K/V rows (non-causal)
    leave O unchanged;
  * invariance under a shared orthogonal rotation of Q and K ("FlashAttention-3:
    async pipelines on Hopper", section "how incoherent processing flattens
    outliers": scores are unchanged in exact arithmetic), with the Hadamard
    matrix from scipy;
  * the tiled online recurrence equals the two-pass result (wmrh.cn article,
    sec. 2.1: the tiled result is the same as the global one);
  * torch.float8_e4m3fn for the E4M3 codec, and 448 as its maximum (wmrh.cn
    article, sec. 3.3); exact rational arithmetic (``fractions``) and a brute
    force search of torch's E4M3 grid for the quantiser's rounding of y / s
    next to E4M3 midpoints, and torch's fp32 division and float8 cast where
    the scale is a power of two (the quotient is then exact in fp32);
  * for the backward pass: torch autograd through CPU float64 SDPA, central
    finite differences of the pinned forward, and the sums fixed by the
    softmax (rows of dS sum to zero, rows of P to one);
  * for the rotary embedding (which the pages only place before the
    quantisation pass): complex multiplication of each channel pair by
    e^{i theta} (numpy complex arithmetic), the permutation relating the two
    channel pairings, and the relative-position property of the scores.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import scipy.linalg
import torch

import attn_inputs as gen

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "pages_constants.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _torch_ref(q, k, v, causal, scale):
    """torch CPU float64 SDPA with an explicit bottom-right causal mask, plus
    torch.logsumexp of the scaled masked scores."""
    q = torch.as_tensor(np.asarray(q, dtype=np.float64))
    k = torch.as_tensor(np.asarray(k, dtype=np.float64))
    v = torch.as_tensor(np.asarray(v, dtype=np.float64))
    Hq, Hkv = q.shape[1], k.shape[1]
    if Hq != Hkv:
        k = k.repeat_interleave(Hq // Hkv, dim=1)
        v = v.repeat_interleave(Hq // Hkv, dim=1)
    Nq, Nk = q.shape[2], k.shape[2]
    mask = None
    if causal:
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nk)[None, :]
        mask = j <= i + (Nk - Nq)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=scale)
    s = scale * (q @ k.transpose(-1, -2))
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    return o.numpy(), lse.numpy()


def _sylvester(d):
    return scipy.linalg.hadamard(d).astype(np.float64)


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def pin_library_cross_check(oracle):
    cases = [
        # (B, Hq, Hkv, Nq, Nk, d, causal, scale)
        (1, 2, 2, 128, 128, 64, False, 1 / 8),
        (1, 2, 2, 128, 128, 64, True, 1 / 8),
        (2, 4, 2, 37, 37, 16, True, 0.3),
        (1, 3, 1, 20, 50, 8, True, 0.5),
        (1, 2, 2, 50, 20, 8, False, -0.7),
    ]
    for t, (B, Hq, Hkv, Nq, Nk, d, causal, scale) in enumerate(cases):
        q = gen.normal((B, Hq, Nq, d), 10 + t, 0).astype(np.float64)
        k = gen.normal((B, Hkv, Nk, d), 10 + t, 1).astype(np.float64)
        v = gen.normal((B, Hkv, Nk, d), 10 + t, 2).astype(np.float64)
        o, lse = oracle.attn_fwd(q, k, v, causal=causal, scale=scale)
        o_ref, lse_ref = _torch_ref(q, k, v, causal, scale)
        assert np.allclose(o, o_ref, rtol=0, atol=1e-12), f"case {t}: O differs from torch SDPA"
        assert np.allclose(lse, lse_ref, rtol=0, atol=1e-12), f"case {t}: LSE differs from torch.logsumexp"


def pin_zero_query(oracle):
    B, H, N, d = 1, 2, 96, 32
    k = gen.normal((B, H, N, d), 20, 1).astype(np.float64)
    v = gen.normal((B, H, N, d), 20, 2).astype(np.float64)
    q = np.zeros((B, H, N, d))
    o, lse = oracle.attn_fwd(q, k, v, causal=False, scale=0.125)
    assert np.allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-13)
    assert np.allclose(lse, math.log(N), atol=1e-13)
    o, lse = oracle.attn_fwd(q, k, v, causal=True, scale=0.125)
    prefix = np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
    assert np.allclose(o, prefix, atol=1e-13)
    assert np.allclose(lse, np.log(np.arange(1, N + 1))[None, None, :], atol=1e-13)


def pin_causal_row0(oracle):
    B, H, N, d = 2, 2, 64, 16
    q, k, v = (a.astype(np.float64) for a in gen.qkv_normal((B, H, N, d), 21))
    scale = 0.37
    o, lse = oracle.attn_fwd(q, k, v, causal=True, scale=scale)
    assert np.array_equal(o[:, :, 0, :], v[:, :, 0, :]), "causal row 0 must be V[0] exactly"
    expect = scale * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
    assert np.allclose(lse[:, :, 0], expect, atol=1e-13)


def pin_special_cases(oracle):
    B, H, N, d = 1, 1, 33, 8
    q, k, v = (a.astype(np.float64) for a in gen.qkv_normal((B, H, N, d), 22))
    # scale 0: uniform weights
    o, lse = oracle.attn_fwd(q, k, v, causal=False, scale=0.0)
    assert np.allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-13)
    assert np.allclose(lse, math.log(N), atol=1e-13)
    # a single key
    o, lse = oracle.attn_fwd(q, k[:, :, :1], v[:, :, :1], causal=False, scale=0.5)
    assert np.allclose(o, np.broadcast_to(v[:, :, :1], o.shape), atol=1e-15)
    assert np.allclose(lse, 0.5 * (q[0, 0] @ k[0, 0, 0])[None, None, :], atol=1e-13)
    # joint permutation of K/V rows
    perm = np.random.Generator(np.random.PCG64(5)).permutation(N)
    o1, l1 = oracle.attn_fwd(q, k, v, scale=0.3)
    o2, l2 = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], scale=0.3)
    assert np.allclose(o1, o2, atol=1e-13) and np.allclose(l1, l2, atol=1e-13)
    # one dominant key: the output is that key's value row
    kk = np.zeros((1, 1, 4, 2))
    kk[0, 0, :, 0] = [0.0, 1.0, 2.0, 3.0]
    vv = np.arange(8, dtype=np.float64).reshape(1, 1, 4, 2)
    qq = np.array([[[[1.0, 0.0]]]])
    o, lse = oracle.attn_fwd(qq, kk, vv, scale=200.0)
    assert np.allclose(o[0, 0, 0], vv[0, 0, 3], atol=1e-12)
    assert abs(lse[0, 0, 0] - 600.0) < 1e-12


def pin_rotation_invariance(oracle):
    B, H, N, d = 1, 2, 40, 32
    q, k, v = (a.astype(np.float64) for a in gen.qkv_normal((B, H, N, d), 23))
    signs = gen.hadamard_signs(d, 7).astype(np.float64)
    M = np.diag(signs) @ _sylvester(d) / math.sqrt(d)
    assert np.allclose(M @ M.T, np.eye(d), atol=1e-14)
    for causal in (False, True):
        o1, l1 = oracle.attn_fwd(q, k, v, causal=causal, scale=0.2)
        o2, l2 = oracle.attn_fwd(q @ M, k @ M, v, causal=causal, scale=0.2)
        assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)


def pin_online_recurrence(oracle):
    B, Hq, Hkv, N, d = 1, 2, 1, 300, 16
    q = gen.normal((B, Hq, N, d), 24, 0).astype(np.float64) * 2.0
    k = gen.normal((B, Hkv, N, d), 24, 1).astype(np.float64)
    v = gen.normal((B, Hkv, N, d), 24, 2).astype(np.float64)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal=causal, scale=0.5)
        for tile in (1, 7, 128, N):
            for tau in (0.0, 8.0 * math.log(2.0)):
                o2, l2 = oracle.online_attn_fwd(q, k, v, causal=causal, scale=0.5, tile=tile, tau=tau)
                assert np.allclose(o, o2, rtol=0, atol=1e-12), (causal, tile, tau)
                assert np.allclose(lse, l2, rtol=0, atol=1e-12), (causal, tile, tau)


def pin_row_subset(oracle):
    B, H, N, d = 1, 2, 200, 16
    q, k, v = (a.astype(np.float64) for a in gen.qkv_normal((B, H, N, d), 25))
    rows = gen.sample_rows(N, 20, 1)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal=causal, scale=0.25)
        os_, ls_ = oracle.attn_fwd(q, k, v, causal=causal, scale=0.25, rows=rows)
        assert np.array_equal(o[:, :, rows], os_) and np.array_equal(lse[:, :, rows], ls_)


# --------------------------------------------------------------------------
# backward pass
# --------------------------------------------------------------------------

def _torch_grads(q, k, v, do, causal, scale):
    """dQ, dK, dV of sum(do * O) by torch autograd through CPU float64 SDPA
    (bottom-right causal mask; K/V heads repeated for grouped queries, so
    autograd sums the group's contributions)."""
    qt, kt, vt = (torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True) for a in (q, k, v))
    Hq, Hkv = qt.shape[1], kt.shape[1]
    kr = kt.repeat_interleave(Hq // Hkv, dim=1) if Hq != Hkv else kt
    vr = vt.repeat_interleave(Hq // Hkv, dim=1) if Hq != Hkv else vt
    Nq, Nk = qt.shape[2], kt.shape[2]
    mask = None
    if causal:
        mask = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kr, vr, attn_mask=mask, scale=scale)
    o.backward(torch.tensor(np.asarray(do, dtype=np.float64)))
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def _bwd_inputs(shape_q, shape_k, seed):
    q = gen.normal(shape_q, seed, 0).astype(np.float64)
    k = gen.normal(shape_k, seed, 1).astype(np.float64)
    v = gen.normal(shape_k, seed, 2).astype(np.float64)
    do = gen.normal(shape_q, seed, 3).astype(np.float64)
    return q, k, v, do


def pin_bwd_autograd(oracle):
    cases = [
        # (B, Hq, Hkv, Nq, Nk, d, causal, scale)
        (1, 2, 2, 64, 64, 16, False, 0.25),
        (1, 2, 2, 64, 64, 16, True, 0.25),
        (2, 4, 2, 37, 37, 8, True, 0.6),
        (1, 3, 1, 20, 50, 8, True, 0.5),
        (1, 2, 2, 50, 20, 8, False, -0.7),
    ]
    for t, (B, Hq, Hkv, Nq, Nk, d, causal, scale) in enumerate(cases):
        q, k, v, do = _bwd_inputs((B, Hq, Nq, d), (B, Hkv, Nk, d), 30 + t)
        got = oracle.attn_bwd(q, k, v, do, causal=causal, scale=scale)
        ref = _torch_grads(q, k, v, do, causal, scale)
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert np.allclose(g, r, rtol=0, atol=1e-11), f"case {t}: {name} differs from torch autograd"


def pin_bwd_finite_difference(oracle):
    """Directional derivatives of L = sum(dO * O), with O from the (separately
    pinned) forward oracle, by central differences."""
    B, Hq, Hkv, N, d = 1, 2, 1, 24, 8
    q, k, v, do = _bwd_inputs((B, Hq, N, d), (B, Hkv, N, d), 40)
    rng = np.random.Generator(np.random.PCG64(41))
    for causal in (False, True):
        grads = oracle.attn_bwd(q, k, v, do, causal=causal, scale=0.4)

        def loss(qq, kk, vv):
            o, _ = oracle.attn_fwd(qq, kk, vv, causal=causal, scale=0.4)
            return float(np.sum(do * o))

        h = 1e-5
        for which in range(3):
            x = [q, k, v]
            u = rng.standard_normal(x[which].shape)
            xp = list(x)
            xm = list(x)
            xp[which] = x[which] + h * u
            xm[which] = x[which] - h * u
            fd = (loss(*xp) - loss(*xm)) / (2 * h)
            an = float(np.sum(grads[which] * u))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (causal, which, fd, an)


def pin_bwd_invariants(oracle):
    B, Hq, Hkv, N, d = 1, 4, 2, 40, 8
    q, k, v, do = _bwd_inputs((B, Hq, N, d), (B, Hkv, N, d), 50)
    g = Hq // Hkv
    for causal in (False, True):
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=causal, scale=0.3)
        # each row of dS sums to zero, so the key gradients sum to zero
        assert np.allclose(dk.sum(axis=2), 0.0, atol=1e-12)
        # each row of P sums to one, so the value gradients sum to sum(dO)
        want = do.reshape(B, Hkv, g, N, d).sum(axis=(2, 3))
        assert np.allclose(dv.sum(axis=2), want, atol=1e-12)
    # scale 0: uniform weights, no gradient into Q or K
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=False, scale=0.0)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0
    want = do.reshape(B, Hkv, g, N, d).sum(axis=(2, 3))[:, :, None, :] / N
    assert np.allclose(dv, np.broadcast_to(want, dv.shape), atol=1e-13)
    # causal, scale 0: row i spreads dO_i evenly over keys 0..i
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=True, scale=0.0)
    w = do.reshape(B, Hkv, g, N, d).sum(axis=2) / np.arange(1, N + 1)[None, None, :, None]
    want = np.cumsum(w[:, :, ::-1], axis=2)[:, :, ::-1]
    assert np.allclose(dv, want, atol=1e-13)
    # a single key: P = 1, so dS = 0 and dV_0 = sum of dO
    dq, dk, dv = oracle.attn_bwd(q, k[:, :, :1], v[:, :, :1], do, causal=False, scale=0.7)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    assert np.allclose(dv[:, :, 0], do.reshape(B, Hkv, g, N, d).sum(axis=(2, 3)), atol=1e-12)
    # dO = 0: no gradient at all
    z = oracle.attn_bwd(q, k, v, np.zeros_like(do), causal=True, scale=0.3)
    assert all(np.abs(a).max() == 0.0 for a in z)


def pin_bwd_empty_rows(oracle):
    """Nq > Nk causal: the first Nq - Nk queries see no key; they get dQ = 0
    and add nothing, and the rest behave as the square problem (their masks
    are the same)."""
    B, H, Nq, Nk, d = 1, 2, 30, 18, 8
    q, k, v, do = _bwd_inputs((B, H, Nq, d), (B, H, Nk, d), 60)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, causal=True, scale=0.5)
    e = Nq - Nk
    assert np.abs(dq[:, :, :e]).max() == 0.0
    ref = _torch_grads(q[:, :, e:], k, v, do[:, :, e:], True, 0.5)
    assert np.allclose(dq[:, :, e:], ref[0], atol=1e-11)
    assert np.allclose(dk, ref[1], atol=1e-11) and np.allclose(dv, ref[2], atol=1e-11)


# --------------------------------------------------------------------------
# FP8 E4M3 codec, rotation and quantiser
# --------------------------------------------------------------------------

def pin_e4m3_decode(oracle):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = oracle.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.nanmax(got) == _golden()["e4m3_max"]["value"]


def pin_e4m3_encode(oracle):
    finite = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    grid = np.unique(np.abs(finite[np.isfinite(finite)]))
    mids = (grid[1:] + grid[:-1]) / 2.0            # exact ties
    rng = np.random.Generator(np.random.PCG64(9))
    vals = np.concatenate([grid, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
                           rng.uniform(-448, 448, 5000), rng.standard_normal(5000) * 1e-2,
                           rng.standard_normal(5000) * 1e-3]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(vals)
    assert np.array_equal(got, ref), "E4M3 encoding must match torch's round-to-nearest-even"
    # saturation at the largest finite value (satfinite)
    big = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, -1e30], dtype=np.float32)
    assert np.array_equal(oracle.e4m3_decode(oracle.e4m3_encode(big)),
                          np.array([448, 448, 448, 448, 448, 448, -448], dtype=np.float32))


def pin_fwht(oracle):
    for d in (8, 64, 128, 256):
        x = gen.normal((5, d), 30 + d)
        signs = gen.hadamard_signs(d, d)
        y = oracle.fwht_f32(x, signs).astype(np.float64)
        exact = (x.astype(np.float64) * signs) @ _sylvester(d).T
        bound = math.log2(d) * np.finfo(np.float32).eps * np.abs(x).astype(np.float64).sum(axis=1,
                                                                                           keepdims=True)
        assert np.all(np.abs(y - exact) <= bound + 1e-30), d
        M = np.diag(signs.astype(np.float64)) @ _sylvester(d) / math.sqrt(d)
        assert np.allclose(oracle.rotate(x, signs), x.astype(np.float64) @ M, atol=1e-12)


def pin_quantiser(oracle):
    rows = _golden()["quant_block_rows"]["value"]
    B, H, N, d = 1, 2, 300, 64                      # ragged last block (44 rows)
    x = gen.outliers((B, H, N, d), 40)
    signs = gen.hadamard_signs(d, 41)
    for sg in (None, signs):
        for per_tensor in (False, True):
            codes, ds = oracle.quant_e4m3(x, signs=sg, per_tensor=per_tensor, block_rows=rows)
            assert ds.shape == (B, H, 3)
            target = x.astype(np.float64) if sg is None else oracle.rotate(x, sg)
            deq = oracle.dequant_e4m3(codes, ds, block_rows=rows)
            # every block: the largest magnitude maps to +-448; error within half
            # an E4M3 step (relative 2^-4 for normals, 2^-10 * scale below)
            blocks = [(b, h, r0) for b in range(B) for h in range(H) for r0 in range(0, N, rows)]
            for (b, h, r0) in blocks:
                cb = codes[b, h, r0:r0 + rows]
                tb = target[b, h, r0:r0 + rows]
                db = deq[b, h, r0:r0 + rows]
                s = ds[b, h, r0 // rows]
                if not per_tensor:
                    mags = oracle.e4m3_decode(cb & 0x7F)
                    assert mags.max() == 448.0
                    amax = np.abs(tb).max()
                    assert abs(amax / 448.0 - s) <= 1e-6 * amax / 448.0
                err = np.abs(db - tb)
                tol = np.maximum(np.abs(tb) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-5)
                assert np.all(err <= tol)
            if per_tensor:
                assert np.all(ds == ds.flat[0])
                assert oracle.e4m3_decode(codes & 0x7F).max() == 448.0


def _e4m3_grid():
    """The non-negative finite E4M3 values, decoded by torch (ascending)."""
    vals = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return np.unique(np.abs(vals[np.isfinite(vals)]))


def _nearest_e4m3_code(q, grid, codes_of):
    """E4M3 code of the exact rational q: the nearest grid value, ties to the
    even code, saturated at the largest finite value (brute force)."""
    from fractions import Fraction
    a = abs(q)
    top = Fraction(float(grid[-1]))
    if a >= top:
        best = grid[-1]
    else:
        i = int(np.searchsorted(grid, float(a), side="right")) - 1
        while i + 1 < len(grid) and Fraction(float(grid[i + 1])) <= a:
            i += 1
        while i > 0 and Fraction(float(grid[i])) > a:
            i -= 1
        lo, hi = Fraction(float(grid[i])), Fraction(float(grid[i + 1]))
        dlo, dhi = a - lo, hi - a
        if dlo < dhi:
            best = grid[i]
        elif dhi < dlo:
            best = grid[i + 1]
        else:
            best = grid[i] if codes_of[float(grid[i])] % 2 == 0 else grid[i + 1]
    code = codes_of[float(best)]
    return code | (0x80 if q < 0 else 0)


def _near_midpoint_block(d=64, rows=128):
    """One block whose elements sit within a few fp32 ulps of s * m for E4M3
    midpoints m, with s = amax / 448 (fp32) not a power of two, plus its
    expected codes from exact rational arithmetic.  Also returns how many
    elements two other readings (y * RN(1/s) rounded to fp32 first, and the
    fp32 quotient RN(y / s) first) would encode differently, so that the pin
    is known to tell them apart."""
    from fractions import Fraction
    grid = _e4m3_grid()
    codes_of = {}
    for c in range(0x7F):
        v = float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64))
        codes_of.setdefault(v, c)
    amax = np.float32(1.7731) * np.float32(448.0)
    s = np.float32(amax) / np.float32(448.0)
    assert math.frexp(float(s))[0] != 0.5                            # not a power of two
    mids = (grid[1:] + grid[:-1]) / 2.0
    mids = mids[mids < 440.0]
    vals, exp_codes = [], []
    n_recip = n_div32 = 0
    r32 = np.float32(1.0) / s
    for m in mids:
        y0 = np.float32(float(Fraction(float(m)) * Fraction(float(s))))
        for k in range(-3, 4):
            y = y0
            for _ in range(abs(k)):
                y = np.nextafter(y, np.float32(np.inf if k > 0 else -np.inf), dtype=np.float32)
            for sgn in (1.0, -1.0):
                yy = np.float32(sgn * y)
                want = _nearest_e4m3_code(Fraction(float(yy)) / Fraction(float(s)), grid, codes_of)
                recip = _nearest_e4m3_code(Fraction(float(np.float32(yy * r32))), grid, codes_of)
                div32 = _nearest_e4m3_code(Fraction(float(np.float32(yy / s))), grid, codes_of)
                n_recip += recip != want
                n_div32 += div32 != want
                vals.append(yy)
                exp_codes.append(want)
    n = len(vals)
    assert n + 1 <= rows * d
    x = np.zeros(rows * d, dtype=np.float32)
    x[:n] = vals
    x[n] = amax                                     # the block's largest magnitude
    exp = np.zeros(rows * d, dtype=np.uint8)
    exp[:n] = exp_codes
    exp[n] = 0x7E
    exp[n + 1:] = 0                                 # +0 encodes to code 0
    return x.reshape(1, 1, rows, d), exp.reshape(1, 1, rows, d), float(s), n_recip, n_div32


def pin_quantiser_exact_rounding(oracle):
    # codes are the E4M3 value nearest to the exact quotient y / s (ties to
    # even), s = fp32(amax / 448): checked with rational arithmetic on values
    # crafted within a few ulps of s times every E4M3 midpoint, where rounding
    # y / s to fp32 first, or multiplying by a rounded reciprocal, would
    # change some codes
    x, exp, s, n_recip, n_div32 = _near_midpoint_block()
    assert n_recip > 0 and n_div32 > 0, "crafted block does not separate the readings"
    codes, ds = oracle.quant_e4m3(x, block_rows=128)
    assert ds.reshape(-1)[0] == np.float32(s)
    assert np.array_equal(codes, exp), f"{int((codes != exp).sum())} codes differ from exact rounding of y / s"


def pin_quantiser_power_of_two_scale(oracle):
    # with amax = 448 * 2^k the scale is exactly 2^k, so y / s is exact in
    # fp32 and torch's float8_e4m3fn cast of it is the single correct rounding
    rng = np.random.Generator(np.random.PCG64(71))
    for k in (-3, 0, 5):
        x = rng.standard_normal((1, 2, 128, 64)).astype(np.float32)
        for h in range(2):
            x[0, h] *= np.float32(448.0 * 2.0 ** k / 4.0) / np.abs(x[0, h]).max() * np.float32(0.999)
            x[0, h, 7, 3] = np.float32(448.0 * 2.0 ** k)
        codes, ds = oracle.quant_e4m3(x, block_rows=128)
        assert np.all(ds == np.float32(2.0 ** k))
        ref = (torch.from_numpy(x) / np.float32(2.0 ** k)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes, ref), k


def _rope_pairs(d, layout):
    half = d // 2
    if layout == 1:
        return np.arange(half) * 2, np.arange(half) * 2 + 1
    return np.arange(half), np.arange(half) + half


def pin_rope_complex(oracle):
    # a pair (a, b) read as a + ib, times e^{i theta}; a quarter turn maps
    # (1, 0) to (0, 1)
    one = np.zeros((1, 4))
    one[0, 0] = 1.0
    s90 = np.array([[1.0, 0.0]])
    y = oracle.rope(one, np.cos(np.pi / 2 * s90), np.sin(np.pi / 2 * s90), 1)
    assert np.allclose(y, [[0.0, 1.0, 0.0, 0.0]], atol=1e-15), y
    for layout in (1, 2):
        for d in (8, 64, 128):
            x = gen.normal((2, 3, 17, d), 50 + d).astype(np.float64)
            theta = gen.normal((17, d // 2), 51 + d).astype(np.float64) * 3.0
            y = oracle.rope(x, np.cos(theta), np.sin(theta), layout)
            ia, ib = _rope_pairs(d, layout)
            z = (x[..., ia] + 1j * x[..., ib]) * np.exp(1j * theta)
            assert np.allclose(y[..., ia], z.real, atol=1e-13) and np.allclose(y[..., ib], z.imag, atol=1e-13)


def pin_rope_layouts(oracle):
    # the half-split pairing is the interleaved one after moving channel i to
    # 2i and channel i + d/2 to 2i + 1
    d = 64
    x = gen.normal((1, 2, 9, d), 60).astype(np.float64)
    cos, sin = gen.rope_tables(9, d)
    perm = np.empty(d, dtype=np.int64)
    perm[0::2] = np.arange(d // 2)
    perm[1::2] = np.arange(d // 2) + d // 2
    inter = oracle.rope(x[..., perm], cos, sin, 1)
    half = oracle.rope(x, cos, sin, 2)
    assert np.allclose(half[..., perm], inter, atol=1e-14)


def pin_rope_relative_position(oracle):
    # with angles n * f_i, the score of positions (m, n) depends on m - n only
    d = 128
    q = gen.normal((1, 1, 1, d), 61).astype(np.float64)
    k = gen.normal((1, 1, 1, d), 62).astype(np.float64)
    freq = 10000.0 ** (-2.0 * np.arange(d // 2) / d)
    for layout in (1, 2):
        def at(x, pos):
            ang = (np.array([[pos]], dtype=np.float64) * freq[None, :])
            return oracle.rope(x, np.cos(ang), np.sin(ang), layout)[0, 0, 0]
        for (m, n, t) in ((5, 3, 7), (100, 0, 900), (17, 40, 3)):
            assert abs(at(q, m) @ at(k, n) - at(q, m + t) @ at(k, n + t)) <= 1e-11, (layout, m, n, t)


def pin_rope_quantiser(oracle):
    rows = _golden()["quant_block_rows"]["value"]
    B, H, N, d = 1, 2, 200, 64
    x = gen.outliers((B, H, N, d), 63)
    signs = gen.hadamard_signs(d, 64)
    # identity angles change nothing, bit for bit
    ones = np.ones((N, d // 2), dtype=np.float32)
    zeros = np.zeros((N, d // 2), dtype=np.float32)
    for sg in (None, signs):
        c0, s0 = oracle.quant_e4m3(x, signs=sg, block_rows=rows)
        for layout in (1, 2):
            c1, s1 = oracle.quant_e4m3(x, signs=sg, block_rows=rows, rope=(ones, zeros, layout))
            assert np.array_equal(c0, c1) and np.array_equal(s0, s1)
    # real angles: dequantised values within half an E4M3 step of the fp64
    # rotary embedding (and rotation) of x
    cos, sin = gen.rope_tables(N, d, offset=3)
    for layout in (1, 2):
        for sg in (None, signs):
            codes, ds = oracle.quant_e4m3(x, signs=sg, block_rows=rows, rope=(cos, sin, layout))
            target = oracle.rope(x, cos, sin, layout)
            if sg is not None:
                target = oracle.rotate(target, sg)
            deq = oracle.dequant_e4m3(codes, ds, block_rows=rows)
            for r0 in range(0, N, rows):
                tb = target[:, :, r0:r0 + rows]
                s = ds[:, :, r0 // rows][..., None, None]
                tol = np.maximum(np.abs(tb) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-4) + 1e-5 * np.abs(tb).max()
                assert np.all(np.abs(deq[:, :, r0:r0 + rows] - tb) <= tol), (layout, sg is None, r0)


def pin_flop_convention(oracle):
    g = _golden()["matmul_flops_per_exp_d128"]["value"]
    B, H, N, d = 1, 1, 1024, 128
    assert gen.flops(B, H, N, d, False) / (N * N) == g
    assert gen.flops(B, H, N, d, True) == gen.flops(B, H, N, d, False) / 2


ALL_PINS = [
    pin_library_cross_check, pin_zero_query, pin_causal_row0, pin_special_cases,
    pin_rotation_invariance, pin_online_recurrence, pin_row_subset,
    pin_e4m3_decode, pin_e4m3_encode, pin_fwht, pin_quantiser, pin_quantiser_exact_rounding,
    pin_quantiser_power_of_two_scale, pin_flop_convention,
    pin_rope_complex, pin_rope_layouts, pin_rope_relative_position, pin_rope_quantiser,
    pin_bwd_autograd, pin_bwd_finite_difference, pin_bwd_invariants, pin_bwd_empty_rows,
]
