"""Where the backward's parity tolerance comes from (CPU only).

The GPU backward is compared with the fp64 oracle's gradients with the
largest error at most 2.5 u of the largest |reference| entry and the rms
error at most 1.25 u of the reference's rms (u = 2^-8 for bf16, 2^-11 for
fp16).  Those bounds are derived from the roundings the kernel makes, and
this test keeps the derivation reproducible: it emulates exactly those
roundings in fp64 on the CPU --

  * O is the forward's output rounded to the element type, LSE is fp32;
  * P = exp(s * scale - LSE) is rounded to the element type before it
    multiplies dO (dV = P^T dO) and before dS is formed;
  * D_i = dO_i . O_i uses the rounded O;
  * dS = P (dP - D) is rounded to the element type before dK = scale dS^T Q
    and dQ = scale dS K;
  * dQ, dK, dV are accumulated exactly (fp32 accumulation adds far less than
    u) and rounded once to the element type --

and checks that such a kernel stays inside the bounds, with room to spare,
over the shapes, scales and masks the GPU tests use.  It also checks that
the bounds are not loose: an emulation that skips none of the roundings but
rounds P and dS to a type with 4 times the unit roundoff must fail them.
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle

UNIT = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}
MAX_U, RMS_U = 2.5, 1.25


def _round(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).to(torch.float64).numpy()


def _coarse(x, bits_dropped):
    """Round to a significand `bits_dropped` bits shorter than fp64's
    (round to nearest), for the looseness check."""
    m, e = np.frexp(x)
    scale = 2.0 ** (53 - bits_dropped)
    return np.ldexp(np.round(m * scale) / scale, e)


def emulate_bwd(q, k, v, do, causal, scale, dtype, p_round=None):
    """Gradients with the kernel's roundings (see the module docstring).
    q, k, v, do: fp64 arrays holding element-type values, [B, H, N, d]
    (Hq = Hkv)."""
    rnd = (lambda x: _round(x, dtype)) if p_round is None else p_round
    o64, l64 = oracle.attn_fwd(q, k, v, causal=causal, scale=scale)
    o = _round(o64, dtype)
    lse = l64.astype(np.float32).astype(np.float64)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, h] @ k[b, h].T)
            with np.errstate(invalid="ignore", over="ignore"):
                p = np.exp(s - lse[b, h][:, None])
            if causal:
                vis = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
                p = np.where(vis, p, 0.0)
            p = np.where(np.isneginf(lse[b, h])[:, None], 0.0, p)
            pr = rnd(p)
            dp = do[b, h] @ v[b, h].T
            D = (do[b, h] * o[b, h]).sum(axis=1)
            ds = rnd(pr * (dp - D[:, None]))
            dv[b, h] = _round(pr.T @ do[b, h], dtype)
            dk[b, h] = _round(scale * (ds.T @ q[b, h]), dtype)
            dq[b, h] = _round(scale * (ds @ k[b, h]), dtype)
    return dq, dk, dv


def _ratios(got, ref):
    out = []
    for g, r in zip(got, ref):
        rmax = np.abs(r).max()
        rrms = math.sqrt((r ** 2).mean())
        e = g - r
        out.append((np.abs(e).max() / rmax, math.sqrt((e ** 2).mean()) / rrms))
    return out


CASES = [
    # B, H, Nq, Nk, d, causal, scale
    (1, 2, 256, 256, 64, False, None),
    (1, 2, 256, 256, 128, True, None),
    (1, 2, 200, 300, 128, True, 0.3),
    (1, 2, 160, 160, 64, False, -0.2),
    (1, 1, 300, 100, 128, True, None),
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "N{}x{}_d{}_c{}_s{}".format(c[2], c[3], c[4], int(c[5]), c[6]))
def test_emulated_kernel_roundings_fit_the_bounds(dtype, case):
    B, H, Nq, Nk, d, causal, scale = case
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    q = _round(gen.normal((B, H, Nq, d), 1500 + Nq, 0).astype(np.float64), dtype)
    k = _round(gen.normal((B, H, Nk, d), 1500 + Nq, 1).astype(np.float64), dtype)
    v = _round(gen.normal((B, H, Nk, d), 1500 + Nq, 2).astype(np.float64), dtype)
    do = _round(gen.normal((B, H, Nq, d), 1500 + Nq, 3).astype(np.float64), dtype)
    ref = oracle.attn_bwd(q, k, v, do, causal=causal, scale=scale)
    got = emulate_bwd(q, k, v, do, causal, scale, dtype)
    u = UNIT[dtype]
    for name, (mx, rms) in zip(("dQ", "dK", "dV"), _ratios(got, ref)):
        assert mx <= 0.8 * MAX_U * u, f"{name}: emulated max error {mx / u:.2f} u"
        assert rms <= 0.8 * RMS_U * u, f"{name}: emulated rms error {rms / u:.2f} u"


def test_bounds_reject_coarser_roundings():
    # P and dS rounded with 2 fewer significand bits than bf16 (4 u): the
    # bounds must catch that, so they are not loose enough to hide a kernel
    # that rounds more than the derivation allows
    dtype = torch.bfloat16
    B, H, N, d = 1, 2, 256, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (_round(gen.normal((B, H, N, d), 1600, i).astype(np.float64), dtype) for i in range(4))
    ref = oracle.attn_bwd(q, k, v, do, causal=False, scale=scale)
    got = emulate_bwd(q, k, v, do, False, scale, dtype, p_round=lambda x: _coarse(x, 53 - 6))
    u = UNIT[dtype]
    worst = max(max(mx / (MAX_U * u), rms / (RMS_U * u)) for mx, rms in _ratios(got, ref))
    assert worst > 1.0, f"coarser roundings stayed inside the bounds ({worst:.2f} of the bound)"
