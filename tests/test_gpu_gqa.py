"""Grouped-query / multi-query attention and Nq != Nk (fa_fwd_gqa,
fa_fwd_fp8_gqa) against the fp64 oracle, which maps query head h to K/V
head h / (Hq / Hkv) and aligns causal masks at the bottom right
(key j visible to query i iff j <= i + Nk - Nq)."""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle
from gpu_util import FP8_O_RMSE, LSE_ABS, O_MAXABS, O_RMSE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_09_gb300 as fa
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()
    return fa


def _inputs(B, Hq, Hkv, Nq, Nk, d, seed, dtype):
    q = torch.from_numpy(gen.normal((B, Hq, Nq, d), seed, 0)).to(dtype)
    k = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 1)).to(dtype)
    v = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 2)).to(dtype)
    return q, k, v


def _check(o, lse, o_ref, l_ref, what):
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: rows without keys must have LSE = -inf"
    assert np.all(o[empty] == 0.0), f"{what}: rows without keys must have O = 0"
    if (~empty).any():
        diff = o[~empty] - o_ref[~empty]
        assert np.isfinite(o).all()
        assert np.abs(diff).max() <= O_MAXABS, f"{what}: O max-abs {np.abs(diff).max():.3e}"
        assert math.sqrt((diff ** 2).mean()) <= O_RMSE, what
        assert np.abs(lse[~empty] - l_ref[~empty]).max() <= LSE_ABS, what

def _check_scaled(o, lse, o_ref, l_ref, v_absmax, what):
    """Rows without keys exactly O = 0, LSE = -inf; the others within the
    element-wise bound derived from the arithmetic (a scale other than
    1/sqrt(d) makes the softmax flatter or peakier than the N(0,1)
    tolerance assumes: P rounded to bf16 costs at most 2^-9 max|V| on O, the
    output rounding 2^-9 |O|; twice that plus 1e-4), LSE within 1e-3."""
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: rows without keys must have LSE = -inf"
    assert np.all(o[empty] == 0.0), f"{what}: rows without keys must have O = 0"
    assert np.isfinite(o).all() and np.isfinite(lse[~empty]).all(), what
    tol = 2.0 ** -8 * (np.abs(o_ref[~empty]) + v_absmax) + 1e-4
    excess = np.abs(o[~empty] - o_ref[~empty]) - tol
    assert (excess <= 0).all(), f"{what}: {int((excess > 0).sum())} elements beyond the bound"
    assert np.abs(lse[~empty] - l_ref[~empty]).max() <= LSE_ABS, what



@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (8, 1)])
@pytest.mark.parametrize("Nq,Nk", [(300, 300), (128, 700), (700, 128), (1, 513), (513, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_bf16(fa, Hq, Hkv, Nq, Nk, causal):
    d = 128
    q, k, v = _inputs(1, Hq, Hkv, Nq, Nk, d, 500 + Nq + Nk + Hkv, torch.bfloat16)
    o, lse = fa.fwd_gqa(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    fa.check_device_error()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=causal, scale=1 / math.sqrt(d))
    _check(o, lse, o_ref, l_ref, f"Hq={Hq} Hkv={Hkv} Nq={Nq} Nk={Nk} causal={causal}")


@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_gqa_head_dims(fa, d, dtype):
    q, k, v = _inputs(2, 6, 3, 400, 650, d, 600 + d, dtype)
    for causal in (False, True):
        o, lse = fa.fwd_gqa(q.cuda(), k.cuda(), v.cuda(), causal=causal)
        o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=causal, scale=1 / math.sqrt(d))
        _check(o, lse, o_ref, l_ref, f"d={d} {dtype} causal={causal}")


def test_gqa_equal_shapes_match_fa_fwd(fa):
    q, k, v = (t.cuda() for t in _inputs(2, 4, 4, 777, 777, 128, 700, torch.bfloat16))
    for causal in (False, True):
        o1, l1 = fa.fwd(q, k, v, causal=causal)
        o2, l2 = fa.fwd_gqa(q, k, v, causal=causal)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_fp8(fa, causal):
    B, Hq, Hkv, Nq, Nk, d = 1, 8, 2, 384, 640, 128
    q, k, v = (a.numpy().astype(np.float32) for a in _inputs(B, Hq, Hkv, Nq, Nk, d, 800, torch.float32))
    signs = gen.hadamard_signs(d, 4)
    qc, qs = oracle.quant_e4m3(q, signs=signs)
    kc, ks = oracle.quant_e4m3(k, signs=signs)
    vc, vs = oracle.quant_e4m3(v)
    dev = lambda a: torch.from_numpy(a).cuda()
    o, lse = fa.fwd_fp8_gqa(dev(qc), dev(kc), dev(vc), dev(qs), dev(ks), dev(vs), causal=causal)
    fa.check_device_error()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=causal, scale=1 / math.sqrt(d))
    o = o.float().cpu().numpy()
    assert math.sqrt(((o - o_ref) ** 2).mean()) <= FP8_O_RMSE
    qd, kd, vd = oracle.dequant_e4m3(qc, qs), oracle.dequant_e4m3(kc, ks), oracle.dequant_e4m3(vc, vs)
    _, l_dq = oracle.attn_fwd(qd, kd, vd, causal=causal, scale=1 / math.sqrt(d))
    assert np.abs(lse.cpu().numpy() - l_dq).max() <= 1e-3


# Zero and negative scales on rows that see no key in a tile (causal with
# Nq > Nk leaves the first Nq - Nk rows without any key; the others see a
# ragged prefix of the last tile).  For a zero scale a fully masked tile's
# row maximum times the scale is inf * 0, so these cases guard that such a
# row keeps m = -inf: rows without keys must come out O = 0, LSE = -inf, and
# every other row must match the oracle.
@pytest.mark.parametrize("scale", [0.0, -0.2])
@pytest.mark.parametrize("Nq,Nk,d", [(700, 128, 128), (513, 1, 128), (300, 260, 64), (400, 150, 256)])
def test_gqa_rows_without_keys_zero_and_negative_scale(fa, scale, Nq, Nk, d):
    q, k, v = _inputs(1, 4, 2, Nq, Nk, d, 950 + Nq + d, torch.bfloat16)
    o, lse = fa.fwd_gqa(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
    fa.check_device_error()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=True, scale=scale)
    assert np.isneginf(l_ref).any()
    _check_scaled(o, lse, o_ref, l_ref, float(v.float().abs().max()), f"Nq={Nq} Nk={Nk} d={d} scale={scale}")


@pytest.mark.parametrize("scale", [0.0, -0.2])
def test_gqa_fp8_rows_without_keys_zero_and_negative_scale(fa, scale):
    B, Hq, Hkv, Nq, Nk, d = 1, 4, 2, 640, 300, 128
    q, k, v = (a.numpy().astype(np.float32) for a in _inputs(B, Hq, Hkv, Nq, Nk, d, 960, torch.float32))
    qc, qs = oracle.quant_e4m3(q)
    kc, ks = oracle.quant_e4m3(k)
    vc, vs = oracle.quant_e4m3(v)
    dev = lambda a: torch.from_numpy(a).cuda()
    o, lse = fa.fwd_fp8_gqa(dev(qc), dev(kc), dev(vc), dev(qs), dev(ks), dev(vs), causal=True, scale=scale)
    fa.check_device_error()
    qd, kd, vd = oracle.dequant_e4m3(qc, qs), oracle.dequant_e4m3(kc, ks), oracle.dequant_e4m3(vc, vs)
    o_ref, l_ref = oracle.attn_fwd(qd, kd, vd, causal=True, scale=scale)
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(l_ref)
    assert empty.any()
    assert np.array_equal(np.isneginf(lse), empty)
    assert np.all(o[empty] == 0.0)
    assert np.isfinite(o).all() and np.isfinite(lse[~empty]).all()
    assert math.sqrt(((o[~empty] - o_ref[~empty]) ** 2).mean()) <= FP8_O_RMSE
    assert np.abs(lse[~empty] - l_ref[~empty]).max() <= 1e-3
