"""Split-KV forward (fa_fwd_splitkv) for decode-like shapes against the fp64
oracle, which maps query head h to key/value head h / (Hq / Hkv) and aligns
causal masks at the bottom right.  The kernel packs the query heads of a
key/value group into one head of (Hq / Hkv) * Nq rows (so causal positions are
taken modulo Nq) and splits the keys into runs merged by LSE weights; every
case is checked on every row with the BF16 tolerances, and rows that see no
key must come out as O = 0, LSE = -inf."""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle
from gpu_util import LSE_ABS, O_MAXABS, O_RMSE

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
        assert np.isfinite(o).all(), what
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



CASES = [
    # B, Hq, Hkv, Nq, Nk, d, causal
    (2, 8, 2, 1, 3000, 128, False),      # decode, GQA 4
    (1, 8, 1, 1, 5000, 64, True),        # MQA, one query (causal = all keys)
    (2, 4, 4, 5, 777, 64, True),         # no packing, short causal query block
    (1, 6, 2, 16, 2049, 256, True),      # d = 256, ragged last key tile
    (1, 16, 4, 40, 1500, 128, True),     # packed rows 160: a Q tile spans heads
    (1, 4, 2, 8, 5, 128, True),          # Nq > Nk: rows without visible keys
    (3, 2, 1, 100, 300, 128, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_Nq{}_Nk{}_d{}_c{}".format(*c))
@pytest.mark.parametrize("splits", [0, 1, 3, 64])
def test_splitkv_bf16(fa, case, splits):
    B, Hq, Hkv, Nq, Nk, d, causal = case
    q, k, v = _inputs(B, Hq, Hkv, Nq, Nk, d, 900 + Nq + Nk + d, torch.bfloat16)
    o, lse = fa.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=causal, num_splits=splits)
    fa.check_device_error()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=causal, scale=1 / math.sqrt(d))
    _check(o, lse, o_ref, l_ref, f"{case} splits={splits}")


def test_splitkv_fp16_and_workspace(fa):
    B, Hq, Hkv, Nq, Nk, d = 2, 8, 2, 3, 4100, 128
    q, k, v = _inputs(B, Hq, Hkv, Nq, Nk, d, 77, torch.float16)
    need = fa.splitkv_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, 5)
    assert need > 0
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    o, lse = fa.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=True, num_splits=5, workspace=ws)
    fa.check_device_error()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=True, scale=1 / math.sqrt(d))
    _check(o, lse, o_ref, l_ref, "fp16")
    # a workspace one byte short is refused before any launch
    st = fa.lib().fa_fwd_splitkv(q.cuda().data_ptr(), k.cuda().data_ptr(), v.cuda().data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d, 1, 0.1, fa.FA_DTYPE_FP16, 5, ws.data_ptr(),
                                 need - 1, torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_ERR_INVALID_ARG
    # one run needs no workspace at all
    assert fa.splitkv_workspace_bytes(B, Hq, Hkv, Nq, Nk, d, 1) == 0


def test_splitkv_matches_unsplit_closely(fa):
    # the merge is exact in real arithmetic: split and unsplit results agree
    # far inside the oracle tolerance
    B, Hq, Hkv, Nq, Nk, d = 1, 8, 2, 2, 6000, 128
    q, k, v = (t.cuda() for t in _inputs(B, Hq, Hkv, Nq, Nk, d, 78, torch.bfloat16))
    o1, l1 = fa.fwd_gqa(q, k, v, causal=True)
    o2, l2 = fa.fwd_splitkv(q, k, v, causal=True, num_splits=7)
    torch.cuda.synchronize()
    assert (o1.float() - o2.float()).abs().max().item() <= 8e-3
    assert (l1 - l2).abs().max().item() <= 1e-4


# Runs beyond a row's last key: with causal masks and Nq close to Nk the
# first rows see no key of the last runs, whose LSE must then be -inf (not
# NaN) so that the merge gives those runs weight 0.  A zero scale makes a
# fully masked tile's maximum times the scale inf * 0; a negative scale
# flips which score is the largest.
SCALE_CASES = [
    # B, Hq, Hkv, Nq, Nk, d
    (1, 4, 2, 600, 700, 128),   # rows 0..411 see no key of the last of 3 runs
    (1, 4, 4, 300, 1100, 64),
    (1, 8, 2, 4, 3000, 128),    # decode-like, packed rows
    (1, 4, 2, 8, 5, 128),       # Nq > Nk: rows without any key
]


@pytest.mark.parametrize("case", SCALE_CASES, ids=lambda c: "B{}_Hq{}_Hkv{}_Nq{}_Nk{}_d{}".format(*c))
@pytest.mark.parametrize("splits", [3, 64])
@pytest.mark.parametrize("scale", [0.0, -0.2])
def test_splitkv_zero_and_negative_scale(fa, case, splits, scale):
    B, Hq, Hkv, Nq, Nk, d = case
    q, k, v = _inputs(B, Hq, Hkv, Nq, Nk, d, 970 + Nq + d, torch.bfloat16)
    o, lse = fa.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale, num_splits=splits)
    fa.check_device_error()
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=True, scale=scale)
    _check_scaled(o, lse, o_ref, l_ref, float(v.float().abs().max()), f"{case} splits={splits} scale={scale}")
