"""Non-finite inputs: what the forward does with a NaN in Q, K or V, checked
against the fp64 oracle on the same inputs (include/fa.h, fa_fwd).  Outputs
the NaN cannot reach must still match the oracle; those it reaches are NaN in
both; with causal masking, a NaN value element also reaches its column in the
rows of its own 128-row tile that precede it (P = 0 times NaN in the P V
product), which the plain definition leaves finite -- that difference is
documented and pinned here."""
import math

import numpy as np
import pytest
import torch

from gpu_util import LSE_ABS, O_MAXABS, make_qkv, oracle_rows

pytestmark = pytest.mark.gpu

B, H, N, d = 1, 2, 640, 128
J = 300  # the poisoned row (tile 2: rows 256..383)


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_09_gb300 as fa
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()
    return fa


def _run(fa, which, causal):
    host, dev = make_qkv(B, H, N, d, 2100 + int(causal))
    t = {"q": 0, "k": 1, "v": 2}[which]
    host[t][0, 0, J, 7] = float("nan")
    dev[t][0, 0, J, 7] = float("nan")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(*dev, causal=causal, scale=scale)
    fa.check_device_error()
    o_ref, l_ref = oracle_rows(host, causal, scale)
    return o.float().cpu().numpy().astype(np.float64), lse.float().cpu().numpy().astype(np.float64), o_ref, l_ref


def _rows_nan(o, lse, rows):
    return bool(np.isnan(o[0, 0, rows]).all() and np.isnan(lse[0, 0, rows]).all())


def _rows_match(o, lse, o_ref, l_ref, h, rows):
    if len(rows) == 0:
        return True
    a, b = o[0, h, rows], o_ref[0, h, rows]
    return bool(np.isfinite(a).all() and np.abs(a - b).max() <= O_MAXABS
                and np.abs(lse[0, h, rows] - l_ref[0, h, rows]).max() <= LSE_ABS)


@pytest.mark.parametrize("causal", [False, True])
def test_nan_in_query_row(fa, causal):
    o, lse, o_ref, l_ref = _run(fa, "q", causal)
    others = [i for i in range(N) if i != J]
    assert _rows_nan(o, lse, [J]) and np.isnan(o_ref[0, 0, J]).all()
    assert _rows_match(o, lse, o_ref, l_ref, 0, others)
    assert _rows_match(o, lse, o_ref, l_ref, 1, list(range(N)))


@pytest.mark.parametrize("causal", [False, True])
def test_nan_in_key_row(fa, causal):
    o, lse, o_ref, l_ref = _run(fa, "k", causal)
    hit = list(range(J, N)) if causal else list(range(N))
    clean = list(range(J)) if causal else []
    assert _rows_nan(o, lse, hit) and np.isnan(o_ref[0, 0, hit]).all()
    assert _rows_match(o, lse, o_ref, l_ref, 0, clean)
    assert _rows_match(o, lse, o_ref, l_ref, 1, list(range(N)))


@pytest.mark.parametrize("causal", [False, True])
def test_nan_in_value_element(fa, causal):
    # V[J, 7] = NaN: only output column 7 can carry it
    o, lse, o_ref, l_ref = _run(fa, "v", causal)
    c, rest = 7, [x for x in range(d) if x != 7]
    tile0 = (J // 128) * 128
    hit = list(range(J, N)) if causal else list(range(N))
    # rows that see key J: column 7 NaN in both
    assert np.isnan(o[0, 0, hit, c]).all() and np.isnan(o_ref[0, 0, hit, c]).all()
    if causal:
        # rows of J's tile before J: NaN here (0 * NaN in P V), finite in the oracle
        assert np.isnan(o[0, 0, tile0:J, c]).all() and np.isfinite(o_ref[0, 0, tile0:J, c]).all()
        # rows of earlier tiles never meet V[J]
        assert _rows_match(o, lse, o_ref, l_ref, 0, list(range(tile0)))
    # every other column, and LSE (which does not involve V), match the oracle
    a, b = o[0, 0][:, rest], o_ref[0, 0][:, rest]
    assert np.isfinite(a).all() and np.abs(a - b).max() <= O_MAXABS
    assert np.isfinite(lse[0, 0]).all() and np.abs(lse[0, 0] - l_ref[0, 0]).max() <= LSE_ABS
    assert _rows_match(o, lse, o_ref, l_ref, 1, list(range(N)))
