"""The ablation library's kernel variants (libfa_ablate.so, fa_ablate_fwd)
compute the same attention as the shipped kernel: every built variant is
compared with the fp64 oracle on small cases with the BF16 / FP8 tolerances,
so that the timings of bench.py --ablate compare correct kernels."""
import ctypes
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle
from gpu_util import FP8_O_RMSE, assert_bf16_parity, errors, make_qkv, oracle_rows

pytestmark = pytest.mark.gpu

BUILT = {(False, False, 128): (0, 1, 2, 4, 8, 16, 64, 128, 256), (False, True, 128): (0, 1, 8, 16, 256),
         (True, False, 128): (0, 1, 2, 4, 8, 16, 64, 128, 256), (False, False, 64): (0, 1, 32, 64, 128, 256),
         (False, True, 64): (0, 32)}


@pytest.fixture(scope="module")
def ab():
    import exact_attention_forward_09_gb300 as fa
    from exact_attention_forward_09_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()
    lib = ctypes.CDLL(build.LIB_ABLATE)
    vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.fa_ablate_fwd.argtypes = [i32, i32, vp, vp, vp, vp, vp, i64, i64, i64, i64, i32, f32, vp, vp, vp, vp]
    lib.fa_ablate_fwd.restype = i32
    return fa, lib


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [640, 1100])
def test_bf16_variants(ab, d, causal, N):
    fa, lib = ab
    host, (q, k, v) = make_qkv(2, 3, N, d, 1700 + N + d)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle_rows(host, causal, scale)
    for var in BUILT[(False, causal, d)]:
        o = torch.empty_like(q)
        lse = torch.empty((2, 3, N), device="cuda", dtype=torch.float32)
        st = lib.fa_ablate_fwd(var, 0, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               2, 3, N, d, int(causal), scale, None, None, None,
                               torch.cuda.current_stream().cuda_stream)
        assert st == fa.FA_OK
        fa.check_device_error()
        assert_bf16_parity(errors(o, lse, o_ref, l_ref), f"variant {var} d={d} causal={causal} N={N}")


def test_fp8_variants(ab):
    fa, lib = ab
    B, H, N, d = 1, 4, 900, 128
    q, k, v = gen.qkv_outliers((B, H, N, d), 1710)
    signs = gen.hadamard_signs(d, 4)
    qc, qs = oracle.quant_e4m3(q, signs=signs)
    kc, ks = oracle.quant_e4m3(k, signs=signs)
    vc, vs = oracle.quant_e4m3(v)
    dev = lambda a: torch.from_numpy(a).cuda()
    qd, kd, vd, qsd, ksd, vsd = (dev(a) for a in (qc, kc, vc, qs, ks, vs))
    o_ex, _ = oracle.attn_fwd(q, k, v, causal=False, scale=1 / math.sqrt(d))
    for var in BUILT[(True, False, 128)]:
        o = torch.empty((B, H, N, d), device="cuda", dtype=torch.bfloat16)
        lse = torch.empty((B, H, N), device="cuda", dtype=torch.float32)
        st = lib.fa_ablate_fwd(var, 1, qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               B, H, N, d, 0, 1 / math.sqrt(d), qsd.data_ptr(), ksd.data_ptr(), vsd.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
        assert st == fa.FA_OK
        fa.check_device_error()
        og = o.float().cpu().numpy()
        assert math.sqrt(((og - o_ex) ** 2).mean()) <= FP8_O_RMSE, var


def test_unbuilt_variant_is_refused(ab):
    fa, lib = ab
    p = torch.empty(16, device="cuda").data_ptr()
    # causal FP8 variants are not built, nor separate P at d = 128, nor d = 256
    assert lib.fa_ablate_fwd(2, 1, p, p, p, p, p, 1, 1, 128, 128, 1, 0.1, p, p, p, None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_ablate_fwd(32, 0, p, p, p, p, p, 1, 1, 128, 128, 0, 0.1, None, None, None, None) == \
        fa.FA_ERR_UNSUPPORTED
    assert lib.fa_ablate_fwd(0, 0, p, p, p, p, p, 1, 1, 128, 256, 0, 0.1, None, None, None, None) == \
        fa.FA_ERR_UNSUPPORTED
