"""The exponential the forward kernels compute on the FMA pipe for a share of
P (range reduction plus a minimax polynomial, the test hook fa_debug_exp2)
against exact 2^x in fp64, and against the special-function unit's ex2 that
computes the rest of P.  The bound per degree is the one the polynomial was
fitted to (its maximum relative error on [-1/2, 1/2] with fp32 coefficients
and fp32 evaluation), plus the final rounding to fp32."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

BOUND = {3: 7.5e-5, 4: 2.7e-6}
ROUND = 2.0 ** -23  # the result's own rounding to fp32


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_09_gb300 as fa
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()
    return fa


def _eval(fa, x, method):
    xd = x.cuda()
    y = torch.empty_like(xd)
    st = fa.lib().fa_debug_exp2(xd.data_ptr(), y.data_ptr(), xd.numel(), method,
                                torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, fa.lib().fa_status_string(st)
    torch.cuda.synchronize()
    return y.cpu()


def _grid():
    # dense over the kernels' range, every half-integer (where the rounded
    # n switches) and its neighbours, and the ends of the valid range
    dense = torch.linspace(-125.0, 20.0, (1 << 22) + 1, dtype=torch.float64)
    half = torch.arange(-125, 127, dtype=torch.float64) + 0.5
    steps = torch.cat([half, torch.nextafter(half, half + 1), torch.nextafter(half, half - 1)])
    ends = torch.tensor([-125.0, 0.0, -0.0, 8.0, 14.0, 126.9, 127.0, 127.49], dtype=torch.float64)
    return torch.cat([dense, steps, ends]).to(torch.float32)


@pytest.mark.parametrize("deg", [3, 4])
def test_polynomial_relative_error_bound(fa, deg):
    x = _grid()
    y = _eval(fa, x, deg).double()
    ref = torch.exp2(x.double())
    rel = ((y - ref) / ref).abs()
    worst = rel.max().item()
    assert worst <= BOUND[deg] + ROUND, f"degree {deg}: max relative error {worst:.3e} at x={x[rel.argmax()].item()}"
    # the bound is not loose: the polynomial's error reaches most of it
    assert worst >= 0.8 * BOUND[deg]


@pytest.mark.parametrize("deg", [3, 4])
def test_polynomial_matches_special_function_unit(fa, deg):
    x = _grid()
    yp = _eval(fa, x, deg).double()
    ym = _eval(fa, x, 0).double()
    assert (ym > 0).all()
    rel = ((yp - ym) / ym).abs().max().item()
    # MUFU ex2's own error is a few fp32 ulps
    assert rel <= BOUND[deg] + 8 * ROUND, rel


@pytest.mark.parametrize("deg", [3, 4])
def test_polynomial_special_values(fa, deg):
    x = torch.tensor([float("nan"), -126.0, -126.4, -127.0, -150.0, -1e30, float("-inf"), -125.6], dtype=torch.float32)
    y = _eval(fa, x, deg).double()
    assert torch.isnan(y[0])
    # below -126 the result is tiny (at most 2^-125.5), never negative, never NaN
    assert ((y[1:7] >= 0) & (y[1:7] <= 2.0 ** -125.5)).all(), y
    # -125.6 (as fp32) is still a normal result within the bound
    ref = 2.0 ** float(x[7])
    assert abs(y[7].item() - ref) / ref <= BOUND[deg] + ROUND


def test_odd_length_and_host_checks(fa):
    x = torch.tensor([0.0, 1.0, -1.0], dtype=torch.float32)
    y = _eval(fa, x, 3)
    assert torch.allclose(y.double(), torch.tensor([1.0, 2.0, 0.5], dtype=torch.float64), rtol=BOUND[3] + ROUND)
    lib = fa.lib()
    s = torch.cuda.current_stream().cuda_stream
    xd = x.cuda()
    assert lib.fa_debug_exp2(xd.data_ptr(), xd.data_ptr(), 3, 5, s) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_debug_exp2(xd.data_ptr(), xd.data_ptr(), -1, 3, s) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_debug_exp2(None, None, 3, 3, s) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_debug_exp2(None, None, 0, 3, s) == fa.FA_OK
    fa.check_device_error()
