"""Failure detection on the GPU without a GPU fault: a pipeline wait that can
never complete (the test hook fa_debug_inject leaves one K/V ring slot of
one CTA unfilled) must end the kernel within its time limit, report
FA_ERR_TIMEOUT through fa_check_device_error, and leave the CUDA context
usable for the next, correct call."""
import math
import time

import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle

from gpu_util import assert_bf16_parity, errors, make_qkv, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_09_gb300 as fa
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()
    return fa


def test_pipeline_timeout_is_reported_and_context_survives(fa):
    host, (q, k, v) = make_qkv(1, 2, 1024, 128, 31)
    lib = fa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    assert lib.fa_debug_inject(1) == fa.FA_OK
    t0 = time.time()
    fa.fwd(q, k, v, causal=False)
    st = lib.fa_check_device_error(stream)
    elapsed = time.time() - t0
    assert st == fa.FA_ERR_TIMEOUT, lib.fa_status_string(st)
    assert elapsed < 30.0
    # the error word is cleared by the check, the hook by the launch
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    o, lse = fa.fwd(q, k, v, causal=False)
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    o_ref, l_ref = oracle_rows(host, False, 1.0 / math.sqrt(128))
    assert_bf16_parity(errors(o, lse, o_ref, l_ref), "after the injected timeout")


@pytest.mark.parametrize("d", [64, 128])
def test_backward_pipeline_timeout_is_reported_and_context_survives(fa, d):
    """The same for fa_bwd: one Q/dO stage of the first CTA is never filled."""
    q, k, v, do = (torch.randn(1, 2, 512, d, device="cuda").to(torch.bfloat16) for _ in range(4))
    lib = fa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    o, lse = fa.fwd(q, k, v, causal=False)
    ref = fa.bwd(q, k, v, o, lse, do)
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    assert lib.fa_debug_inject(1) == fa.FA_OK
    t0 = time.time()
    fa.bwd(q, k, v, o, lse, do)
    st = lib.fa_check_device_error(stream)
    assert st == fa.FA_ERR_TIMEOUT, lib.fa_status_string(st)
    assert time.time() - t0 < 30.0
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    dq, dk, dv = fa.bwd(q, k, v, o, lse, do)
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert (dq.float() - ref[0].float()).abs().max().item() <= 1e-2 * ref[0].float().abs().max().item()


@pytest.mark.parametrize("per_tensor", [False, True])
@pytest.mark.parametrize("rope", [False, True])
def test_quantiser_timeout_is_reported_and_next_call_exact(fa, per_tensor, rope):
    """The quantiser's first CTA never gets one input slot: the bounded waits
    run out, FA_ERR_TIMEOUT is reported, the blocks that CTA could not finish
    carry a NaN descale (per tensor: an infinite maximum, so every descale is
    infinite) instead of old values, and the next call is bit-exact.  With
    the rotary embedding the angle tables are staged in shared memory, and
    the other warps of that CTA stop at their table waits too."""
    x = gen.outliers((2, 4, 1000, 128), 33)
    xd = torch.from_numpy(x).cuda()
    tables = gen.rope_tables(1000, 128) if rope else None
    rp = (torch.from_numpy(tables[0]).cuda(), torch.from_numpy(tables[1]).cuda(), 2) if rope else None
    lib = fa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    assert lib.fa_debug_inject(2) == fa.FA_OK
    t0 = time.time()
    _, ds = fa.quant_fp8(xd, per_tensor=per_tensor, rope=rp)
    st = lib.fa_check_device_error(stream)
    assert st == fa.FA_ERR_TIMEOUT, lib.fa_status_string(st)
    assert time.time() - t0 < 30.0
    ds = ds.cpu().numpy()
    if per_tensor:
        assert np.isinf(ds).all()
    else:
        assert np.isnan(ds.reshape(-1)[0])
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    codes, ds = fa.quant_fp8(xd, per_tensor=per_tensor, rope=rp)
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    codes_ref, ds_ref = oracle.quant_e4m3(x, per_tensor=per_tensor, rope=(tables[0], tables[1], 2) if rope else None)
    assert np.array_equal(codes.cpu().numpy(), codes_ref)
    assert np.array_equal(ds.cpu().numpy(), ds_ref)


def test_inject_rejects_bad_flags(fa):
    assert fa.lib().fa_debug_inject(7) == fa.FA_ERR_INVALID_ARG
    assert fa.lib().fa_debug_inject(-1) == fa.FA_ERR_INVALID_ARG
    assert fa.lib().fa_debug_inject(0) == fa.FA_OK
