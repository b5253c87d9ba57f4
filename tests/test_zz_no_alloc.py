"""The allocation-free per-tensor quantiser (fa_quant_fp8_per_tensor_noalloc).

Callers that cannot allocate device memory (a framework that owns every
buffer, a plug-in host that forbids cudaMalloc, a fixed memory budget) use
this entry point: its scratch is a static device array inside the library.
It must produce exactly what fa_quant_fp8 with per_tensor = 1 produces (the
quantiser tests here are bit-exact), on two calls in a row -- the scratch
keeps the previous call's contents, so the second call checks that nothing
stale leaks through -- and it must refuse problems larger than its scratch.

This file sorts last so that a run stopping at the first failure has run
every other test first; it also passes alone in a fresh process.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import attn_inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    from exact_attention_forward_09_gb300 import build
    build.build()
    import exact_attention_forward_09_gb300 as fa
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()
    return fa


def _noalloc_c(fa, x, signs):
    """Direct C-ABI call; outputs are allocated by the test, not the library."""
    B, H, N, d = x.shape
    nblk = (N + 127) // 128
    x8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
    ds = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device)
    keep = None
    sp = None
    if signs is not None:
        keep = (ctypes.c_int8 * d)(*[int(s) for s in signs])
        sp = ctypes.cast(keep, ctypes.c_void_p)
    st = fa.lib().fa_quant_fp8_per_tensor_noalloc(x.data_ptr(), x8.data_ptr(), ds.data_ptr(), B, H, N, d, sp,
                                                  torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK, fa.lib().fa_status_string(st).decode()
    return x8, ds


@pytest.mark.parametrize("shape,rot", [((2, 3, 300, 128), True), ((1, 2, 1000, 64), False),
                                       ((1, 1, 129, 256), True), ((16, 16, 1024, 128), True)])
def test_noalloc_matches_workspace_entry_point(fa, shape, rot):
    d = shape[-1]
    signs = gen.hadamard_signs(d, 4) if rot else None
    # two calls in a row on different tensors; the second one has a much
    # smaller amax, so a stale maximum from the first call would show
    xs = [gen.outliers(shape, 900 + i, sigma=10.0) * (1.0 if i == 0 else 0.01) for i in range(2)]
    for x_np in xs:
        x = torch.from_numpy(x_np.astype(np.float32)).cuda()
        ref8, ref_ds = fa.quant_fp8(x, signs=signs, per_tensor=True)
        got8, got_ds = _noalloc_c(fa, x, signs)
        torch.cuda.synchronize()
        assert torch.equal(got8, ref8), "E4M3 codes differ from fa_quant_fp8(per_tensor=1)"
        assert torch.equal(got_ds.view(torch.int32), ref_ds.view(torch.int32)), "descales differ"
    fa.check_device_error()


def test_noalloc_binding_and_limit(fa):
    x = torch.from_numpy(gen.outliers((1, 2, 200, 128), 77)).cuda()
    a8, ads = fa.quant_fp8_per_tensor_noalloc(x)
    b8, bds = fa.quant_fp8(x, per_tensor=True)
    assert torch.equal(a8, b8) and torch.equal(ads, bds)
    # beyond the static scratch: refused before any launch
    p = x.data_ptr()
    lim = fa.QUANT_NOALLOC_MAX_BLOCKS
    st = fa.lib().fa_quant_fp8_per_tensor_noalloc(p, p, p, 1, lim + 1, 128, 128, None, None)
    assert st == fa.FA_ERR_SCRATCH_LIMIT
    st = fa.lib().fa_quant_fp8_per_tensor_noalloc(p, p, p, 2, 1, 128 * (lim // 2 + 1), 128, None, None)
    assert st == fa.FA_ERR_SCRATCH_LIMIT


def test_noalloc_smaller_call_after_larger(fa):
    # a large call leaves 16 * 16 * 8 partial maxima behind; a following call
    # with one block and a far smaller maximum must not see any of them
    big = torch.from_numpy(gen.outliers((16, 16, 1024, 128), 910, sigma=10.0)).cuda()
    small = torch.from_numpy((gen.normal((1, 1, 129, 64), 911) * np.float32(1e-3)).astype(np.float32)).cuda()
    for x, signs in ((big, gen.hadamard_signs(128, 4)), (small, None), (big, None), (small, None)):
        ref8, ref_ds = fa.quant_fp8(x, signs=signs, per_tensor=True)
        got8, got_ds = _noalloc_c(fa, x, signs)
        torch.cuda.synchronize()
        assert torch.equal(got8, ref8) and torch.equal(got_ds.view(torch.int32), ref_ds.view(torch.int32))
    fa.check_device_error()


def test_noalloc_many_heads_at_the_limit(fa):
    # B * H = 65536 heads of one row: exactly the scratch limit, accepted
    x = torch.from_numpy(gen.outliers((4, 16384, 1, 64), 912)).cuda()
    ref8, ref_ds = fa.quant_fp8(x, per_tensor=True)
    got8, got_ds = _noalloc_c(fa, x, None)
    torch.cuda.synchronize()
    assert torch.equal(got8, ref8) and torch.equal(got_ds, ref_ds)
    fa.check_device_error()


def test_noalloc_timeout_is_reported_and_next_call_exact(fa):
    """A bounded wait that runs out (the test hook leaves one input slot of
    the first CTA unfilled) sets the library's error word, and the blocks it
    could not finish write +inf partials rather than keep the previous
    call's: every descale comes out infinite, and the next call is exact."""
    x = torch.from_numpy(gen.outliers((2, 4, 1000, 128), 913)).cuda()
    lib = fa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    ref8, ref_ds = fa.quant_fp8(x, per_tensor=True)
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    assert lib.fa_debug_inject(2) == fa.FA_OK
    t0 = time.time()
    _, ds = _noalloc_c(fa, x, None)
    st = lib.fa_check_device_error(stream)
    assert st == fa.FA_ERR_TIMEOUT, lib.fa_status_string(st)
    assert time.time() - t0 < 30.0
    assert torch.isinf(ds).all()
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    got8, got_ds = _noalloc_c(fa, x, None)
    assert lib.fa_check_device_error(stream) == fa.FA_OK
    assert torch.equal(got8, ref8) and torch.equal(got_ds, ref_ds)
