"""Attention backward (fa_bwd) against the fp64 oracle's gradients.

The backward kernel gets the forward's O and LSE as inputs.  The parity
tests give it the oracle's (O rounded to the element type like the forward's
output, LSE in fp32), so that what is measured is the backward kernel's own
error; ``test_bwd_end_to_end`` chains the GPU forward into it, as in
training.  The oracle differentiates the definition directly from the same
low-precision q, k, v, dO.  Errors are normalised by the reference: the
largest error by the largest |reference| entry, the rms error by the
reference's rms.  Bounds come from the element type's unit roundoff u (2^-8
bf16, 2^-11 fp16): the outputs are rounded once (up to u/2 relative), P and
dS are rounded to the element type before their products, and D = dO . O
inherits O's rounding (a per-row error that grows as the softmax gets
peakier); the bounds allow 2.5 u for the largest error and 1.25 u for the
rms.  A CPU emulation of exactly these roundings gives up to 1.6 u and
0.9 u over the scales tested here.
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle
from gpu_util import bwd_check as _check

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
    do = torch.from_numpy(gen.normal((B, Hq, Nq, d), seed, 3)).to(dtype)
    return q, k, v, do


def _gpu_grads(fa, q, k, v, do, causal, scale, forward="oracle"):
    """GPU gradients; O and LSE from the oracle (rounded like the kernel's
    outputs) or, with forward="gpu", from the GPU forward."""
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    if forward == "gpu":
        o, lse = fa.fwd_gqa(qd, kd, vd, causal=causal, scale=scale)
    else:
        o64, l64 = oracle.attn_fwd(q, k, v, causal=causal, scale=scale)
        o = torch.from_numpy(o64).to(q.dtype).cuda()
        lse = torch.from_numpy(l64).to(torch.float32).cuda()
    dq, dk, dv = fa.bwd(qd, kd, vd, o, lse, dod, causal=causal, scale=scale)
    fa.check_device_error()
    return dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk", [
    (1, 2, 2, 128, 128),    # one key tile, two query tiles
    (2, 2, 2, 200, 200),    # ragged tails of both
    (1, 4, 2, 256, 384),    # grouped queries, Nq != Nk
    (1, 2, 2, 100, 300),    # few queries, many keys
    (1, 2, 2, 300, 100),    # causal: the first 200 rows see no key
    (1, 3, 1, 64, 64),      # multi-query
    (1, 1, 1, 1, 1),        # smallest
    (1, 2, 1, 37, 1000),    # short queries against a long sequence
])
def test_bwd_parity(fa, d, dtype, causal, B, Hq, Hkv, Nq, Nk):
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = _inputs(B, Hq, Hkv, Nq, Nk, d, 900 + Nq + 7 * Nk + Hkv + d, dtype)
    got = _gpu_grads(fa, q, k, v, do, causal, scale)
    ref = oracle.attn_bwd(q, k, v, do, causal=causal, scale=scale)
    _check(got, ref, dtype, f"d={d} B={B} Hq={Hq} Hkv={Hkv} Nq={Nq} Nk={Nk} causal={causal} {dtype}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("scale", [0.0, -0.2, 0.3])
def test_bwd_scales(fa, d, scale):
    q, k, v, do = _inputs(1, 2, 2, 192, 192, d, 77, torch.bfloat16)
    for causal in (False, True):
        got = _gpu_grads(fa, q, k, v, do, causal, scale)
        ref = oracle.attn_bwd(q, k, v, do, causal=causal, scale=scale)
        _check(got, ref, torch.bfloat16, f"scale={scale} causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_end_to_end(fa, d, dtype, causal):
    """GPU forward -> GPU backward at the usual scale 1/sqrt(d)."""
    q, k, v, do = _inputs(2, 4, 2, 333, 333, d, 4242, dtype)
    got = _gpu_grads(fa, q, k, v, do, causal, 1.0 / math.sqrt(d), forward="gpu")
    ref = oracle.attn_bwd(q, k, v, do, causal=causal, scale=1.0 / math.sqrt(d))
    _check(got, ref, dtype, f"end to end causal={causal} {dtype}")


@pytest.mark.parametrize("B,H,N,d", [(4, 16, 2048, 128), (4, 32, 2048, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_mid_sampled_heads(fa, B, H, N, d, causal):
    """The benchmark's backward workloads (N=2048, bf16; d=128 with H=16,
    d=64 with H=32) in one call; the oracle checks whole heads (every
    gradient entry of the head), the first and the last."""
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = _inputs(B, H, H, N, N, d, 1234, torch.bfloat16)
    dq, dk, dv = _gpu_grads(fa, q, k, v, do, causal, scale, forward="gpu")
    for b, h in ((0, 0), (B - 1, H - 1)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.attn_bwd(q[sl], k[sl], v[sl], do[sl], causal=causal, scale=scale)
        _check((dq[sl], dk[sl], dv[sl]), ref, torch.bfloat16, f"mid head ({b},{h}) causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_repeatable_dk_dv(fa, d):
    """dK and dV are summed in a fixed order inside one CTA: bit-identical
    over repeated calls (dQ is added across CTAs in any order)."""
    q, k, v, do = _inputs(1, 4, 2, 320, 320, d, 55, torch.bfloat16)
    a = _gpu_grads(fa, q, k, v, do, True, 0.1)
    b = _gpu_grads(fa, q, k, v, do, True, 0.1)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_cuda_graph(fa, d):
    """fa_bwd is capturable: a replayed graph gives the eager result (dK, dV
    bit for bit; dQ within fp32 reduce-add reordering)."""
    q, k, v, do = (t.cuda() for t in _inputs(2, 4, 4, 256, 256, d, 66, torch.bfloat16))
    o, lse = fa.fwd(q, k, v, causal=True)
    ws = torch.empty(fa.bwd_workspace_bytes(2, 4, 256, d), dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa.bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
    ref = (dq.clone(), dk.clone(), dv.clone())
    for t in (dq, dk, dv):
        t.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fa.bwd(q, k, v, o, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    fa.check_device_error()
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert (dq.float() - ref[0].float()).abs().max().item() <= 1e-2 * ref[0].float().abs().max().item()


def test_bwd_no_query(fa):
    k = torch.randn(1, 2, 130, 128, device="cuda").to(torch.bfloat16)
    v = torch.randn_like(k)
    q = torch.empty(1, 2, 0, 128, device="cuda", dtype=torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty(1, 2, 0, device="cuda", dtype=torch.float32)
    dk = torch.full_like(k, 7.0)
    dv = torch.full_like(v, 7.0)
    fa.bwd(q, k, v, o, lse, torch.empty_like(q), dk=dk, dv=dv)
    fa.check_device_error()
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0


def test_bwd_rejects(fa):
    q = torch.randn(1, 1, 64, 256, device="cuda").to(torch.bfloat16)
    o, lse = fa.fwd(q, q, q)
    with pytest.raises(fa.FaError) as ei:
        fa.bwd(q, q, q, o, lse, q)
    assert ei.value.status == fa.FA_ERR_UNSUPPORTED
    q = torch.randn(1, 1, 64, 128, device="cuda").to(torch.bfloat16)
    o, lse = fa.fwd(q, q, q)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError) as ei:
        fa.bwd(q, q, q, o, lse, q, workspace=small)
    assert ei.value.status == fa.FA_ERR_INVALID_ARG
