"""FP8 E4M3 path on the GPU against the oracle, through the C ABI.

* fa_quant_fp8 must reproduce the oracle's quantiser bit for bit (codes and
  descales), with and without the Hadamard rotation, per block and per tensor.
* fa_fwd_fp8 is fed codes made by the ORACLE quantiser (never the GPU's) and
  compared (a) with the oracle on the dequantised inputs -- LSE to 1e-3, O
  RMSE to 3e-2 (P is rounded to E4M3 in the kernel) -- and (b) with the
  oracle on the unquantised fp32 inputs: O RMSE <= 3e-2.
* Block scales + Hadamard must give a lower O RMSE than a per-tensor scale on
  inputs with rare large outliers ("FlashAttention-3: async pipelines on
  Hopper", section "why FP8 numeric tests must match the model's
  distribution").
"""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle
from gpu_util import FP8_O_RMSE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_09_gb300 as fa
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()
    return fa


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("N", [1, 127, 300, 1024])
@pytest.mark.parametrize("rot", [False, True])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_quant_bit_exact(fa, d, N, rot, per_tensor):
    x = gen.outliers((2, 3, N, d), 50 + N + d)
    signs = gen.hadamard_signs(d, 4) if rot else None
    codes_ref, ds_ref = oracle.quant_e4m3(x, signs=signs, per_tensor=per_tensor)
    codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), signs=signs, per_tensor=per_tensor)
    fa.check_device_error()
    codes = codes.cpu().numpy()
    ds = ds.cpu().numpy()
    mism = int((codes != codes_ref).sum())
    assert mism == 0, f"{mism} E4M3 codes differ from the oracle quantiser"
    assert np.array_equal(ds.view(np.uint32), ds_ref.view(np.uint32)), "descales differ"


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_quant_codes_16_byte_aligned(fa, d, per_tensor):
    # the C ABI promises 16-byte alignment of the codes only: a buffer 16 bytes
    # past a 32-byte boundary takes the 16-byte stores and must give the same
    # codes as the oracle (with the rotation, every lane holding a whole row
    # at d = 128)
    import ctypes
    x = gen.outliers((2, 3, 300, d), 70 + d)
    signs = gen.hadamard_signs(d, 4)
    codes_ref, ds_ref = oracle.quant_e4m3(x, signs=signs, per_tensor=per_tensor)
    xd = torch.from_numpy(x).cuda()
    buf = torch.zeros(x.size + 64, dtype=torch.uint8, device="cuda")
    off = (16 - buf.data_ptr() % 32) % 32
    assert (buf.data_ptr() + off) % 32 == 16
    x8 = buf[off:off + x.size]
    ds = torch.empty((2, 3, 3), dtype=torch.float32, device="cuda")
    ws = torch.empty((1,), dtype=torch.float32, device="cuda")
    keep = (ctypes.c_int8 * d)(*[int(v) for v in signs])
    st = fa.lib().fa_quant_fp8(xd.data_ptr(), x8.data_ptr(), ds.data_ptr(), 2, 3, 300, d,
                               ctypes.cast(keep, ctypes.c_void_p), int(per_tensor),
                               ws.data_ptr() if per_tensor else None, torch.cuda.current_stream().cuda_stream)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    fa.check_device_error()
    codes = x8.cpu().numpy().reshape(x.shape)
    assert int((codes != codes_ref).sum()) == 0
    assert np.array_equal(ds.cpu().numpy().view(np.uint32), ds_ref.view(np.uint32))
    # the bytes around the codes are untouched
    assert int(buf[:off].sum()) == 0 and int(buf[off + x.size:].sum()) == 0


@pytest.mark.parametrize("d", [64, 128, 256])
def test_quant_many_blocks_per_cta(fa, d):
    # about seven 128-row blocks per CTA of the persistent grid, so the
    # shared-memory ring wraps several times, in every mode
    x = gen.outliers((1, 17, 8192, d), 63 + d)    # 1088 blocks
    signs = gen.hadamard_signs(d, 4)
    for sg, per_tensor in ((None, False), (signs, False), (None, True), (signs, True)):
        codes_ref, ds_ref = oracle.quant_e4m3(x, signs=sg, per_tensor=per_tensor)
        codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), signs=sg, per_tensor=per_tensor)
        fa.check_device_error()
        assert np.array_equal(codes.cpu().numpy(), codes_ref), (sg is None, per_tensor)
        assert np.array_equal(ds.cpu().numpy(), ds_ref), (sg is None, per_tensor)


def test_quant_zero_block(fa):
    x = np.zeros((1, 1, 200, 128), dtype=np.float32)
    x[0, 0, 150, 3] = 2.0  # second block non-zero, first all zero
    codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda())
    codes_ref, ds_ref = oracle.quant_e4m3(x)
    assert np.array_equal(codes.cpu().numpy(), codes_ref)
    assert np.array_equal(ds.cpu().numpy(), ds_ref)
    assert ds_ref[0, 0, 0] == 1.0 and codes_ref[0, 0, 150, 3] == 0x7E


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_quant_exact_rounding_near_midpoints(fa, d, per_tensor):
    # values within a few ulps of s times every E4M3 midpoint: the code must
    # be the rounding of the exact quotient y / s, as rational arithmetic
    # gives it (neither the fp32 quotient nor a product with a rounded
    # reciprocal would match every one of these)
    import oracle_pins as P
    x, exp, s, _, _ = P._near_midpoint_block(d=d)
    codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), per_tensor=per_tensor)
    fa.check_device_error()
    got = codes.cpu().numpy()
    assert np.array_equal(got, exp), f"{int((got != exp).sum())} codes differ from exact rounding"
    assert ds.cpu().numpy().reshape(-1)[0] == np.float32(s)


@pytest.mark.parametrize("mag", [1e-20, 1e-30, 1e-38, 1e-41])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_quant_tiny_scales(fa, mag, per_tensor):
    # block maxima far below 1: the scale's reciprocal leaves the fp32 range
    # for the smallest ones (subnormal inputs and scales), which the kernel
    # handles exactly; bit-exact against the oracle
    x = (gen.normal((1, 2, 300, 128), 61) * np.float32(mag)).astype(np.float32)
    signs = gen.hadamard_signs(128, 4)
    for sg in (None, signs):
        codes_ref, ds_ref = oracle.quant_e4m3(x, signs=sg, per_tensor=per_tensor)
        codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), signs=sg, per_tensor=per_tensor)
        fa.check_device_error()
        assert np.array_equal(codes.cpu().numpy(), codes_ref), (mag, sg is None)
        assert np.array_equal(ds.cpu().numpy().view(np.uint32), ds_ref.view(np.uint32)), (mag, sg is None)


def test_quant_many_heads(fa):
    # 65536 heads of one row: more blocks than a 2-D grid could index by head
    x = gen.outliers((4, 16384, 1, 64), 62)
    for per_tensor in (False, True):
        codes_ref, ds_ref = oracle.quant_e4m3(x, per_tensor=per_tensor)
        codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), per_tensor=per_tensor)
        fa.check_device_error()
        assert np.array_equal(codes.cpu().numpy(), codes_ref)
        assert np.array_equal(ds.cpu().numpy(), ds_ref)


@pytest.mark.parametrize("shape", [(2, 4, 2, 300, 700, 128), (1, 3, 3, 129, 129, 64), (1, 2, 1, 1000, 257, 256),
                                   (4, 16, 16, 4096, 4096, 128)])
@pytest.mark.parametrize("rot", [False, True])
def test_quant_qkv_matches_separate_calls(fa, shape, rot):
    # fa_quant_fp8_qkv gives each tensor exactly what fa_quant_fp8 gives it
    # (Q and K rotated with the same signs, V never), GQA and Nq != Nk too
    B, Hq, Hkv, Nq, Nk, d = shape
    g = torch.Generator(device="cuda")
    g.manual_seed(900 + Nq + d)
    q = torch.randn((B, Hq, Nq, d), device="cuda", generator=g) * 3
    k = torch.randn((B, Hkv, Nk, d), device="cuda", generator=g)
    v = torch.randn((B, Hkv, Nk, d), device="cuda", generator=g) * 0.5
    signs = gen.hadamard_signs(d, 4) if rot else None
    got = fa.quant_fp8_qkv(q, k, v, signs=signs)
    ref = fa.quant_fp8(q, signs=signs) + fa.quant_fp8(k, signs=signs) + fa.quant_fp8(v)
    torch.cuda.synchronize()
    fa.check_device_error()
    for a, b in zip(got, (ref[0], ref[2], ref[4], ref[1], ref[3], ref[5])):
        assert torch.equal(a, b)


def test_quant_qkv_against_oracle_and_stream_order(fa):
    # on a side stream, the attention enqueued right after the call reads the
    # finished codes; the codes are the oracle quantiser's, bit for bit
    x = [gen.outliers((1, 2, 300, 128), 950 + i) for i in range(3)]
    signs = gen.hadamard_signs(128, 4)
    refs = [oracle.quant_e4m3(x[0], signs=signs), oracle.quant_e4m3(x[1], signs=signs), oracle.quant_e4m3(x[2])]
    xd = [torch.from_numpy(a).cuda() for a in x]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        q8, k8, v8, qs, ks, vs = fa.quant_fp8_qkv(*xd, signs=signs)
        o, lse = fa.fwd_fp8(q8, k8, v8, qs, ks, vs)
    s.synchronize()
    fa.check_device_error()
    for (c, dsc), (rc, rds) in zip(((q8, qs), (k8, ks), (v8, vs)), refs):
        assert np.array_equal(c.cpu().numpy(), rc) and np.array_equal(dsc.cpu().numpy(), rds)
    o2, lse2 = fa.fwd_fp8(*[torch.from_numpy(a).cuda() for a in (refs[0][0], refs[1][0], refs[2][0],
                                                                  refs[0][1], refs[1][1], refs[2][1])])
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_quant_qkv_cuda_graph(fa):
    x = [torch.randn((2, 4, 500, 128), device="cuda") for _ in range(3)]
    signs = gen.hadamard_signs(128, 4)
    ref = fa.quant_fp8_qkv(*x, signs=signs)
    out = tuple(torch.empty_like(t) for t in ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        fa.quant_fp8_qkv(*x, signs=signs, out=out)   # warm-up outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            fa.quant_fp8_qkv(*x, signs=signs, out=out)
    for t in out:
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    fa.check_device_error()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)


def test_quant_qkv_empty_and_errors(fa):
    q = torch.randn((1, 2, 0, 128), device="cuda")
    k = torch.randn((1, 1, 200, 128), device="cuda")
    q8, k8, v8, qs, ks, vs = fa.quant_fp8_qkv(q, k, k.clone())
    torch.cuda.synchronize()
    assert q8.numel() == 0 and torch.equal(k8, fa.quant_fp8(k)[0])
    with pytest.raises(ValueError):
        fa.quant_fp8_qkv(q, k, torch.randn((1, 1, 100, 128), device="cuda"))
    lib = fa.lib()
    p = k.data_ptr()
    bad = [p] * 9
    bad[5] = None   # v8 missing
    assert lib.fa_quant_fp8_qkv(*bad, 1, 1, 1, 200, 200, 128, None,
                                torch.cuda.current_stream().cuda_stream) == fa.FA_ERR_INVALID_ARG


def _fp8_case(fa, B, H, N, d, causal, rot, per_tensor, seed, rows=None, sigma=10.0):
    q, k, v = gen.qkv_outliers((B, H, N, d), seed, sigma=sigma)
    signs = gen.hadamard_signs(d, 4) if rot else None
    qc, qs = oracle.quant_e4m3(q, signs=signs, per_tensor=per_tensor)
    kc, ks = oracle.quant_e4m3(k, signs=signs, per_tensor=per_tensor)
    vc, vs = oracle.quant_e4m3(v, signs=None, per_tensor=per_tensor)
    dev = lambda a: torch.from_numpy(a).cuda()
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd_fp8(dev(qc), dev(kc), dev(vc), dev(qs), dev(ks), dev(vs), causal=causal, scale=scale)
    fa.check_device_error()
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, lse = o[:, :, rows], lse[:, :, rows]
    # (a) oracle on the dequantised inputs (same rotated coordinates)
    qd, kd, vd = oracle.dequant_e4m3(qc, qs), oracle.dequant_e4m3(kc, ks), oracle.dequant_e4m3(vc, vs)
    o_dq, l_dq = oracle.attn_fwd(qd, kd, vd, causal=causal, scale=scale, rows=rows)
    # (b) oracle on the unquantised fp32 inputs
    o_ex, l_ex = oracle.attn_fwd(q, k, v, causal=causal, scale=scale, rows=rows)
    rmse = lambda a, b: float(math.sqrt(((a - b) ** 2).mean()))
    return dict(rmse_dq=rmse(o, o_dq), lse_dq=float(np.abs(lse - l_dq).max()),
                rmse_exact=rmse(o, o_ex), lse_exact=float(np.abs(lse - l_ex).max()),
                finite=bool(np.isfinite(o).all() and np.isfinite(lse).all()))


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("N", [1, 130, 640])
@pytest.mark.parametrize("causal", [False, True])
def test_fwd_fp8_small(fa, d, N, causal):
    e = _fp8_case(fa, 2, 2, N, d, causal, rot=True, per_tensor=False, seed=300 + N + d)
    assert e["finite"]
    assert e["lse_dq"] <= 1e-3, e
    assert e["rmse_dq"] <= FP8_O_RMSE, e
    assert e["rmse_exact"] <= FP8_O_RMSE, e


@pytest.mark.parametrize("N", gen.FP8_N)
def test_fwd_fp8_config_sampled(fa, N):
    # the FP8 workload: B = 16384/N, H = 16, d = 128, non-causal, outliers
    B = gen.TOTAL_TOKENS // N
    rows = gen.sample_rows(N, 32, N)
    e = _fp8_case(fa, B, 16, N, 128, False, rot=True, per_tensor=False, seed=3, rows=rows)
    assert e["finite"]
    assert e["lse_dq"] <= 1e-3, e
    assert e["rmse_exact"] <= FP8_O_RMSE, e


def test_block_hadamard_beats_per_tensor(fa):
    B, H, N, d = 2, 4, 1024, 128
    rows = gen.sample_rows(N, 96, 7)
    res = {}
    for name, rot, pt in (("per_tensor", False, True), ("block", False, False), ("block_hadamard", True, False)):
        res[name] = _fp8_case(fa, B, H, N, d, False, rot=rot, per_tensor=pt, seed=3, rows=rows)
    assert res["block_hadamard"]["rmse_exact"] < res["per_tensor"]["rmse_exact"], res
    assert res["block"]["rmse_exact"] <= res["per_tensor"]["rmse_exact"] * 1.05, res


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("rot", [False, True])
@pytest.mark.parametrize("per_tensor", [False, True])
def test_quant_rope_bit_exact(fa, d, layout, rot, per_tensor):
    # rotary embedding fused into the quantisation pass: codes and descales
    # equal the oracle's (same fp32 angle tables), for both channel pairings
    N = 300                                              # ragged last block
    x = gen.outliers((2, 3, N, d), 70 + d + layout)
    cos, sin = gen.rope_tables(N, d, offset=5)
    signs = gen.hadamard_signs(d, 4) if rot else None
    codes_ref, ds_ref = oracle.quant_e4m3(x, signs=signs, per_tensor=per_tensor, rope=(cos, sin, layout))
    codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), signs=signs, per_tensor=per_tensor,
                             rope=(torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(), layout))
    fa.check_device_error()
    mism = int((codes.cpu().numpy() != codes_ref).sum())
    assert mism == 0, f"{mism} E4M3 codes differ from the oracle quantiser"
    assert np.array_equal(ds.cpu().numpy().view(np.uint32), ds_ref.view(np.uint32)), "descales differ"


@pytest.mark.parametrize("shape", [(2, 16, 4096, 128), (1, 1, 65536, 128), (4, 8, 1000, 64), (1, 3, 20000, 64),
                                   (3, 5, 777, 128)])
@pytest.mark.parametrize("layout", [1, 2])
@pytest.mark.parametrize("rot", [False, True])
def test_quant_rope_many_blocks_per_cta(fa, shape, layout, rot):
    # d = 64 and 128 stage the angle tables of one 128-row position block at
    # a time in shared memory, shared by the heads of the CTA's block range:
    # many heads per position (several per CTA), one head of 512 positions
    # (a new table for every block), ragged lengths
    B, H, N, d = shape
    x = gen.outliers(shape, 90 + N % 97 + layout)
    cos, sin = gen.rope_tables(N, d, offset=3)
    signs = gen.hadamard_signs(d, 4) if rot else None
    codes_ref, ds_ref = oracle.quant_e4m3(x, signs=signs, rope=(cos, sin, layout))
    codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), signs=signs,
                             rope=(torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(), layout))
    fa.check_device_error()
    assert np.array_equal(ds.cpu().numpy().view(np.uint32), ds_ref.view(np.uint32)), "descales differ"
    mism = int((codes.cpu().numpy() != codes_ref).sum())
    assert mism == 0, f"{mism} E4M3 codes differ from the oracle quantiser"


@pytest.mark.parametrize("d", [64, 128])
def test_quant_rope_per_tensor_many_blocks(fa, d):
    x = gen.outliers((2, 8, 3000, d), 95 + d)
    cos, sin = gen.rope_tables(3000, d, offset=1)
    signs = gen.hadamard_signs(d, 4)
    codes_ref, ds_ref = oracle.quant_e4m3(x, signs=signs, per_tensor=True, rope=(cos, sin, 2))
    codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), signs=signs, per_tensor=True,
                             rope=(torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(), 2))
    fa.check_device_error()
    assert np.array_equal(ds.cpu().numpy().view(np.uint32), ds_ref.view(np.uint32)), "descales differ"
    assert np.array_equal(codes.cpu().numpy(), codes_ref)


@pytest.mark.parametrize("layout", [1, 2])
def test_fwd_fp8_with_rope(fa, layout):
    # Q and K get the rotary embedding (and the Hadamard rotation) in the
    # quantiser; the attention then matches the fp64 oracle on the embedded,
    # unquantised inputs within the FP8 tolerance
    B, H, N, d = 2, 4, 700, 128
    q, k, v = gen.qkv_outliers((B, H, N, d), 71 + layout)
    cos, sin = gen.rope_tables(N, d)
    signs = gen.hadamard_signs(d, 4)
    dev = lambda a: torch.from_numpy(a).cuda()
    rope = (dev(cos), dev(sin), layout)
    qc, qs = fa.quant_fp8(dev(q), signs=signs, rope=rope)
    kc, ks = fa.quant_fp8(dev(k), signs=signs, rope=rope)
    vc, vs = fa.quant_fp8(dev(v))
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        o, lse = fa.fwd_fp8(qc, kc, vc, qs, ks, vs, causal=causal, scale=scale)
        fa.check_device_error()
        o_ex, l_ex = oracle.attn_fwd(oracle.rope(q, cos, sin, layout), oracle.rope(k, cos, sin, layout), v,
                                     causal=causal, scale=scale)
        rmse = float(np.sqrt(((o.float().cpu().numpy() - o_ex) ** 2).mean()))
        assert np.isfinite(rmse) and rmse <= FP8_O_RMSE, (causal, rmse)


@pytest.mark.parametrize("sigma", [10.0, 100.0])
def test_fp8_error_study(fa, sigma):
    """The FP8 error study at the FP8 workloads (B = 16384 / N, H = 16,
    d = 128, N in {1k, 4k, 16k}, non-causal): inputs N(0,1) plus rare
    outliers N(0, sigma^2) (sigma = 10 is the workload's reading; 100 the
    other reading of its notation), quantised on the GPU three ways --
    per-tensor scale, block scales, block scales + Hadamard on Q and K --
    then FP8 attention; O RMSE against the fp64 oracle on the unquantised
    inputs over 64 sampled query rows of every head.  Block + Hadamard must
    beat the per-tensor baseline (the pages report 2.6x on H100 as context,
    not as a bar).  With FA_REPORT_DIR set, the figures are written there as
    JSON."""
    import json
    import os
    d, H = 128, 16
    signs = gen.hadamard_signs(d, 4)
    report = {}
    for N in gen.FP8_N:
        B = gen.TOTAL_TOKENS // N
        rows = gen.sample_rows(N, 64, 8)
        q, k, v = gen.qkv_outliers((B, H, N, d), 3, sigma=sigma)
        o_ref, _ = oracle.attn_fwd(q, k, v, causal=False, scale=1.0 / math.sqrt(d), rows=rows)
        qd, kd, vd = (torch.from_numpy(a).cuda() for a in (q, k, v))
        res = {}
        for name, rot, pt in (("per_tensor", False, True), ("block", False, False),
                              ("block_hadamard", True, False)):
            sg = signs if rot else None
            q8, qs = fa.quant_fp8(qd, signs=sg, per_tensor=pt)
            k8, ks = fa.quant_fp8(kd, signs=sg, per_tensor=pt)
            v8, vs = fa.quant_fp8(vd, per_tensor=pt)
            o, _ = fa.fwd_fp8(q8, k8, v8, qs, ks, vs, causal=False, scale=1.0 / math.sqrt(d))
            fa.check_device_error()
            og = o.float().cpu().numpy().astype(np.float64)[:, :, rows]
            res[name] = float(math.sqrt(((og - o_ref) ** 2).mean()))
        res["ratio_per_tensor_over_block_hadamard"] = res["per_tensor"] / res["block_hadamard"]
        report[f"N{N}"] = res
        assert res["block_hadamard"] < res["per_tensor"], (N, res)
        if sigma == 10.0:
            assert res["block_hadamard"] <= FP8_O_RMSE and res["block"] <= FP8_O_RMSE, (N, res)
        del qd, kd, vd
    print(f"\nFP8 error study, sigma = {sigma}: {json.dumps(report)}")
    out = os.environ.get("FA_REPORT_DIR")
    if out:
        os.makedirs(out, exist_ok=True)
        with open(os.path.join(out, f"fp8_error_study_sigma{int(sigma)}.json"), "w") as f:
            json.dump({"sigma": sigma, "rows_per_head": 64, "rmse_vs_fp64_oracle": report}, f, indent=1)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_fp8_rising_maxima(fa, causal):
    # keys scaled up along the sequence (0.2x to 3x) with scale 0.5: every
    # row's running maximum rises past the lazy threshold many times, so O is
    # rescaled in TMEM again and again and P~ runs up to the top of the E4M3
    # range.  LSE comes from fp32 p, m and l and must match the oracle on the
    # dequantised inputs to 1e-3; O may differ from it only by the E4M3
    # rounding of P~ -- at most half an E4M3 step of each weight, 2^-4
    # relative for normal values (at most 2^-4 of max|V| on O, as l >= 1) and
    # 2^-10 absolute in P~ units for subnormal ones (at most N * 2^-15 of
    # 448 * max s_V ~ max|V|) -- plus its bf16 output rounding.
    B, H, N, d = 1, 2, 1024, 128
    q, k, v = (gen.normal((B, H, N, d), 2200, s) for s in range(3))
    k = (k * np.linspace(0.2, 3.0, N, dtype=np.float32)[None, None, :, None]).astype(np.float32)
    signs = gen.hadamard_signs(d, 4)
    qc, qs = oracle.quant_e4m3(q, signs=signs)
    kc, ks = oracle.quant_e4m3(k, signs=signs)
    vc, vs = oracle.quant_e4m3(v)
    dev = lambda a: torch.from_numpy(a).cuda()
    o, lse = fa.fwd_fp8(dev(qc), dev(kc), dev(vc), dev(qs), dev(ks), dev(vs), causal=causal, scale=0.5)
    fa.check_device_error()
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    qd, kd, vd = oracle.dequant_e4m3(qc, qs), oracle.dequant_e4m3(kc, ks), oracle.dequant_e4m3(vc, vs)
    o_dq, l_dq = oracle.attn_fwd(qd, kd, vd, causal=causal, scale=0.5)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    assert np.abs(lse - l_dq).max() <= 1e-3
    # the maxima really rise by many lazy-threshold steps along the rows
    s_end = 0.5 * math.log2(math.e) * np.einsum("bhd,bhnd->bhn", qd[:, :, -1], kd).max()
    s_start = 0.5 * math.log2(math.e) * np.einsum("bhd,bhnd->bhn", qd[:, :, -1], kd[:, :, :128]).max()
    assert s_end - s_start > 4 * 3.8
    bound = (2.0 ** -4 * np.abs(vd).max() + N * 2.0 ** -15 * 448 * float(vs.max())) * 1.05 \
        + 2.0 ** -8 * np.abs(o_dq).max()
    assert np.abs(o - o_dq).max() <= bound, (np.abs(o - o_dq).max(), bound)
