"""Seeded random shapes through the C ABI against the fp64 oracle on sampled
query rows: BF16/FP16 forward (any head dimension, grouped heads, Nq != Nk,
causal or not, the default scale, 0, a negative and an enlarged scale), the
E4M3 quantiser bit for bit (also with the rotary embedding), the FP8 forward
on its codes, the split-KV forward (with the split-KV tests' element-wise
bound), the host-buffer forward (bit-identical to the device call), and the
backward (whole gradients, with the backward tests' bounds).  The shapes
come from one fixed generator, so a failure names a case that reruns
exactly; they fill the gaps between the hand-picked sizes of the other
parity tests (odd lengths, lengths below one tile, one head per group)."""
import math

import numpy as np
import pytest
import torch

import attn_inputs as gen
import oracle
from gpu_util import FP8_O_RMSE, LSE_ABS, O_MAXABS, bwd_check

pytestmark = pytest.mark.gpu


def _draw_fwd(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    for i in range(n):
        d = int(rng.choice([64, 128, 256]))
        g = int(rng.choice([1, 1, 2, 4]))
        Hkv = int(rng.integers(1, 3))
        Nq = int(rng.integers(1, 1500))
        Nk = int(rng.choice([Nq, int(rng.integers(1, 1500))]))
        scale = float(rng.choice([1.0 / math.sqrt(d), 0.0, -0.2, 0.3]))
        cases.append(dict(i=i, B=int(rng.integers(1, 3)), Hq=Hkv * g, Hkv=Hkv, Nq=Nq, Nk=Nk, d=d,
                          causal=bool(rng.integers(0, 2)), scale=scale,
                          fp16=bool(rng.integers(0, 2)), rows_seed=int(rng.integers(1 << 30))))
    return cases


def _draw_quant(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [dict(i=i, d=int(rng.choice([64, 128, 256])), N=int(rng.integers(1, 900)),
                 B=int(rng.integers(1, 3)), H=int(rng.integers(1, 4)), rot=bool(rng.integers(0, 2)),
                 per_tensor=bool(rng.integers(0, 2))) for i in range(n)]


def _draw_fp8(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    for i in range(n):
        d = int(rng.choice([128, 256]))
        g = int(rng.choice([1, 2, 4]))
        Hkv = int(rng.integers(1, 3))
        Nq = int(rng.integers(1, 1300))
        Nk = int(rng.choice([Nq, int(rng.integers(1, 1300))]))
        cases.append(dict(i=i, B=int(rng.integers(1, 3)), Hq=Hkv * g, Hkv=Hkv, Nq=Nq, Nk=Nk, d=d,
                          causal=bool(rng.integers(0, 2)), rot=bool(rng.integers(0, 2)),
                          rows_seed=int(rng.integers(1 << 30))))
    return cases


def _draw_bwd(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    for i in range(n):
        d = int(rng.choice([64, 128]))
        g = int(rng.choice([1, 2, 4]))
        Hkv = int(rng.integers(1, 3))
        Nq = int(rng.integers(1, 500))
        Nk = int(rng.choice([Nq, int(rng.integers(1, 500))]))
        cases.append(dict(i=i, B=int(rng.integers(1, 3)), Hq=Hkv * g, Hkv=Hkv, Nq=Nq, Nk=Nk, d=d,
                          causal=bool(rng.integers(0, 2)),
                          scale=float(rng.choice([1.0 / math.sqrt(d), 0.0, -0.2, 0.3])),
                          fp16=bool(rng.integers(0, 2))))
    return cases


def _draw_splitkv(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    for i in range(n):
        Hkv = int(rng.integers(1, 3))
        g = int(rng.choice([1, 2, 4, 8]))
        Nq = int(rng.choice([1, int(rng.integers(1, 17)), int(rng.integers(1, 300))]))
        cases.append(dict(i=i, B=int(rng.integers(1, 3)), Hq=Hkv * g, Hkv=Hkv, Nq=Nq,
                          Nk=int(rng.integers(1, 6000)), d=int(rng.choice([64, 128, 256])),
                          causal=bool(rng.integers(0, 2)), splits=int(rng.choice([0, 1, 2, 3, 7, 64])),
                          rows_seed=int(rng.integers(1 << 30))))
    return cases


def _draw_rope(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return [dict(i=i, d=int(rng.choice([64, 128, 256])), N=int(rng.integers(1, 3000)),
                 B=int(rng.integers(1, 3)), H=int(rng.integers(1, 5)), layout=int(rng.integers(1, 3)),
                 rot=bool(rng.integers(0, 2)), per_tensor=bool(rng.integers(0, 2))) for i in range(n)]


def _draw_host(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    cases = []
    for i in range(n):
        Hkv = int(rng.integers(1, 3))
        Nq = int(rng.integers(1, 2000))
        cases.append(dict(i=i, B=int(rng.integers(1, 3)), Hq=Hkv * int(rng.choice([1, 2])), Hkv=Hkv, Nq=Nq,
                          Nk=int(rng.choice([Nq, int(rng.integers(1, 2000))])), d=int(rng.choice([64, 128, 256])),
                          causal=bool(rng.integers(0, 2)), pinned=bool(rng.integers(0, 2))))
    return cases


FWD = _draw_fwd(150, 20261203)
SPLITKV = _draw_splitkv(30, 20261207)
ROPE = _draw_rope(24, 20261208)
HOST = _draw_host(12, 20261209)
BWD = _draw_bwd(40, 20261206)
QUANT = _draw_quant(40, 20261204)
FP8 = _draw_fp8(60, 20261205)


def _ids(cases):
    return [",".join(f"{k}={v}" for k, v in c.items() if k != "rows_seed") for c in cases]


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_09_gb300 as fa
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()
    return fa


def _rows(Nq, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.unique(np.concatenate([rng.integers(0, Nq, 24), [0, Nq - 1]]))


def _check_lse(lse, l_ref, tol, what):
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: rows without keys must have LSE = -inf"
    if (~empty).any():
        e = np.abs(lse[~empty] - l_ref[~empty]).max()
        assert e <= tol, f"{what}: max|dLSE| = {e:.3e}"


@pytest.mark.parametrize("c", FWD, ids=_ids(FWD))
def test_random_fwd(fa, c):
    dt = torch.float16 if c["fp16"] else torch.bfloat16
    B, Hq, Hkv, Nq, Nk, d = c["B"], c["Hq"], c["Hkv"], c["Nq"], c["Nk"], c["d"]
    seed = 5000 + c["i"]
    q = torch.from_numpy(gen.normal((B, Hq, Nq, d), seed, 0)).to(dt)
    k = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 1)).to(dt)
    v = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 2)).to(dt)
    o, lse = fa.fwd_gqa(q.cuda(), k.cuda(), v.cuda(), causal=c["causal"], scale=c["scale"])
    fa.check_device_error()
    rows = _rows(Nq, c["rows_seed"])
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=c["causal"], scale=c["scale"], rows=rows)
    o = o.float().cpu().numpy().astype(np.float64)[:, :, rows]
    lse = lse.cpu().numpy().astype(np.float64)[:, :, rows]
    assert np.isfinite(o).all()
    _check_lse(lse, l_ref, LSE_ABS, "forward")
    # at |scale| above 1/sqrt(d) the softmax is peakier and one rounded P
    # weight carries more of O, so the bound doubles there
    tol = O_MAXABS if c["scale"] == 1.0 / math.sqrt(d) or c["scale"] == 0.0 else 2 * O_MAXABS
    e = np.abs(o - o_ref).max()
    assert e <= tol, f"forward: max|dO| = {e:.3e}"


@pytest.mark.parametrize("c", QUANT, ids=_ids(QUANT))
def test_random_quant(fa, c):
    x = gen.outliers((c["B"], c["H"], c["N"], c["d"]), 7000 + c["i"])
    signs = gen.hadamard_signs(c["d"], 4) if c["rot"] else None
    codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), signs=signs, per_tensor=c["per_tensor"])
    fa.check_device_error()
    rc, rs = oracle.quant_e4m3(x, signs=signs, per_tensor=c["per_tensor"])
    assert np.array_equal(ds.cpu().numpy(), rs), "descales"
    assert np.array_equal(codes.cpu().numpy(), rc), "codes"


@pytest.mark.parametrize("c", FP8, ids=_ids(FP8))
def test_random_fp8(fa, c):
    B, Hq, Hkv, Nq, Nk, d = c["B"], c["Hq"], c["Hkv"], c["Nq"], c["Nk"], c["d"]
    seed = 9000 + c["i"]
    signs = gen.hadamard_signs(d, 4) if c["rot"] else None
    xq = gen.outliers((B, Hq, Nq, d), seed, 0)
    xk = gen.outliers((B, Hkv, Nk, d), seed, 1)
    xv = gen.outliers((B, Hkv, Nk, d), seed, 2)
    # codes from the oracle quantiser, so this case does not depend on the
    # quantiser kernel
    qc, qs = oracle.quant_e4m3(xq, signs=signs)
    kc, ks = oracle.quant_e4m3(xk, signs=signs)
    vc, vs = oracle.quant_e4m3(xv)
    dev = lambda a: torch.from_numpy(a).cuda()
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd_fp8_gqa(dev(qc), dev(kc), dev(vc), dev(qs), dev(ks), dev(vs), causal=c["causal"], scale=scale)
    fa.check_device_error()
    rows = _rows(Nq, c["rows_seed"])
    deq = [oracle.dequant_e4m3(a, s) for a, s in ((qc, qs), (kc, ks), (vc, vs))]
    o_ref, l_ref = oracle.attn_fwd(*deq, causal=c["causal"], scale=scale, rows=rows)
    o = o.float().cpu().numpy().astype(np.float64)[:, :, rows]
    lse = lse.cpu().numpy().astype(np.float64)[:, :, rows]
    assert np.isfinite(o).all()
    _check_lse(lse, l_ref, LSE_ABS, "fp8 forward")
    rmse = math.sqrt(float(((o - o_ref) ** 2).mean()))
    assert rmse <= FP8_O_RMSE, f"fp8 forward: O rmse = {rmse:.3e}"


@pytest.mark.parametrize("c", BWD, ids=_ids(BWD))
def test_random_bwd(fa, c):
    # the backward gets the oracle's O (rounded to the element type) and LSE,
    # so that its own error is measured, as in the backward tests
    dt = torch.float16 if c["fp16"] else torch.bfloat16
    B, Hq, Hkv, Nq, Nk, d = c["B"], c["Hq"], c["Hkv"], c["Nq"], c["Nk"], c["d"]
    seed = 11000 + c["i"]
    q = torch.from_numpy(gen.normal((B, Hq, Nq, d), seed, 0)).to(dt)
    k = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 1)).to(dt)
    v = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 2)).to(dt)
    do = torch.from_numpy(gen.normal((B, Hq, Nq, d), seed, 3)).to(dt)
    o64, l64 = oracle.attn_fwd(q, k, v, causal=c["causal"], scale=c["scale"])
    o = torch.from_numpy(o64).to(dt).cuda()
    lse = torch.from_numpy(l64).to(torch.float32).cuda()
    got = fa.bwd(q.cuda(), k.cuda(), v.cuda(), o, lse, do.cuda(), causal=c["causal"], scale=c["scale"])
    fa.check_device_error()
    ref = oracle.attn_bwd(q, k, v, do, causal=c["causal"], scale=c["scale"])
    bwd_check(got, ref, dt, "backward")


@pytest.mark.parametrize("c", SPLITKV, ids=_ids(SPLITKV))
def test_random_splitkv(fa, c):
    B, Hq, Hkv, Nq, Nk, d = c["B"], c["Hq"], c["Hkv"], c["Nq"], c["Nk"], c["d"]
    seed = 13000 + c["i"]
    q = torch.from_numpy(gen.normal((B, Hq, Nq, d), seed, 0)).to(torch.bfloat16)
    k = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 1)).to(torch.bfloat16)
    v = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 2)).to(torch.bfloat16)
    o, lse = fa.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), causal=c["causal"], num_splits=c["splits"])
    fa.check_device_error()
    rows = _rows(Nq, c["rows_seed"])
    o_ref, l_ref = oracle.attn_fwd(q, k, v, causal=c["causal"], rows=rows)
    o = o.float().cpu().numpy().astype(np.float64)[:, :, rows]
    lse = lse.cpu().numpy().astype(np.float64)[:, :, rows]
    assert np.isfinite(o).all()
    _check_lse(lse, l_ref, LSE_ABS, "split-KV")
    # runs merged by their LSE weights in fp32: the split-KV tests' bound,
    # 2^-8 (|O| + max|V|) + 1e-4 per element
    vmax = float(np.abs(v.float().numpy()).max())
    tol = 2.0 ** -8 * (np.abs(o_ref) + vmax) + 1e-4
    assert (np.abs(o - o_ref) <= tol).all(), f"split-KV: {int((np.abs(o - o_ref) > tol).sum())} beyond the bound"


@pytest.mark.parametrize("c", ROPE, ids=_ids(ROPE))
def test_random_rope_quant(fa, c):
    B, H, N, d = c["B"], c["H"], c["N"], c["d"]
    x = gen.outliers((B, H, N, d), 15000 + c["i"])
    cos, sin = gen.rope_tables(N, d, offset=c["i"])
    signs = gen.hadamard_signs(d, 4) if c["rot"] else None
    rc, rs = oracle.quant_e4m3(x, signs=signs, per_tensor=c["per_tensor"], rope=(cos, sin, c["layout"]))
    codes, ds = fa.quant_fp8(torch.from_numpy(x).cuda(), signs=signs, per_tensor=c["per_tensor"],
                             rope=(torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(), c["layout"]))
    fa.check_device_error()
    assert np.array_equal(ds.cpu().numpy().view(np.uint32), rs.view(np.uint32)), "descales"
    assert np.array_equal(codes.cpu().numpy(), rc), "codes"


@pytest.mark.parametrize("c", HOST, ids=_ids(HOST))
def test_random_host(fa, c):
    B, Hq, Hkv, Nq, Nk, d = c["B"], c["Hq"], c["Hkv"], c["Nq"], c["Nk"], c["d"]
    seed = 17000 + c["i"]
    q, k, v = (torch.from_numpy(gen.normal(shape, seed, j)).to(torch.bfloat16)
               for j, shape in enumerate(((B, Hq, Nq, d), (B, Hkv, Nk, d), (B, Hkv, Nk, d))))
    if c["pinned"]:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_dev, l_dev = fa.fwd_gqa(q.cuda(), k.cuda(), v.cuda(), causal=c["causal"])
    o_h, l_h = fa.fwd_host(q, k, v, causal=c["causal"])
    torch.cuda.current_stream().synchronize()
    fa.check_device_error()
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(l_h, l_dev.cpu()), "host path differs from the device path"
