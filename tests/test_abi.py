"""The C-ABI library loads, exports every entry point include/fa.h declares,
and rejects bad arguments on the host (CPU only: no compute call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa_lib():
    from exact_attention_forward_09_gb300 import build
    build.build()
    import exact_attention_forward_09_gb300 as fa
    return fa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_fp8", "fa_quant_fp8", "fa_status_string", "fa_check_device_error"):
        assert n in names


def test_every_declared_symbol_is_exported(fa_lib):
    for name in declared_functions():
        assert hasattr(fa_lib, name), f"{name} declared in fa.h but not exported by libfa.so"


def test_symbols_are_plain_c(fa_lib):
    # extern "C": the unmangled name resolves
    for name in declared_functions():
        ctypes.cast(getattr(fa_lib, name), ctypes.c_void_p)


def test_status_strings(fa_lib):
    for code in range(5):
        s = fa_lib.fa_status_string(code).decode()
        assert s.startswith("FA_")
    assert fa_lib.fa_status_string(99).decode() == "FA_ERR_UNKNOWN"
    assert fa_lib.fa_version() >= 100


def test_host_argument_checks(fa_lib):
    import exact_attention_forward_09_gb300 as fa
    p = 1 << 20  # any 16-byte-aligned non-null value: these calls return before any CUDA call
    # negative size
    assert fa_lib.fa_fwd(p, p, p, p, p, -1, 1, 1, 64, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    # non-finite scale
    assert fa_lib.fa_fwd(p, p, p, p, p, 1, 1, 1, 64, 0, float("nan"), 0, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd(p, p, p, p, p, 1, 1, 1, 64, 0, float("inf"), 0, None) == fa.FA_ERR_INVALID_ARG
    # bad dtype / causal flag
    assert fa_lib.fa_fwd(p, p, p, p, p, 1, 1, 1, 64, 0, 0.1, 7, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd(p, p, p, p, p, 1, 1, 1, 64, 2, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    # unsupported head dimension
    assert fa_lib.fa_fwd(p, p, p, p, p, 1, 1, 1, 96, 0, 0.1, 0, None) == fa.FA_ERR_UNSUPPORTED
    # null / misaligned pointers
    assert fa_lib.fa_fwd(None, p, p, p, p, 1, 1, 1, 64, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd(p + 2, p, p, p, p, 1, 1, 1, 64, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    # empty problem: a no-op, even with null pointers
    assert fa_lib.fa_fwd(None, None, None, None, None, 0, 4, 128, 64, 0, 0.1, 0, None) == fa.FA_OK
    assert fa_lib.fa_fwd(None, None, None, None, None, 2, 4, 0, 128, 1, 0.1, 1, None) == fa.FA_OK
    # FP8: d = 64 unsupported, missing descales invalid
    assert fa_lib.fa_fwd_fp8(p, p, p, p, p, 1, 1, 1, 64, 0, 0.1, p, p, p, None) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_fwd_fp8(p, p, p, p, p, 1, 1, 1, 128, 0, 0.1, None, p, p, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_fp8(None, None, None, None, None, 0, 1, 1, 128, 0, 0.1, None, None, None,
                             None) == fa.FA_OK
    # grouped-query entry point: Hq must be a multiple of Hkv, Nk >= 1
    assert fa_lib.fa_fwd_gqa(p, p, p, p, p, 1, 6, 4, 8, 8, 64, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_gqa(p, p, p, p, p, 1, 4, 0, 8, 8, 64, 0, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_gqa(p, p, p, p, p, 1, 4, 2, 8, 0, 64, 1, 0.1, 0, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_gqa(None, None, None, None, None, 1, 4, 2, 0, 9, 64, 1, 0.1, 0, None) == fa.FA_OK
    assert fa_lib.fa_fwd_fp8_gqa(p, p, p, p, p, 1, 4, 2, 8, 8, 64, 0, 0.1, p, p, p, None) == fa.FA_ERR_UNSUPPORTED
    # quantiser
    assert fa_lib.fa_quant_fp8(p, p, p, 1, 1, 1, 100, None, 0, None, None) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_quant_fp8(p, p, p, 1, 1, 1, 128, None, 1, None, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_quant_fp8(p, p, p, 1, 1, 1, 128, None, 3, None, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_quant_fp8(None, None, None, 1, 0, 1, 128, None, 0, None, None) == fa.FA_OK
    # split-KV: a negative split count or a bad dtype is refused, an empty problem is a no-op
    assert fa_lib.fa_fwd_splitkv(p, p, p, p, p, 1, 4, 2, 1, 100, 128, 0, 0.1, 0, -1, None, 0,
                                 None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_splitkv(p, p, p, p, p, 1, 4, 2, 1, 100, 128, 0, 0.1, 5, 0, None, 0,
                                 None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_splitkv(None, None, None, None, None, 1, 4, 2, 0, 100, 128, 0, 0.1, 0, 0, None, 0,
                                 None) == fa.FA_OK
    nbytes = ctypes.c_size_t(7)
    assert fa_lib.fa_splitkv_workspace_bytes(1, 4, 2, 1, 100, 96, 0, ctypes.byref(nbytes)) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_splitkv_workspace_bytes(1, 4, 3, 1, 100, 128, 0, ctypes.byref(nbytes)) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_splitkv_workspace_bytes(0, 4, 2, 1, 100, 128, 0, ctypes.byref(nbytes)) == fa.FA_OK
    assert nbytes.value == 0
    # Q, K and V in one call: every tensor is checked before anything runs
    z = [None] * 9
    pp = [p] * 9
    assert fa_lib.fa_quant_fp8_qkv(*pp[:8], None, 1, 2, 1, 128, 256, 128, None, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_quant_fp8_qkv(p, p, p + 4, *pp[:6], 1, 2, 1, 128, 256, 128, None,
                                   None) == fa.FA_ERR_INVALID_ARG  # v 16-byte aligned
    assert fa_lib.fa_quant_fp8_qkv(*pp, 1, 2, 1, 128, 256, 96, None, None) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_quant_fp8_qkv(*pp, 1, 2, -1, 128, 256, 128, None, None) == fa.FA_ERR_INVALID_ARG
    bad = (ctypes.c_int8 * 128)(*([1] * 127 + [0]))
    assert fa_lib.fa_quant_fp8_qkv(*pp, 1, 2, 1, 128, 256, 128, ctypes.cast(bad, ctypes.c_void_p),
                                   None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_quant_fp8_qkv(*z, 0, 2, 1, 128, 256, 128, None, None) == fa.FA_OK
    # quantiser with rotary embedding: a known layout and both tables are required
    assert fa_lib.fa_quant_fp8_rope(p, p, p, 1, 1, 1, 128, p, p, 0, None, 0, None, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_quant_fp8_rope(p, p, p, 1, 1, 1, 128, p, p, 3, None, 0, None, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_quant_fp8_rope(p, p, p, 1, 1, 1, 128, None, p, fa.FA_ROPE_HALF, None, 0, None,
                                    None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_quant_fp8_rope(p, p, p, 1, 1, 1, 128, p, p + 2, fa.FA_ROPE_INTERLEAVED, None, 0, None,
                                    None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_quant_fp8_rope(p, p, p, 1, 1, 1, 128, p + 8, p, fa.FA_ROPE_HALF, None, 0, None,
                                    None) == fa.FA_ERR_INVALID_ARG  # tables must be 16-byte aligned
    assert fa_lib.fa_quant_fp8_rope(p, p, p, 1, 1, 1, 100, p, p, fa.FA_ROPE_HALF, None, 0, None,
                                    None) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_quant_fp8_rope(None, None, None, 0, 1, 1, 128, None, None, fa.FA_ROPE_HALF, None, 0, None,
                                    None) == fa.FA_OK
    # backward: d = 64 or 128; workspace present, aligned and large enough; empty batch a no-op
    ws = 1 << 24
    assert fa_lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 2, 2, 64, 64, 256, 0, 0.1, 0, ws, 1 << 20,
                         None) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 2, 2, 64, 64, 96, 0, 0.1, 0, ws, 1 << 20,
                         None) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 2, 2, 64, 64, 128, 0, 0.1, 0, None, 1 << 20,
                         None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 2, 2, 64, 64, 128, 0, 0.1, 0, ws + 16, 1 << 20,
                         None) == fa.FA_ERR_INVALID_ARG  # 256-byte alignment
    assert fa_lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 2, 2, 64, 64, 128, 0, 0.1, 0, ws, 100,
                         None) == fa.FA_ERR_INVALID_ARG  # too small
    assert fa_lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 3, 2, 64, 64, 128, 0, 0.1, 0, ws, 1 << 20,
                         None) == fa.FA_ERR_INVALID_ARG  # Hq % Hkv
    assert fa_lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 2, 2, 64, 64, 128, 2, 0.1, 0, ws, 1 << 20,
                         None) == fa.FA_ERR_INVALID_ARG  # causal flag
    assert fa_lib.fa_bwd(p, p, p, p, p + 4, p, p, p, p, 1, 2, 2, 64, 64, 128, 0, 0.1, 0, ws, 1 << 20,
                         None) == fa.FA_ERR_INVALID_ARG  # misaligned lse
    assert fa_lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 2, 2, 64, 64, 128, 0, float("nan"), 0, ws, 1 << 20,
                         None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_bwd(None, None, None, None, None, None, None, None, None, 0, 2, 2, 64, 64, 128, 0, 0.1, 0,
                         None, 0, None) == fa.FA_OK
    # host-buffer forward: workspace present, aligned and large enough; empty batch a no-op
    assert fa_lib.fa_fwd_host(p, p, p, p, p, 1, 2, 2, 64, 64, 128, 0, 0.1, 0, None, 1 << 20,
                              None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_host(p, p, p, p, p, 1, 2, 2, 64, 64, 128, 0, 0.1, 0, ws + 16, 1 << 20,
                              None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_host(p, p, p, p, p, 1, 2, 2, 64, 64, 128, 0, 0.1, 0, ws, 1000, None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_host(None, p, p, p, p, 1, 2, 2, 64, 64, 128, 0, 0.1, 0, ws, 1 << 20,
                              None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_host(p, p, p, p, p, 1, 2, 2, 64, 64, 96, 0, 0.1, 0, ws, 1 << 20,
                              None) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_fwd_host(p, p, p, p, p, 1, 3, 2, 64, 64, 128, 0, 0.1, 0, ws, 1 << 20,
                              None) == fa.FA_ERR_INVALID_ARG
    assert fa_lib.fa_fwd_host(None, None, None, None, None, 0, 2, 2, 64, 64, 128, 0, 0.1, 0, None, 0,
                              None) == fa.FA_OK
    assert fa_lib.fa_fwd_host_workspace_bytes(2, 4, 2, 100, 300, 128, ctypes.byref(nbytes)) == fa.FA_OK
    up = lambda x: (x + 255) // 256 * 256
    assert nbytes.value == 2 * up(2 * 4 * 100 * 128 * 2) + 2 * up(2 * 2 * 300 * 128 * 2) + up(2 * 4 * 100 * 4)
    # more query rows than the preprocessing grid can cover
    assert fa_lib.fa_bwd(p, p, p, p, p, p, p, p, p, 1, 1 << 10, 1 << 10, 1 << 25, 64, 128, 0, 0.1, 0, ws, 1 << 62,
                         None) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_bwd_workspace_bytes(2, 4, 100, 128, ctypes.byref(nbytes)) == fa.FA_OK
    assert nbytes.value == 2 * 4 * 100 * 128 * 4 + 2 * 4 * 2 * 512
    assert fa_lib.fa_bwd_workspace_bytes(2, 4, 100, 64, ctypes.byref(nbytes)) == fa.FA_OK
    assert nbytes.value == 2 * 4 * 100 * 64 * 4 + 2 * 4 * 2 * 512  # one 128-row step = two records
    assert fa_lib.fa_bwd_workspace_bytes(2, 4, 100, 96, ctypes.byref(nbytes)) == fa.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_bwd_workspace_bytes(-1, 4, 100, 128, ctypes.byref(nbytes)) == fa.FA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import exact_attention_forward_09_gb300 as fa
    monkeypatch.setattr(fa, "_LIB", None)
    monkeypatch.setattr(fa, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        fa.lib()


def test_ablation_library_exports_its_header():
    from exact_attention_forward_09_gb300 import build
    build.build()
    lib = ctypes.CDLL(build.LIB_ABLATE)
    text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "fa_ablate.h")).read(), flags=re.S)
    names = sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))
    assert names == ["fa_ablate_fwd"]
    for name in names:
        ctypes.cast(getattr(lib, name), ctypes.c_void_p)
