"""fa_fwd_host: attention on host buffers (copies to the device, kernel,
copies back, overlapped chunk by chunk on internal streams joined to the
caller's stream).  Results must equal fa_fwd_gqa on device copies of the
same inputs bit for bit (the same kernel runs on the same rows), for
page-locked and pageable host memory."""
import math

import pytest
import torch

import attn_inputs as gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_forward_09_gb300 as fa
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa.lib()
    return fa


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("B,Hq,Hkv,Nq,Nk,d,causal", [
    (2, 4, 4, 300, 300, 128, False),
    (2, 4, 4, 300, 300, 128, True),
    (1, 8, 2, 129, 700, 64, True),     # grouped queries, Nq != Nk
    (3, 2, 1, 1, 513, 256, False),     # decode-like row
    (1, 1, 1, 128, 128, 128, False),   # a single head: one chunk
    (4, 16, 16, 256, 256, 128, False), # more heads than chunks
])
def test_host_path_matches_device_path(fa, pinned, B, Hq, Hkv, Nq, Nk, d, causal):
    seed = 70 + Nq + Nk + d
    q = torch.from_numpy(gen.normal((B, Hq, Nq, d), seed, 0)).to(torch.bfloat16)
    k = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 1)).to(torch.bfloat16)
    v = torch.from_numpy(gen.normal((B, Hkv, Nk, d), seed, 2)).to(torch.bfloat16)
    if pinned:
        q, k, v = (t.pin_memory() for t in (q, k, v))
    o, lse = fa.fwd_host(q, k, v, causal=causal)
    torch.cuda.current_stream().synchronize()
    fa.check_device_error()
    o_ref, l_ref = fa.fwd_gqa(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    assert not o.is_cuda and not lse.is_cuda
    assert torch.equal(o, o_ref.cpu()), "O differs from the device path"
    assert torch.equal(lse, l_ref.cpu()), "LSE differs from the device path"


def test_host_path_is_ordered_on_the_stream(fa):
    """Work enqueued on the caller's stream after the call sees the results
    (the internal streams are joined back), and the call overlaps nothing
    enqueued before it."""
    B, H, N, d = 4, 8, 512, 128
    q, k, v = (torch.randn(B, H, N, d).to(torch.bfloat16).pin_memory() for _ in range(3))
    o = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty(fa.fwd_host_workspace_bytes(B, H, H, N, N, d), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            fa.fwd_host(q, k, v, out=o, lse=lse, workspace=ws)
        o_dev = torch.empty_like(q, device="cuda")
        o_dev.copy_(o, non_blocking=True)   # after the call on the same stream
    s.synchronize()
    o_ref, _ = fa.fwd(q.cuda(), k.cuda(), v.cuda())
    assert torch.equal(o_dev, o_ref)
