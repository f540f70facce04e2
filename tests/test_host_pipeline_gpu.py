"""attn_fwd_from_host: host inputs and outputs, copies overlapped with the kernels.

The chunked, multi-stream call must give exactly the device call's results (each
row is computed by the same kernel code whatever the grid), wait for work already
on the caller's stream, and finish everything -- host outputs included -- once
that stream is synchronised.
"""
import numpy as np
import pytest

import tiled_attention_forward_fa2_gb300 as pkg
from parity import to_dev
from tiled_attention_forward_fa2_gb300.inputs import make_qkv, normal_bf16_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkg.library()


def host(a, pin):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


def device_reference(q, k, v, causal, scale):
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    B, H, Nq, D = q.shape
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    st = pkg.attn_fwd_qk(qd, kd, vd, o, lse, B, H, Nq, k.shape[2], D, causal, scale, torch.cuda.current_stream())
    assert st == pkg.ATTN_OK
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def qkv_qk(B, H, Nq, Nk, D, seed):
    q = normal_bf16_bits(B * H * Nq * D, seed, 0).reshape(B, H, Nq, D)
    k = normal_bf16_bits(B * H * Nk * D, seed, 1).reshape(B, H, Nk, D)
    v = normal_bf16_bits(B * H * Nk * D, seed, 2).reshape(B, H, Nk, D)
    return q, k, v


@pytest.mark.parametrize("pin", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("B,H,Nq,Nk,D,causal", [
    (1, 1, 256, 256, 64, False),     # one chunk
    (1, 3, 333, 333, 128, True),     # fewer heads than chunks, ragged
    (2, 10, 640, 640, 64, False),    # 20 heads in 8 chunks of 2 or 3
    (3, 7, 200, 1000, 128, True),    # queries against a longer key cache
    (2, 5, 300, 300, 256, True),     # the D = 256 kernel
])
def test_matches_device_call_exactly(B, H, Nq, Nk, D, causal, pin):
    q, k, v = qkv_qk(B, H, Nq, Nk, D, seed=31 + B * H + Nq)
    scale = 1.0 / np.sqrt(D)
    o_ref, lse_ref = device_reference(q, k, v, causal, scale)
    qh, kh, vh = host(q, pin), host(k, pin), host(v, pin)
    o, lse = pkg.fwd_from_host(qh, kh, vh, causal=causal, scale=scale)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse, lse_ref)


def test_back_to_back_calls_share_device_buffers():
    """The second call's uploads wait for the first call's kernels on the shared buffers."""
    B, H, N, D = 2, 16, 1024, 128
    a = make_qkv(B, H, N, D, seed=5)
    b = make_qkv(B, H, N, D, seed=6)
    ref_a = device_reference(*a, False, 0.1)
    ref_b = device_reference(*b, False, 0.1)
    dev = torch.device("cuda")
    bufs = (torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev),
            torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev),
            torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev),
            torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev),
            torch.empty((B, H, N), dtype=torch.float32, device=dev))
    outs, keep = [], []
    for q, k, v in (a, b, a):
        # The host inputs must outlive the asynchronous copies: torch's pinned-memory
        # cache would otherwise hand their blocks to the next call's inputs.
        keep.append((host(q, True), host(k, True), host(v, True)))
        outs.append(pkg.fwd_from_host(*keep[-1], scale=0.1, device_buffers=bufs))
    torch.cuda.current_stream().synchronize()
    for (o, lse), (o_ref, lse_ref) in zip(outs, (ref_a, ref_b, ref_a)):
        assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
        assert torch.equal(lse, lse_ref)


def test_side_stream():
    """The call runs on a non-default stream; synchronising that stream completes it."""
    B, H, N, D = 1, 8, 512, 64
    q, k, v = make_qkv(B, H, N, D, seed=9)
    o_ref, lse_ref = device_reference(q, k, v, True, 0.125)
    s = torch.cuda.Stream()
    inputs = (host(q, True), host(k, True), host(v, True))
    with torch.cuda.stream(s):
        o, lse = pkg.fwd_from_host(*inputs, causal=True, scale=0.125, stream=s)
    s.synchronize()
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse, lse_ref)
    assert pkg.attn_last_status(s) == pkg.ATTN_OK
