"""Failure detection on the GPU without faulting it.

Every pipeline wait in the kernel is bounded.  The test hook
ATTN_TEST_WITHHOLD_KV=1 makes the kernel issue no K/V loads, so the waits for
them can never complete; with the bound lowered to about a millisecond
(ATTN_WAIT_LIMIT_CYCLES) the kernel must record ATTN_ERR_TIMEOUT for
attn_last_status, drain its in-flight copies and MMAs, free its tensor memory
and return, leaving the device usable for the next, normal call.  Nothing here
traps, hangs or touches memory out of bounds.
"""
import numpy as np
import pytest

import oracle
import tiled_attention_forward_fa2_gb300 as pkg
from parity import assert_close, o_to_f64, to_dev
from tiled_attention_forward_fa2_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkg.library()


@pytest.mark.parametrize("tiles", ["1", "2"])
def test_wait_timeout_is_reported_and_device_stays_usable(tiles, monkeypatch):
    monkeypatch.setenv("ATTN_TILES_PER_CTA", tiles)
    B, H, N, D = 1, 4, 512, 64
    q, k, v = make_qkv(B, H, N, D, seed=90)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), device="cuda")
    s = torch.cuda.current_stream()

    monkeypatch.setenv("ATTN_WAIT_LIMIT_CYCLES", "2000000")
    monkeypatch.setenv("ATTN_TEST_WITHHOLD_KV", "1")
    assert pkg.attn_fwd(qd, kd, vd, o, lse, B, H, N, D, True, 0.125, s) == pkg.ATTN_OK
    assert pkg.attn_last_status(s) == pkg.ATTN_ERR_TIMEOUT
    assert pkg.attn_last_status(s) == pkg.ATTN_OK  # reading the status clears it

    monkeypatch.delenv("ATTN_WAIT_LIMIT_CYCLES")
    monkeypatch.delenv("ATTN_TEST_WITHHOLD_KV")
    assert pkg.attn_fwd(qd, kd, vd, o, lse, B, H, N, D, True, 0.125, s) == pkg.ATTN_OK
    assert pkg.attn_last_status(s) == pkg.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 0.125)
    assert_close(o_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "after a timeout")
