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


def sampled(B, H, N, n, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, B * H, n).astype(np.int64), rng.integers(0, N, n).astype(np.int64)


@pytest.mark.parametrize("D,persist", [(64, "1"), (64, "0"), (128, "1"), (128, "0"), (256, "0")])
@pytest.mark.parametrize("tiles", ["1", "2"])
def test_wait_timeout_is_reported_and_device_stays_usable(tiles, D, persist, monkeypatch):
    """320 heads: on the persistent grid every CTA holds about four units when the wait runs out."""
    monkeypatch.setenv("ATTN_TILES_PER_CTA", tiles)
    monkeypatch.setenv("ATTN_PERSISTENT", persist)
    B, H, N = 1, 320, 512
    q, k, v = make_qkv(B, H, N, D, seed=90 + D)
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
    bh, ri = sampled(B, H, N, 2048, 91)
    o_ref, lse_ref = oracle.attn_rows(q, k, v, True, 0.125, bh, ri)
    of = o_to_f64(o).reshape(B * H, N, D)[bh, ri]
    lf = lse.cpu().numpy().astype(np.float64).reshape(B * H, N)[bh, ri]
    assert_close(of, lf, o_ref, lse_ref, f"after a timeout D={D} persistent={persist} T={tiles}")
