"""Failure detection on the GPU without faulting it.

Every pipeline wait in the kernel is bounded.  The test build of the library
(lib/libattn_fwd_gb300_testhooks.so, the same sources compiled with
-DATTN_TEST_HOOKS) has one extra entry point, attn_test_withhold_kv: with it on,
the forward issues no K/V loads, so the waits for them can never complete.
With the bound lowered to about a millisecond (attn_set_tuning) the kernel must
record ATTN_ERR_TIMEOUT for attn_last_status, drain its in-flight copies and
MMAs, free its tensor memory and return, leaving the device usable for the
next, normal call.  Nothing here traps, hangs or touches memory out of bounds.
The production library has no such hook (tests/test_abi_cpu.py checks that).
"""
import numpy as np
import pytest

import oracle
from parity import assert_close, o_to_f64, to_dev
from tiled_attention_forward_fa2_gb300 import _binding, build
from tiled_attention_forward_fa2_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

OK, TIMEOUT = 0, 4


@pytest.fixture(scope="module")
def tlib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    build.build()
    lib = _binding.load(build.LIB_TEST)
    yield lib
    lib.attn_test_withhold_kv(0)
    lib.attn_set_tuning(0, 0, 0, 0)


def sampled(B, H, N, n, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, B * H, n).astype(np.int64), rng.integers(0, N, n).astype(np.int64)


@pytest.mark.parametrize("D,grid", [(64, 2), (64, 1), (128, 2), (128, 1), (256, 1)])
@pytest.mark.parametrize("unit", [1, 2])
def test_wait_timeout_is_reported_and_device_stays_usable(tlib, unit, D, grid):
    """320 heads: on the persistent grid every CTA holds about four units when the wait runs out."""
    B, H, N = 1, 320, 512
    q, k, v = make_qkv(B, H, N, D, seed=90 + D)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    fwd = lambda: tlib.attn_fwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),  # noqa: E731
                                lse.data_ptr(), B, H, N, D, 1, 0.125, s)

    assert tlib.attn_set_tuning(unit, grid, 0, 2000000) == OK
    assert tlib.attn_test_withhold_kv(1) == OK
    try:
        assert fwd() == OK
        assert tlib.attn_last_status(s) == TIMEOUT
        assert tlib.attn_last_status(s) == OK  # reading the status clears it
    finally:
        tlib.attn_test_withhold_kv(0)
        tlib.attn_set_tuning(unit, grid, 0, 0)

    try:
        assert fwd() == OK
        assert tlib.attn_last_status(s) == OK
    finally:
        tlib.attn_set_tuning(0, 0, 0, 0)
    bh, ri = sampled(B, H, N, 2048, 91)
    o_ref, lse_ref = oracle.attn_rows(q, k, v, True, 0.125, bh, ri)
    of = o_to_f64(o).reshape(B * H, N, D)[bh, ri]
    lf = lse.cpu().numpy().astype(np.float64).reshape(B * H, N)[bh, ri]
    assert_close(of, lf, o_ref, lse_ref, f"after a timeout D={D} grid={grid} T={unit}")
