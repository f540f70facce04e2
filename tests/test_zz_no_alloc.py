"""attn_fwd_from_host_static: host inputs and outputs staged through the library's
fixed 64 MiB device array instead of caller-allocated device buffers.

The GPU tests compare it with attn_fwd_from_host (caller-owned staging buffers)
on two calls in a row that share the array; the argument and size checks run
before the device is touched, so they are tested on the CPU as well.  This file
is collected last so that the array is also exercised after every other test
has used the library.
"""
import ctypes

import numpy as np
import pytest

import tiled_attention_forward_fa2_gb300 as pkg
from tiled_attention_forward_fa2_gb300 import _binding
from tiled_attention_forward_fa2_gb300.inputs import normal_bf16_bits

torch = pytest.importorskip("torch")

STAGING_BYTES = 64 << 20
# O in bf16: two results of the same kernel on the same inputs; half a bf16 ulp
# at |o| <= 4 would already be 2^-7.  LSE in fp32.
O_ATOL, LSE_ATOL = 2.0 ** -8, 1e-5


def staged_bytes(B, H, Nq, Nk, D):
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    q, kv, lse = B * H * Nq * D * 2, B * H * Nk * D * 2, B * H * Nq * 4
    return r(q) + 2 * r(kv) + r(q) + lse


def static_call(lib, q, k, v, o, lse, B, H, Nq, Nk, D, causal=False, scale=0.125, stream=0):
    return lib.attn_fwd_from_host_static(q, k, v, o, lse, B, H, Nq, Nk, D, int(causal), ctypes.c_float(scale),
                                         ctypes.c_void_p(stream))


@pytest.fixture(scope="module")
def lib():
    return _binding.library()


# ---- argument and size checks: no device needed ----------------------------

def test_header_size_matches():
    assert staged_bytes(1, 15, 4096, 4096, 128) <= STAGING_BYTES < staged_bytes(1, 16, 4096, 4096, 128)


def test_rejects_more_than_the_staging_array(lib):
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.addressof(buf)
    # 16 heads of 4096 x 128: Q, K, V, O 16 MiB each, plus the LSE rows.
    assert static_call(lib, p, p, p, p, p, 1, 16, 4096, 4096, 128) == pkg.ATTN_ERR_UNSUPPORTED
    # a long key cache alone overflows it
    assert static_call(lib, p, p, p, p, p, 1, 1, 128, 1 << 20, 64) == pkg.ATTN_ERR_UNSUPPORTED
    # row counts past the array, whatever the head dimension
    assert static_call(lib, p, p, p, p, p, 1 << 30, 1 << 30, 1 << 30, 1, 8) in (pkg.ATTN_ERR_UNSUPPORTED,
                                                                              pkg.ATTN_ERR_INVALID_ARG)


def test_argument_rules(lib):
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.addressof(buf)
    assert static_call(lib, 0, 0, 0, 0, 0, 0, 4, 128, 128, 64) == pkg.ATTN_OK  # empty: nothing touched
    assert static_call(lib, 0, p, p, p, p, 1, 1, 128, 128, 64) == pkg.ATTN_ERR_INVALID_ARG
    assert static_call(lib, p, p, p, p, 0, 1, 1, 128, 128, 64) == pkg.ATTN_ERR_INVALID_ARG
    assert static_call(lib, p, p, p, p, p, -1, 1, 128, 128, 64) == pkg.ATTN_ERR_INVALID_ARG
    assert static_call(lib, p, p, p, p, p, 1, 1, 128, 128, 64, scale=0.0) == pkg.ATTN_ERR_INVALID_ARG
    assert static_call(lib, p, p, p, p, p, 1, 1, 128, 128, 60) == pkg.ATTN_ERR_UNSUPPORTED
    assert static_call(lib, p, p, p, p, p, 1, 1, 128, 128, 512) == pkg.ATTN_ERR_UNSUPPORTED


# ---- on the GPU --------------------------------------------------------------

def _host(a, pin=True):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory() if pin else t.clone()


def _problem(B, H, Nq, Nk, D, seed, pin=True):
    q = normal_bf16_bits(B * H * Nq * D, seed, 0).reshape(B, H, Nq, D)
    k = normal_bf16_bits(B * H * Nk * D, seed, 1).reshape(B, H, Nk, D)
    v = normal_bf16_bits(B * H * Nk * D, seed, 2).reshape(B, H, Nk, D)
    return _host(q, pin), _host(k, pin), _host(v, pin)


def _static(q, k, v, causal, scale, stream, pin=True):
    B, H, Nq, D = q.shape
    o = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, pin_memory=pin)
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, pin_memory=pin)
    st = pkg.attn_fwd_from_host_static(q, k, v, o, lse, B, H, Nq, k.shape[2], D, causal, scale, stream)
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    return o, lse


def _check(got, ref):
    (o, lse), (o_ref, lse_ref) = got, ref
    torch.testing.assert_close(o.float(), o_ref.float(), atol=O_ATOL, rtol=0)
    torch.testing.assert_close(lse, lse_ref, atol=LSE_ATOL, rtol=0)


@pytest.mark.gpu
@pytest.mark.parametrize("first,second", [
    ((2, 4, 500, 500, 128, True), (1, 3, 300, 700, 64, False)),     # ragged tails, two head dims
    ((1, 15, 4096, 4096, 128, False), (3, 2, 257, 257, 256, True)),  # the largest staged size, then D = 256
], ids=["ragged", "largest"])
def test_two_calls_in_a_row_match_caller_buffers(first, second):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    stream = torch.cuda.current_stream()
    a = _problem(*first[:5], seed=71)
    b = _problem(*second[:5], seed=72)
    assert staged_bytes(*first[:5]) <= STAGING_BYTES and staged_bytes(*second[:5]) <= STAGING_BYTES
    ref_a = pkg.fwd_from_host(*a, causal=first[5], scale=0.09)
    ref_b = pkg.fwd_from_host(*b, causal=second[5], scale=0.11)
    stream.synchronize()
    # Back to back on one stream, no synchronisation between: the second call's
    # uploads into the shared array are ordered after the first call's downloads.
    got_a = _static(*a, first[5], 0.09, stream)
    got_b = _static(*b, second[5], 0.11, stream)
    stream.synchronize()
    _check(got_a, ref_a)
    _check(got_b, ref_b)
    assert pkg.attn_last_status(stream) == pkg.ATTN_OK


@pytest.mark.gpu
def test_pageable_host_buffers_and_a_repeat():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    stream = torch.cuda.current_stream()
    a = _problem(1, 2, 384, 384, 64, seed=73, pin=False)
    ref = pkg.fwd_from_host(*a, causal=True, scale=0.125)
    stream.synchronize()
    for _ in range(2):
        got = _static(*a, True, 0.125, stream, pin=False)
        stream.synchronize()
        _check(got, ref)
