"""The C-ABI library loads and validates arguments without a GPU (no compute calls)."""
import ctypes
import glob
import os
import re

import pytest

import tiled_attention_forward_fa2_gb300 as pkg
from tiled_attention_forward_fa2_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
A16 = 0x10000  # fake, 16-byte aligned addresses: every call below returns before touching them
MB = 1 << 20


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return pkg.library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"attn_fwd", "attn_last_status", "attn_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def call(q=A16, k=A16 + 64 * MB, v=A16 + 128 * MB, o=A16 + 192 * MB, lse=A16 + 256 * MB,
         B=1, H=2, N=256, D=64, causal=0, scale=0.125):
    return pkg.attn_fwd(q, k, v, o, lse, B, H, N, D, causal, scale, None)


def test_null_pointers(lib):
    for kw in ("q", "k", "v", "o", "lse"):
        assert call(**{kw: None}) == pkg.ATTN_ERR_INVALID_ARG


def test_bad_sizes_and_scale(lib):
    assert call(B=-1) == pkg.ATTN_ERR_INVALID_ARG
    assert call(N=-5) == pkg.ATTN_ERR_INVALID_ARG
    assert call(D=0) == pkg.ATTN_ERR_INVALID_ARG
    for s in (0.0, -0.125, float("inf"), float("nan")):
        assert call(scale=s) == pkg.ATTN_ERR_INVALID_ARG
    assert call(N=2**31) == pkg.ATTN_ERR_INVALID_ARG
    assert call(B=2**20, H=2**20) == pkg.ATTN_ERR_INVALID_ARG


def test_unit_count_stays_in_int32(lib):
    """B*H*query tiles near 2^31 would overflow the persistent grid's int32 unit
    index (up to two grid sizes past the last unit): rejected up front.  The
    buffers are placed 2^40 bytes apart so only the size check can object."""
    T = 1 << 40
    big = dict(q=A16, k=A16 + T, v=A16 + 2 * T, o=A16 + 3 * T, lse=A16 + 4 * T)
    assert call(B=1, H=2**31 - 1, N=1, D=8, **big) == pkg.ATTN_ERR_INVALID_ARG
    assert call(B=1, H=2**31 - 4096, N=1, D=8, **big) == pkg.ATTN_ERR_INVALID_ARG
    assert call(B=2**15, H=2**15 - 1, N=129, D=8, **big) == pkg.ATTN_ERR_INVALID_ARG  # 2 tiles each


def test_tuning_overrides_validate(lib):
    assert pkg.attn_set_tuning(5, 0, 0, 0) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_set_tuning(4, 0, 0, 0) == pkg.ATTN_OK
    assert pkg.attn_set_tuning(-1, 0, 0, 0) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_set_tuning(3, 0, 0, 0) == pkg.ATTN_OK
    assert pkg.attn_set_tuning(0, 3, 0, 0) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_set_tuning(0, 0, 33, 0) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_set_tuning(0, 0, 0, -1) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_set_tuning(2, 1, 4, 1000) == pkg.ATTN_OK
    assert pkg.attn_set_tuning() == pkg.ATTN_OK


def test_test_hook_only_in_the_test_build(lib):
    """The production library cannot drop its K/V loads; only the test build
    (compiled with -DATTN_TEST_HOOKS) exports the hook that does."""
    from tiled_attention_forward_fa2_gb300 import _binding
    assert not hasattr(lib, "attn_test_withhold_kv")
    tl = _binding.load(cuda_build.LIB_TEST)
    assert hasattr(tl, "attn_test_withhold_kv")
    for n in declared_functions():
        assert hasattr(tl, n)
    src = open(os.path.join(ROOT, "tiled_attention_forward_fa2_gb300", "csrc", "attn_fwd.cu")).read()
    assert "getenv" not in src


def test_unsupported_head_dims(lib):
    for d in (4, 12, 100, 260, 264, 512):
        assert call(D=d) == pkg.ATTN_ERR_UNSUPPORTED


def call_bwd(D=64, **kw):
    a = dict(q=A16, k=A16 + 64 * MB, v=A16 + 128 * MB, o=A16 + 192 * MB, lse=A16 + 256 * MB, dout=A16 + 320 * MB,
             dq=A16 + 384 * MB, dk=A16 + 448 * MB, dv=A16 + 512 * MB, delta=A16 + 576 * MB)
    a.update(kw)
    return pkg.attn_bwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["dout"], a["dq"], a["dk"], a["dv"], a["delta"],
                        1, 2, 256, D, 0, 0.125, None)


def test_backward_head_dims(lib):
    """The backward takes contiguous head dims that are multiples of 8 up to 256, like the forward."""
    import torch
    for d in (4, 100, 260, 264, 512):
        assert call_bwd(D=d) == pkg.ATTN_ERR_UNSUPPORTED
    if not torch.cuda.is_available():
        for d in (8, 136, 192, 256):
            assert call_bwd(D=d) == pkg.ATTN_ERR_CUDA  # past validation, no device
    assert call_bwd(D=64, dq=None) == pkg.ATTN_ERR_INVALID_ARG


def test_padded_head_dims_pass_validation(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for d in (8, 32, 48, 96, 112, 136, 192, 200, 256):
        assert call(D=d) == pkg.ATTN_ERR_CUDA  # past validation, stopped only by the missing device


def test_empty_problem_is_a_no_op(lib):
    for kw in ({"B": 0}, {"H": 0}, {"N": 0}):
        assert call(**kw) == pkg.ATTN_OK
        assert call(q=None, k=None, v=None, o=None, lse=None, **kw) == pkg.ATTN_OK
    assert call(B=0, D=100) == pkg.ATTN_ERR_UNSUPPORTED
    assert call(B=0, scale=-1.0) == pkg.ATTN_ERR_INVALID_ARG


def test_misaligned_pointers(lib):
    assert call(q=A16 + 8) == pkg.ATTN_ERR_INVALID_ARG
    assert call(o=A16 + 192 * MB + 2) == pkg.ATTN_ERR_INVALID_ARG
    assert call(lse=A16 + 256 * MB + 2) == pkg.ATTN_ERR_INVALID_ARG


def test_overlapping_outputs(lib):
    assert call(o=A16) == pkg.ATTN_ERR_INVALID_ARG               # o over q
    assert call(o=A16 + 64 * MB + 4096) == pkg.ATTN_ERR_INVALID_ARG  # o inside k
    assert call(lse=A16 + 128 * MB + 16) == pkg.ATTN_ERR_INVALID_ARG  # lse inside v
    assert call(lse=A16 + 192 * MB + 64) == pkg.ATTN_ERR_INVALID_ARG  # lse inside o


def test_status_strings_and_flops(lib):
    assert pkg.attn_status_string(pkg.ATTN_ERR_TIMEOUT) == "ATTN_ERR_TIMEOUT"
    assert pkg.attn_status_string(99) == "ATTN_ERR_UNKNOWN"
    assert pkg.attn_fwd_flops(4, 16, 4096, 128, False) == 4.0 * 4 * 16 * 4096 ** 2 * 128
    assert pkg.attn_fwd_flops(1, 16, 16384, 128, True) == 2.0 * 16 * 16384 ** 2 * 128


def test_no_gpu_means_cuda_error_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call() == pkg.ATTN_ERR_CUDA


def call_qk(Nq=100, Nk=300, causal=1, **kw):
    args = dict(q=A16, k=A16 + 64 * MB, v=A16 + 128 * MB, o=A16 + 192 * MB, lse=A16 + 256 * MB,
                B=1, H=2, D=64, scale=0.125)
    args.update(kw)
    return pkg.attn_fwd_qk(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["H"], Nq, Nk,
                           args["D"], causal, args["scale"], None)


def test_qk_rows_without_keys_are_unsupported(lib):
    assert call_qk(Nq=300, Nk=100, causal=1) == pkg.ATTN_ERR_UNSUPPORTED  # first 200 queries see nothing
    assert call_qk(Nq=10, Nk=0, causal=0) == pkg.ATTN_ERR_UNSUPPORTED
    assert call_qk(Nq=0, Nk=50) == pkg.ATTN_OK
    assert call_qk(Nq=0, Nk=50, q=None, k=None, v=None, o=None, lse=None) == pkg.ATTN_OK
    assert call_qk(Nq=-1, Nk=50) == pkg.ATTN_ERR_INVALID_ARG


def test_qk_overlap_uses_each_tensors_own_length(lib):
    # k holds Nk = 300 rows: an o placed right after a 100-row q but inside k overlaps.
    assert call_qk(Nq=100, Nk=300, o=A16 + 64 * MB + 100 * 64 * 2 * 2) == pkg.ATTN_ERR_INVALID_ARG
    assert call_qk(Nq=100, Nk=300, lse=A16 + 128 * MB + 16) == pkg.ATTN_ERR_INVALID_ARG


def test_qk_flops(lib):
    assert pkg.attn_fwd_qk_flops(2, 3, 256, 256, 64, True) == pkg.attn_fwd_flops(2, 3, 256, 64, True)
    assert pkg.attn_fwd_qk_flops(2, 3, 256, 256, 64, False) == pkg.attn_fwd_flops(2, 3, 256, 64, False)
    assert pkg.attn_fwd_qk_flops(1, 1, 100, 300, 64, False) == 4.0 * 100 * 300 * 64
    assert pkg.attn_fwd_qk_flops(1, 1, 100, 300, 64, True) == 4.0 * (100 * 200 + 0.5 * 100 * 100) * 64


def call_host(Nq=100, Nk=300, causal=0, **kw):
    args = dict(qh=A16 + 512 * MB, kh=A16 + 576 * MB, vh=A16 + 640 * MB, oh=A16 + 704 * MB, lh=A16 + 768 * MB,
                q=A16, k=A16 + 64 * MB, v=A16 + 128 * MB, o=A16 + 192 * MB, lse=A16 + 256 * MB,
                B=1, H=2, D=64, scale=0.125)
    args.update(kw)
    a = args
    return pkg.attn_fwd_from_host(a["qh"], a["kh"], a["vh"], a["oh"], a["lh"], a["q"], a["k"], a["v"], a["o"],
                                  a["lse"], a["B"], a["H"], Nq, Nk, a["D"], causal, a["scale"], None)


def test_from_host_validation(lib):
    for kw in ("qh", "kh", "vh", "oh", "lh", "q", "k", "v", "o", "lse"):
        assert call_host(**{kw: None}) == pkg.ATTN_ERR_INVALID_ARG, kw
    assert call_host(scale=0.0) == pkg.ATTN_ERR_INVALID_ARG
    assert call_host(D=100) == pkg.ATTN_ERR_UNSUPPORTED
    assert call_host(Nq=300, Nk=100, causal=1) == pkg.ATTN_ERR_UNSUPPORTED
    assert call_host(o=A16 + 64 * MB) == pkg.ATTN_ERR_INVALID_ARG  # device o overlaps device k
    assert call_host(Nq=0, qh=None, kh=None, vh=None, oh=None, lh=None, q=None, k=None, v=None, o=None,
                     lse=None) == pkg.ATTN_OK
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call_host() == pkg.ATTN_ERR_CUDA  # valid request, no device: nothing enqueued


def call_based(N=256, F=16, D=64, **kw):
    a = dict(q=A16, k=A16 + 64 * MB, v=A16 + 128 * MB, y=A16 + 192 * MB, z=A16 + 256 * MB, B=1, H=2, scale=0.25)
    a.update(kw)
    return pkg.attn_based_fwd(a["q"], a["k"], a["v"], a["y"], a["z"], a["B"], a["H"], N, F, D, a["scale"], None)


def test_based_validation(lib):
    for kw in ("q", "k", "v", "y", "z"):
        assert call_based(**{kw: None}) == pkg.ATTN_ERR_INVALID_ARG, kw
    for F in (4, 12, 24, 32):
        assert call_based(F=F) == pkg.ATTN_ERR_UNSUPPORTED
    for D in (4, 100, 128):
        assert call_based(D=D) == pkg.ATTN_ERR_UNSUPPORTED
    assert call_based(scale=0.0) == pkg.ATTN_ERR_INVALID_ARG
    assert call_based(scale=float("nan")) == pkg.ATTN_ERR_INVALID_ARG
    assert call_based(N=-1) == pkg.ATTN_ERR_INVALID_ARG
    assert call_based(N=0, q=None, k=None, v=None, y=None, z=None) == pkg.ATTN_OK
    assert call_based(y=A16) == pkg.ATTN_ERR_INVALID_ARG                 # y over q
    assert call_based(z=A16 + 192 * MB + 64) == pkg.ATTN_ERR_INVALID_ARG  # z inside y
    assert call_based(q=A16 + 4) == pkg.ATTN_ERR_INVALID_ARG
    assert call_based(z=A16 + 256 * MB + 2) == pkg.ATTN_ERR_INVALID_ARG


def test_based_flops(lib):
    # 1 + 16 + 136 = 153 features, 65 value columns, state update and readout.
    assert pkg.attn_based_fwd_flops(2, 3, 100, 16, 64) == 4.0 * 153 * 65 * 600


def test_based_no_gpu_means_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call_based() == pkg.ATTN_ERR_CUDA
    assert call_based(F=8, D=8) == pkg.ATTN_ERR_CUDA


def call_ld(D=100, ld=104, **kw):
    a = dict(q=A16, k=A16 + 64 * MB, v=A16 + 128 * MB, o=A16 + 192 * MB, lse=A16 + 256 * MB, B=1, H=2, Nq=256, Nk=256)
    a.update(kw)
    return pkg.attn_fwd_ld(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"], D, ld, 0, 0.125,
                           None)


def test_padded_rows_validation(lib):
    """attn_fwd_ld / attn_bwd_ld: any head dim with rows padded to a multiple of 8 elements."""
    import torch
    gpu = torch.cuda.is_available()
    for D, ld in ((4, 8), (12, 16), (100, 104), (100, 200), (255, 256), (1, 8), (96, 96)):
        if not gpu:
            assert call_ld(D=D, ld=ld) == pkg.ATTN_ERR_CUDA, (D, ld)  # past validation, no device
    # ld must be a multiple of 8 and hold roundup8(D) columns
    for D, ld in ((100, 100), (100, 96), (12, 12), (8, 4), (64, 0), (64, -8), (97, 100), (97, 96)):
        assert call_ld(D=D, ld=ld) == pkg.ATTN_ERR_INVALID_ARG, (D, ld)
    assert call_ld(D=260, ld=264) == pkg.ATTN_ERR_UNSUPPORTED
    # o inside k when k is measured with its padded rows (2*256*104*2 bytes)
    assert call_ld(o=A16 + 64 * MB + 2 * 256 * 100 * 2) == pkg.ATTN_ERR_INVALID_ARG
    b = dict(q=A16, k=A16 + 64 * MB, v=A16 + 128 * MB, o=A16 + 192 * MB, lse=A16 + 256 * MB, do=A16 + 320 * MB,
             dq=A16 + 384 * MB, dk=A16 + 448 * MB, dv=A16 + 512 * MB, dl=A16 + 576 * MB)
    bwd = lambda D, ld: pkg.attn_bwd_ld(b["q"], b["k"], b["v"], b["o"], b["lse"], b["do"], b["dq"], b["dk"],  # noqa: E731
                                        b["dv"], b["dl"], 1, 2, 256, 256, D, ld, 0, 0.125, None)
    assert bwd(100, 100) == pkg.ATTN_ERR_INVALID_ARG
    assert bwd(260, 264) == pkg.ATTN_ERR_UNSUPPORTED
    if not gpu:
        assert bwd(100, 104) == pkg.ATTN_ERR_CUDA
        assert bwd(4, 8) == pkg.ATTN_ERR_CUDA
        assert bwd(250, 256) == pkg.ATTN_ERR_CUDA


def test_kernel_name_rejects_what_the_forward_rejects(lib):
    import torch
    for args in ((0, 1, 128, 128, 64, 0), (1, 1, 128, 128, 264, 1), (1, 1, -5, 128, 64, 0), (1, 1, 128, 0, 64, 0)):
        assert pkg.attn_fwd_kernel_name(*args) is None, args
    if not torch.cuda.is_available():
        assert pkg.attn_fwd_kernel_name(1, 1, 128, 128, 64, 0) is None  # no device to plan for
