"""Backward kernels against the fp64 backward oracle, through the C ABI.

Tolerance (per output X in dQ, dK, dV, and D): with u = 2^-9 the bf16 rounding
bound, max|X - X_ref| <= 8u * max|X_ref| and mean|X - X_ref| <= 3u * mean|X_ref|.
The outputs are rounded to bf16 once (<= u each), and P, dS and the forward's
O (which D is computed from) enter the products in bf16; measured errors sit
near 2.5u (max) and 1.2u (mean).  The normalisers are floored at 1e-2 for
references that are exactly zero (N = 1: one key gives P = 1 and dS = 0).
"""
import math

import numpy as np
import pytest

import oracle
import tiled_attention_forward_fa2_gb300 as pkg
from parity import to_dev
from tiled_attention_forward_fa2_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

U = 2.0 ** -9
MAX_REL, MEAN_REL = 8 * U, 3 * U


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkg.library()


def grads(B, H, Nq, Nk, D, causal, seed, q_std=1.0):
    q, _, _ = make_qkv(B, H, Nq, D, seed=seed, q_std=q_std)
    _, k, v = make_qkv(B, H, Nk, D, seed=seed + 1)
    do, _, _ = make_qkv(B, H, Nq, D, seed=seed + 2)
    scale = 1.0 / math.sqrt(D)
    qd, kd, vd, dod = to_dev(q), to_dev(k), to_dev(v), to_dev(do)
    o, lse = pkg.fwd(qd, kd, vd, causal=causal, scale=scale)
    s = torch.cuda.current_stream()
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    delta = torch.full((B, H, Nq), float("nan"), device="cuda")
    st = pkg.attn_bwd_qk(qd, kd, vd, o, lse, dod, dq, dk, dv, delta, B, H, Nq, Nk, D, causal, scale, s)
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    assert pkg.attn_last_status(s) == pkg.ATTN_OK
    got = {n: t.float().cpu().numpy().astype(np.float64) for n, t in (("dq", dq), ("dk", dk), ("dv", dv), ("delta", delta))}
    return got, oracle.attn_bwd(q, k, v, do, causal, scale)


def assert_grads_close(got, ref, what):
    for n in ("dq", "dk", "dv", "delta"):
        g, r = got[n], ref[n]
        assert np.all(np.isfinite(g)), f"{what}: {n} has unwritten or non-finite entries"
        err = np.abs(g - r)
        # Normalisers floored at 1e-2 (these problems' gradients are O(0.1-1)): with a
        # single key the references dQ, dK are exactly 0 and the GPU's are rounding noise.
        mx = err.max() / max(np.abs(r).max(), 1e-2)
        mean = err.mean() / max(np.abs(r).mean(), 1e-2)
        assert mx <= MAX_REL and mean <= MEAN_REL, f"{what}: {n} max/max={mx:.2e} mean/mean={mean:.2e}"


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 128, 200, 640])
def test_backward_square(N, D, causal):
    got, ref = grads(2, 3, N, N, D, causal, seed=1200 + N + D)
    assert_grads_close(got, ref, f"N={N} D={D} causal={causal}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Nq,Nk,causal", [(1, 500, True), (130, 700, True), (700, 300, False), (64, 1024, False)])
def test_backward_queries_and_keys_of_different_lengths(Nq, Nk, causal, D):
    got, ref = grads(1, 2, Nq, Nk, D, causal, seed=1300 + Nq + Nk)
    assert_grads_close(got, ref, f"Nq={Nq} Nk={Nk} D={D} causal={causal}")


def test_backward_large_logits():
    got, ref = grads(1, 2, 1024, 1024, 128, True, seed=1400, q_std=4.0)
    assert_grads_close(got, ref, "q_std=4 N=1024 causal")


def test_backward_workload_b2h8n1024d64():
    for causal in (False, True):
        got, ref = grads(2, 8, 1024, 1024, 64, causal, seed=1002)
        assert_grads_close(got, ref, f"B2 H8 N1024 D64 causal={causal}")


def test_backward_deterministic():
    a, _ = grads(1, 4, 512, 512, 128, True, seed=1500)
    b, _ = grads(1, 4, 512, 512, 128, True, seed=1500)
    for n in a:
        assert np.array_equal(a[n], b[n])


def test_backward_argument_errors():
    x = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
    f = torch.zeros((1, 1, 256), device="cuda")
    s = torch.cuda.current_stream()
    outs = [torch.empty_like(x) for _ in range(3)]
    assert pkg.attn_bwd(x, x, x, x, f, x, *outs, f, 1, 1, 256, 64, False, 0.125, s) == pkg.ATTN_ERR_INVALID_ARG  # delta over lse
    assert pkg.attn_bwd(x, x, x, x, f, x, x, outs[1], outs[2], torch.empty_like(f), 1, 1, 256, 64, False, 0.125, s) \
        == pkg.ATTN_ERR_INVALID_ARG  # dq over q
    assert pkg.attn_bwd_qk(x, x, x, x, f, x, *outs, torch.empty_like(f), 1, 1, 256, 128, 64, True, 0.125, s) \
        == pkg.ATTN_ERR_UNSUPPORTED  # causal with more queries than keys
    assert pkg.attn_last_status(s) == pkg.ATTN_OK


@pytest.mark.parametrize("D", [8, 32, 96, 112])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_padded_head_dims(D, causal):
    got, ref = grads(1, 3, 300, 300, D, causal, seed=1700 + D)
    assert_grads_close(got, ref, f"D={D} causal={causal}")


@pytest.mark.parametrize("D", [136, 192, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 33, 200, 640])
def test_backward_head_dims_above_128(N, D, causal):
    """The D = 256 kernels (64-key steps for dQ; dK and dV in two 128-column halves over
    32-query stages), with D = 136 and 192 zero-padded to 256: several key tiles, ragged tails."""
    got, ref = grads(2, 2, N, N, D, causal, seed=1900 + N + D)
    assert_grads_close(got, ref, f"N={N} D={D} causal={causal}")


@pytest.mark.parametrize("D", [256, 200])
@pytest.mark.parametrize("Nq,Nk,causal", [(1, 500, True), (130, 700, True), (700, 300, False)])
def test_backward_head_dims_above_128_different_lengths(Nq, Nk, causal, D):
    got, ref = grads(1, 2, Nq, Nk, D, causal, seed=1950 + Nq + Nk)
    assert_grads_close(got, ref, f"Nq={Nq} Nk={Nk} D={D} causal={causal}")


def test_backward_d256_large_logits():
    got, ref = grads(1, 2, 512, 512, 256, True, seed=1990, q_std=4.0)
    assert_grads_close(got, ref, "q_std=4 N=512 D=256 causal")


def sample_idx(n_bh, n, n_random, seed):
    """Random (head, index) pairs plus the first and last 64 indices of the first and last head."""
    rng = np.random.default_rng(seed)
    bh = [rng.integers(0, n_bh, n_random)]
    ix = [rng.integers(0, n, n_random)]
    for h in (0, n_bh - 1):
        for i0 in (0, max(0, n - 64)):
            m = min(64, n)
            bh.append(np.full(m, h))
            ix.append(np.arange(i0, i0 + m))
    return np.concatenate(bh).astype(np.int64), np.concatenate(ix).astype(np.int64)


def assert_sample_close(g, r, what):
    assert np.all(np.isfinite(g)), f"{what}: unwritten or non-finite entries"
    err = np.abs(g - r)
    mx = err.max() / max(np.abs(r).max(), 1e-2)
    mean = err.mean() / max(np.abs(r).mean(), 1e-2)
    assert mx <= MAX_REL and mean <= MEAN_REL, f"{what}: max/max={mx:.2e} mean/mean={mean:.2e}"


@pytest.mark.parametrize("name,key_heads", [("b4h16n4096d128", 2), ("b1h16n16384d128_causal_q4", 1),
                                            ("b8h16nq512nk8192d128_causal", 2)])
def test_backward_full_size_sampled(name, key_heads):
    """The bench's backward workloads at full size, in its launch configuration: dQ and D of sampled
    query rows, dK and dV of sampled keys of the last head (and the first: one head's softmax
    statistics cost the oracle O(Nq Nk D), so N = 16384 checks one head)."""
    from tiled_attention_forward_fa2_gb300.inputs import WORKLOADS, normal_bf16_bits
    w = WORKLOADS[name]
    q, k, v = w.qkv()
    do = normal_bf16_bits(q.size, w.seed + 7, 3).reshape(q.shape)  # seeded upstream gradient
    B, H, Nq, D, Nk = w.B, w.H, w.N, w.D, w.n_keys
    qd, kd, vd, dod = to_dev(q), to_dev(k), to_dev(v), to_dev(do)
    o, lse = pkg.fwd(qd, kd, vd, causal=w.causal, scale=w.scale)
    s = torch.cuda.current_stream()
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    delta = torch.empty((B, H, Nq), device="cuda")
    st = pkg.attn_bwd_qk(qd, kd, vd, o, lse, dod, dq, dk, dv, delta, B, H, Nq, Nk, D, w.causal, w.scale, s)
    assert st == pkg.ATTN_OK and pkg.attn_last_status(s) == pkg.ATTN_OK
    bh, ri = sample_idx(B * H, Nq, 256, w.seed)
    dq_ref, delta_ref = oracle.attn_bwd_rows(q, k, v, do, w.causal, w.scale, bh, ri)
    g = dq.float().cpu().numpy().astype(np.float64).reshape(B * H, Nq, D)
    assert_sample_close(g[bh, ri], dq_ref, f"{name} dQ rows")
    assert_sample_close(delta.cpu().numpy().astype(np.float64).reshape(B * H, Nq)[bh, ri], delta_ref, f"{name} D")
    gk = dk.float().cpu().numpy().astype(np.float64).reshape(B * H, Nk, D)
    gv = dv.float().cpu().numpy().astype(np.float64).reshape(B * H, Nk, D)
    rng = np.random.default_rng(w.seed + 1)
    for h in (B * H - 1, 0)[:key_heads]:
        kj = np.concatenate([rng.integers(0, Nk, 96), np.arange(64), np.arange(Nk - 64, Nk)]).astype(np.int64)
        dk_ref, dv_ref = oracle.attn_bwd_keys(q, k, v, do, w.causal, w.scale, h, kj)
        assert_sample_close(gk[h, kj], dk_ref, f"{name} dK of head {h}")
        assert_sample_close(gv[h, kj], dv_ref, f"{name} dV of head {h}")


@pytest.mark.parametrize("D,ld", [(4, 8), (12, 24), (100, 104), (73, 80), (250, 256), (129, 144)])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_padded_rows_any_head_dim(D, ld, causal):
    """attn_bwd_ld: rows ld elements apart, head dims that are not multiples of 8; zeros up to
    roundup8(D) and NaN beyond in the inputs (never read), a sentinel beyond roundup8(D) in the
    gradient outputs (never written)."""
    B, H, N = 1, 2, 300
    q, k, v = make_qkv(B, H, N, D, seed=1800 + D)
    do = make_qkv(B, H, N, D, seed=1801 + D)[0]
    scale = 1.0 / math.sqrt(D)
    d8 = (D + 7) // 8 * 8

    def pad(bits, fill):
        buf = np.full((B, H, N, ld), fill, dtype=np.uint16)
        buf[..., :d8] = 0
        buf[..., :D] = bits
        return to_dev(buf)

    nan, sentinel = 0x7FC0, 0x4049
    qd, kd, vd, dod = pad(q, nan), pad(k, nan), pad(v, nan), pad(do, nan)
    o = pad(np.zeros_like(q), nan)
    lse = torch.empty((B, H, N), device="cuda")
    s = torch.cuda.current_stream()
    assert pkg.attn_fwd_ld(qd, kd, vd, o, lse, B, H, N, N, D, ld, causal, scale, s) == pkg.ATTN_OK
    dq, dk, dv = (pad(np.zeros_like(q), sentinel) for _ in range(3))
    delta = torch.full((B, H, N), float("nan"), device="cuda")
    st = pkg.attn_bwd_ld(qd, kd, vd, o, lse, dod, dq, dk, dv, delta, B, H, N, N, D, ld, causal, scale, s)
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    assert pkg.attn_last_status(s) == pkg.ATTN_OK
    got = {}
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        bits = t.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.all(bits[..., d8:] == sentinel), f"columns past roundup8(D) of {n} were written"
        assert np.all(bits[..., D:d8] == 0), f"columns D..roundup8(D)-1 of {n} are not zero"
        got[n] = t[..., :D].float().cpu().numpy().astype(np.float64)
    got["delta"] = delta.cpu().numpy().astype(np.float64)
    assert_grads_close(got, oracle.attn_bwd(q, k, v, do, causal, scale), f"D={D} ld={ld} causal={causal}")
