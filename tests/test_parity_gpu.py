"""CUDA path against the CPU oracle, element by element, through the C ABI."""
import math

import numpy as np
import pytest

import oracle
import tiled_attention_forward_fa2_gb300 as pkg
from parity import assert_close, o_to_f64, parity_report, to_dev, tune
from tiled_attention_forward_fa2_gb300.inputs import WORKLOADS, f64_to_bf16_bits, make_qkv

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkg.library()


def run(q, k, v, causal, scale, poison=True):
    """Call the C ABI on fresh device copies; outputs are poisoned first so an unwritten element shows."""
    B, H, N, D = q.shape
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o = torch.full_like(qd, float("nan")) if poison else torch.empty_like(qd)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    st = pkg.attn_fwd(qd, kd, vd, o, lse, B, H, N, D, causal, scale, stream)
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    st = pkg.attn_last_status(stream)
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    return o_to_f64(o), lse.cpu().numpy().astype(np.float64)


def full_check(q, k, v, causal, scale, what):
    o, lse = run(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    return assert_close(o, lse, o_ref, lse_ref, what)


SMALL = ["b1h1n256d64", "b2h8n1024d64", "b2h8n1024d64_causal", "b16h32n512d64_causal"]


@pytest.mark.parametrize("name", SMALL)
def test_workload_full(name):
    w = WORKLOADS[name]
    q, k, v = w.qkv()
    full_check(q, k, v, w.causal, w.scale, name)


def run_qk_any(q, k, v, causal, scale):
    """attn_fwd (square) or attn_fwd_qk, as the bench launches the workload."""
    return run(q, k, v, causal, scale) if q.shape[2] == k.shape[2] else run_qk(q, k, v, causal, scale)


@pytest.mark.parametrize("name", ["b4h16n4096d128", "b1h16n16384d128_causal_q4", "b8h16nq512nk8192d128_causal"])
def test_full_size_every_row(name):
    """Full-size problems, every output row against the oracle: first in the
    bench's own launch configuration, then on the other grid (one CTA per unit
    <-> persistent) and with the other number of query tiles per unit."""
    w = WORKLOADS[name]
    q, k, v = w.qkv()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale)
    for grid, unit in ((0, 0), (1, 0), (2, 0), (0, 1)):
        tune(grid=grid, unit=unit)
        try:
            o, lse = run_qk_any(q, k, v, w.causal, w.scale)
        finally:
            tune(grid=0, unit=0)
        what = f"{name} grid={grid or 'auto'} unit={unit or 'auto'}"
        assert_close(o, lse, o_ref, lse_ref, what)
        print(what, parity_report(o, lse, o_ref, lse_ref))
        del o, lse


@pytest.fixture(params=[1, 2, 3, 4], ids=["one_tile_per_cta", "two_tiles_per_cta", "key_split", "short_kernel"])
def tiles_per_cta(request):
    """Force the launcher's choice of work unit (normally picked from the grid size): one or
    two query tiles, one tile with its key tiles split over both softmax warpgroups, or one
    tile on the short-unit kernel that runs two CTAs per SM (the last two D <= 64; at larger
    head dims the request runs as one tile per unit)."""
    tune(unit=request.param)
    yield request.param
    tune(unit=0)


@pytest.fixture(params=[1, 2], ids=["one_unit_per_cta", "persistent"])
def schedule(request):
    """Force the launcher's grid: one CTA per unit, or one CTA per SM walking the units."""
    tune(grid=request.param)
    yield request.param
    tune(grid=0)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 17, 127, 128, 129, 200, 383, 640])
def test_ragged_and_tiny_lengths(N, D, causal, tiles_per_cta, schedule):
    q, k, v = make_qkv(2, 3, N, D, seed=500 + N + D)
    full_check(q, k, v, causal, 1.0 / math.sqrt(D), f"N={N} D={D} causal={causal} T={tiles_per_cta}")


@pytest.mark.parametrize("D", [64, 128])
def test_large_logits_stress_rescaling(D, tiles_per_cta, schedule):
    # Q spread 8x: logits up to ~40 in magnitude; the running max moves often.
    q, k, v = make_qkv(1, 4, 1000, D, seed=77, q_std=8.0)
    for causal in (False, True):
        full_check(q, k, v, causal, 1.0 / math.sqrt(D), f"q_std=8 D={D} causal={causal} T={tiles_per_cta}")


@pytest.mark.parametrize("name", SMALL)
def test_workload_full_both_tilings(name, tiles_per_cta, schedule):
    w = WORKLOADS[name]
    q, k, v = w.qkv()
    full_check(q, k, v, w.causal, w.scale, f"{name} T={tiles_per_cta}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [640, 333])
def test_many_units_per_cta(N, D, causal, tiles_per_cta):
    """Persistent grid with several units per CTA (B*H*units well above the SM
    count): every unit's Q load, P V restart and epilogue reuse the buffers of
    the unit before.  Heads of different lengths' worth of work in causal order."""
    tune(grid=2)
    try:
        q, k, v = make_qkv(4, 100, N, D, seed=900 + N + D)
        full_check(q, k, v, causal, 1.0 / math.sqrt(D), f"N={N} D={D} causal={causal} T={tiles_per_cta} persistent")
    finally:
        tune(grid=0)


@pytest.mark.parametrize("D", [8, 40, 64])
@pytest.mark.parametrize("Nq,Nk,causal", [(1, 700, True), (200, 1000, True), (333, 333, True), (640, 200, False),
                                          (1000, 1000, False)])
def test_short_kernel_lengths(Nq, Nk, causal, D):
    """The short-unit kernel (two CTAs per SM, one tile per unit) on queries and keys of
    different lengths, head dims padded to 64, several units per CTA."""
    tune(unit=4)
    try:
        q = make_qkv(3, 70, Nq, D, seed=950 + Nq + D)[0]
        _, k, v = make_qkv(3, 70, Nk, D, seed=951 + Nk + D)
        o, lse = run_qk(q, k, v, causal, 1.0 / math.sqrt(D))
    finally:
        tune(unit=0)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(D))
    assert_close(o, lse, o_ref, lse_ref, f"short kernel Nq={Nq} Nk={Nk} D={D} causal={causal}")


def test_kernel_names_follow_the_launcher():
    """attn_fwd_kernel_name reports the launcher's choice, tuning included."""
    name = pkg.attn_fwd_kernel_name
    assert name(4, 16, 4096, 4096, 128, False) == "attn_fwd_sm103<128,full,persistent,2 tiles/unit>"
    assert name(1, 16, 16384, 16384, 128, True) == "attn_fwd_sm103<128,causal,one unit per CTA,2 tiles/unit>"
    assert name(4, 16, 4096, 4096, 128, True) == "attn_fwd_sm103<128,causal,one unit per CTA,2 tiles/unit>"
    assert name(8, 16, 2048, 2048, 128, True) == "attn_fwd_sm103<128,causal,persistent,2 tiles/unit>"
    assert name(16, 32, 512, 512, 64, True) == "attn_fwd_short_sm103<causal>"
    assert name(16, 32, 512, 512, 64, False) == "attn_fwd_short_sm103<full>"
    assert name(4, 16, 4096, 4096, 64, False) == "attn_fwd_sm103<64,full,persistent,2 tiles/unit>"
    assert name(2, 8, 1024, 1024, 64, False) == "attn_fwd_sm103<64,full,persistent,key split>"
    assert name(1, 2, 300, 300, 200, True).startswith("attn_fwd_sm103<256,causal,one unit per CTA,1 tile/unit")
    tune(unit=1, grid=1)
    try:
        assert name(16, 32, 512, 512, 64, True) == "attn_fwd_sm103<64,causal,one unit per CTA,1 tile/unit>"
    finally:
        tune(unit=0, grid=0)


def test_identical_keys_give_mean_of_v():
    B, H, N, D = 1, 2, 300, 128
    q, k, v = make_qkv(B, H, N, D, seed=78)
    k = np.broadcast_to(k[:, :, :1], k.shape).copy()
    full_check(q, k, v, True, 0.1, "identical keys")


def test_zero_queries_and_one_hot():
    B, H, N, D = 1, 1, 256, 64
    _, k, v = make_qkv(B, H, N, D, seed=79)
    full_check(np.zeros_like(k), k, v, False, 0.125, "Q = 0")
    sixteen = f64_to_bf16_bits(np.array([16.0]))[0]
    q = np.zeros_like(k)
    q[..., 0] = sixteen
    k1 = np.zeros_like(k)
    k1[0, 0, 100, 0] = sixteen
    full_check(q, k1, v, False, 0.125, "one-hot logit")
    full_check(q, k1, v, True, 0.125, "one-hot logit, causal")


def test_scale_variants():
    q, k, v = make_qkv(1, 2, 384, 64, seed=80)
    for scale in (1e-3, 0.05, 0.5):
        full_check(q, k, v, False, scale, f"scale={scale}")


def test_deterministic():
    q, k, v = make_qkv(2, 4, 1024, 128, seed=81)
    o1, l1 = run(q, k, v, True, 0.088)
    o2, l2 = run(q, k, v, True, 0.088)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_many_heads_beyond_int32_offsets():
    # 270000 (batch, head) slices of one 128-row tile: a grid of 270000 CTAs and
    # 2.2e9 elements per tensor, so element offsets pass 2^31.  The inputs are 16
    # seeded heads repeated on the device; the oracle checks sampled rows.
    H0, reps, N, D = 16, 16875, 128, 64
    q0, k0, v0 = make_qkv(1, H0, N, D, seed=82)
    BH = H0 * reps
    big = lambda a: to_dev(a).expand(reps, H0, N, D).reshape(1, BH, N, D).contiguous()  # noqa: E731
    qd, kd, vd = big(q0), big(k0), big(v0)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((1, BH, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream()
    assert pkg.attn_fwd(qd, kd, vd, o, lse, 1, BH, N, D, True, 0.125, s) == pkg.ATTN_OK
    assert pkg.attn_last_status(s) == pkg.ATTN_OK
    rng = np.random.default_rng(82)
    bh = np.concatenate([rng.integers(0, BH, 2048), np.full(128, BH - 1)]).astype(np.int64)
    ri = np.concatenate([rng.integers(0, N, 2048), np.arange(128)]).astype(np.int64)
    idx_bh = torch.from_numpy(bh).cuda()
    idx_r = torch.from_numpy(ri).cuda()
    of = o.view(BH, N, D)[idx_bh, idx_r].float().cpu().numpy().astype(np.float64)
    lf = lse.view(BH, N)[idx_bh, idx_r].cpu().numpy().astype(np.float64)
    o_ref, lse_ref = oracle.attn_rows(q0, k0, v0, True, 0.125, bh % H0, ri)
    assert_close(of, lf, o_ref, lse_ref, "270000 heads")
    # Every row: each repetition of the 16 heads against the oracle's output for
    # them, compared on the device chunk by chunk (the output is 4.4 GB).
    o16, l16 = oracle.attn_fwd(q0, k0, v0, True, 0.125)
    o16d = torch.from_numpy(o16).cuda().reshape(1, H0, N, D)
    l16d = torch.from_numpy(l16).cuda().reshape(1, H0, N)
    ov, lv = o.view(reps, H0, N, D), lse.view(reps, H0, N)
    mx, tot, lerr = 0.0, 0.0, 0.0
    for r0 in range(0, reps, 1024):
        d = (ov[r0:r0 + 1024].double() - o16d).abs()
        mx = max(mx, float(d.max()))
        tot += float(d.sum())
        dl = (lv[r0:r0 + 1024].double() - l16d).abs() / l16d.abs().clamp(min=1.0)
        lerr = max(lerr, float(dl.max()))
        del d, dl
    mean = tot / (BH * N * D)
    assert mx <= 2e-2 and mean <= 2e-3 and lerr <= 1e-3, f"270000 heads: {mx:.3e} {mean:.3e} {lerr:.3e}"
    del qd, kd, vd, o, lse, ov, lv
    torch.cuda.empty_cache()


def test_long_sequence():
    B, H, N, D = 1, 1, 32768 + 77, 128
    q, k, v = make_qkv(B, H, N, D, seed=83)
    o, lse = run(q, k, v, True, 1.0 / math.sqrt(D))
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 1.0 / math.sqrt(D))
    assert_close(o, lse, o_ref, lse_ref, "N=32845 causal, every row")


def test_empty_problem_leaves_outputs_untouched():
    o = torch.full((0, 2, 128, 64), 1.0, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros_like(o)
    lse = torch.zeros((0, 2, 128), device="cuda")
    assert pkg.attn_fwd(q, q, q, o, lse, 0, 2, 128, 64, False, 0.125, None) == pkg.ATTN_OK


def test_boundary_errors_with_real_buffers():
    q = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 256), device="cuda")
    s = torch.cuda.current_stream()
    assert pkg.attn_fwd(q.data_ptr() + 2, q, q, o, lse, 1, 1, 255, 64, False, 0.125, s) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_fwd(q, q, q, q, lse, 1, 1, 256, 64, False, 0.125, s) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_fwd(q, q, q, o, lse, 1, 1, 256, 100, False, 0.125, s) == pkg.ATTN_ERR_UNSUPPORTED
    assert pkg.attn_last_status(s) == pkg.ATTN_OK


def test_side_stream_and_fwd_wrapper():
    q, k, v = make_qkv(1, 2, 512, 128, seed=84)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = pkg.fwd(to_dev(q), to_dev(k), to_dev(v), causal=True)
    s.synchronize()
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 1.0 / math.sqrt(128))
    assert_close(o_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "side stream")


def run_qk(q, k, v, causal, scale):
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    st = pkg.attn_fwd_qk(qd, kd, vd, o, lse, B, H, Nq, Nk, D, causal, scale, stream)
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    assert pkg.attn_last_status(stream) == pkg.ATTN_OK
    return o_to_f64(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Nq,Nk,causal", [
    (1, 1000, True), (1, 1000, False), (17, 300, True), (128, 4096, True), (200, 333, True),
    (300, 300, True), (700, 129, False), (1000, 77, False), (384, 2048, False),
])
def test_queries_and_keys_of_different_lengths(Nq, Nk, causal, D, tiles_per_cta, schedule):
    q, _, _ = make_qkv(2, 3, Nq, D, seed=900 + Nq)
    _, k, v = make_qkv(2, 3, Nk, D, seed=901 + Nk)
    scale = 1.0 / math.sqrt(D)
    o, lse = run_qk(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    assert_close(o, lse, o_ref, lse_ref, f"Nq={Nq} Nk={Nk} D={D} causal={causal} T={tiles_per_cta}")


def test_square_qk_call_is_attn_fwd():
    q, k, v = make_qkv(1, 4, 640, 128, seed=950)
    a = run_qk(q, k, v, True, 0.09)
    b = run(q, k, v, True, 0.09)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_fwd_wrapper_with_a_key_cache():
    q, _, _ = make_qkv(1, 2, 256, 64, seed=951)
    _, k, v = make_qkv(1, 2, 1500, 64, seed=952)
    o, lse = pkg.fwd(to_dev(q), to_dev(k), to_dev(v), causal=True)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 0.125)
    assert_close(o_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, "fwd() Nq=256 Nk=1500")


@pytest.mark.parametrize("D", [8, 32, 48, 96, 112])
@pytest.mark.parametrize("causal", [False, True])
def test_padded_head_dims(D, causal, tiles_per_cta, schedule):
    q, k, v = make_qkv(2, 3, 333, D, seed=1600 + D)
    full_check(q, k, v, causal, 1.0 / math.sqrt(D), f"D={D} causal={causal} T={tiles_per_cta}")
    qr, _, _ = make_qkv(1, 2, 100, D, seed=1601 + D)
    _, kr, vr = make_qkv(1, 2, 450, D, seed=1602 + D)
    o, lse = run_qk(qr, kr, vr, causal, 0.3)
    o_ref, lse_ref = oracle.attn_fwd(qr, kr, vr, causal, 0.3)
    assert_close(o, lse, o_ref, lse_ref, f"Nq=100 Nk=450 D={D} causal={causal}")


@pytest.mark.parametrize("D", [136, 192, 256])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 127, 300, 640])
def test_wide_head_dims(N, D, causal):
    """Head dims above 128 run on the D = 256 kernel (one query tile per CTA, zero padding below 256)."""
    q, k, v = make_qkv(2, 3, N, D, seed=1300 + N + D)
    full_check(q, k, v, causal, 1.0 / math.sqrt(D), f"N={N} D={D} causal={causal}")


@pytest.mark.parametrize("Nq,Nk,causal", [(100, 700, True), (384, 129, False), (513, 1000, True)])
def test_wide_head_dims_queries_and_keys_of_different_lengths(Nq, Nk, causal):
    D = 256
    q = make_qkv(2, 2, Nq, D, seed=1400 + Nq)[0]
    _, k, v = make_qkv(2, 2, Nk, D, seed=1500 + Nk)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((2, 2, Nq), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    assert pkg.attn_fwd_qk(qd, kd, vd, o, lse, 2, 2, Nq, Nk, D, causal, 0.0625, stream) == pkg.ATTN_OK
    assert pkg.attn_last_status(stream) == pkg.ATTN_OK
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 0.0625)
    assert_close(o_to_f64(o), lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, f"D=256 Nq={Nq} Nk={Nk}")


def test_wide_head_dims_large_logits_and_many_tiles():
    """D = 256, Q spread 4x, 2048 keys (16 key steps through the two-slot ring), causal and not."""
    q, k, v = make_qkv(1, 4, 2048, 256, seed=1600, q_std=4.0)
    for causal in (False, True):
        full_check(q, k, v, causal, 1.0 / 16, f"D=256 N=2048 q_std=4 causal={causal}")




def padded(bits, ld, fill):
    """A [B, H, N, ld] device buffer: ``bits`` in the first D columns, zeros up to roundup8(D)
    (the group of 16 bytes the kernels use), ``fill`` bits beyond."""
    B, H, N, D = bits.shape
    buf = np.full((B, H, N, ld), fill, dtype=np.uint16)
    buf[..., :(D + 7) // 8 * 8] = 0
    buf[..., :D] = bits
    return to_dev(buf)


@pytest.mark.parametrize("D,ld", [(4, 8), (12, 24), (100, 104), (100, 112), (200, 208), (1, 16)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(300, 300), (100, 450)])
def test_padded_rows_any_head_dim(D, ld, causal, Nq, Nk):
    """attn_fwd_ld: rows ld elements apart, head dims that are not multiples of 8.  Beyond
    roundup8(D) the inputs hold NaN (never read) and o a sentinel (never written); the columns
    D..roundup8(D)-1 of o come back zero."""
    q = make_qkv(2, 3, Nq, D, seed=1700 + D + Nq)[0]
    _, k, v = make_qkv(2, 3, Nk, D, seed=1701 + D + Nk)
    nan, sentinel = 0x7FC0, 0x4049  # bf16 NaN, 3.140625
    qd, kd, vd = padded(q, ld, nan), padded(k, ld, nan), padded(v, ld, nan)
    od = padded(np.zeros((2, 3, Nq, D), np.uint16), ld, sentinel)
    od[..., :D] = float("nan")
    lse = torch.full((2, 3, Nq), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    scale = 1.0 / math.sqrt(D)
    st = pkg.attn_fwd_ld(qd, kd, vd, od, lse, 2, 3, Nq, Nk, D, ld, causal, scale, s)
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    assert pkg.attn_last_status(s) == pkg.ATTN_OK
    d8 = (D + 7) // 8 * 8
    ob = od.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.all(ob[..., d8:] == sentinel), "columns past roundup8(D) of o were written"
    assert np.all(ob[..., D:d8] == 0), "columns D..roundup8(D)-1 of o are not zero"
    o = od[..., :D].float().cpu().numpy().astype(np.float64)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    assert_close(o, lse.cpu().numpy().astype(np.float64), o_ref, lse_ref, f"D={D} ld={ld} causal={causal} Nq={Nq} Nk={Nk}")
