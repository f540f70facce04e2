"""Based linear-attention CUDA path against the CPU oracle, element by element, through the C ABI.

Tolerance (derived from the arithmetic; a CPU emulation of the kernel's
rounding -- bf16 features, weights and state, fp32 accumulation -- gives
max |dy| 7e-3 (the bf16 rounding of y at |y| ~ 3.6), mean |dy| 1.4e-4 and a
relative z error of 0.6 % on these inputs): max |dy| <= 2e-2, mean |dy| <= 1e-3,
|dz| / z <= 2^-6.
"""
import numpy as np
import pytest

import oracle
import tiled_attention_forward_fa2_gb300 as pkg
from oracle_based_pins import based_inputs
from parity import o_to_f64, to_dev
from tiled_attention_forward_fa2_gb300.inputs import BASED_WORKLOADS

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MAX_DY, MEAN_DY, Z_REL = 2e-2, 1e-3, 2.0 ** -6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    pkg.library()


def run(q, k, v, scale):
    B, H, N, F = q.shape
    D = v.shape[3]
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    y = torch.full_like(vd, float("nan"))
    z = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream()
    st = pkg.attn_based_fwd(qd, kd, vd, y, z, B, H, N, F, D, scale, s)
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    st = pkg.attn_last_status(s)
    assert st == pkg.ATTN_OK, pkg.attn_status_string(st)
    return o_to_f64(y), z.cpu().numpy().astype(np.float64)


def check(y, z, y_ref, z_ref, what):
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(z)), f"{what}: non-finite or unwritten output"
    dy = np.abs(y - y_ref)
    zr = float((np.abs(z - z_ref) / z_ref).max())
    assert dy.max() <= MAX_DY and dy.mean() <= MEAN_DY and zr <= Z_REL, \
        f"{what}: max|dy|={dy.max():.3e} mean|dy|={dy.mean():.3e} z_rel={zr:.3e}"
    return float(dy.max()), float(dy.mean()), zr


def full_check(q, k, v, scale, what):
    y, z = run(q, k, v, scale)
    y_ref, z_ref = oracle.based_fwd(q, k, v, scale)
    return check(y, z, y_ref, z_ref, what)


@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 300, 640, 1000])
@pytest.mark.parametrize("F,D", [(16, 64), (8, 32), (16, 8)])
def test_lengths_and_dims(N, F, D):
    q, k, v = based_inputs(2, 3, N, F, D, seed=3000 + N + F + D)
    full_check(q, k, v, 1.0 / np.sqrt(F), f"N={N} F={F} D={D}")


@pytest.mark.parametrize("name", sorted(BASED_WORKLOADS))
def test_workloads_every_row(name):
    """The named problems at full size (the bench's launch), every output row."""
    w = BASED_WORKLOADS[name]
    q, k, v = w.qkv()
    print(name, full_check(q, k, v, w.scale, name))


def test_large_features_and_scales():
    """q spread 3x (s up to ~10: the quadratic term dominates), and scales off the default."""
    q, k, v = based_inputs(1, 4, 2000, 16, 64, seed=3100, q_std=3.0)
    full_check(q, k, v, 0.25, "q_std=3")
    for scale in (0.05, 0.4):
        full_check(q, k, v, scale, f"scale={scale}")


def test_zero_queries_give_prefix_means():
    _, k, v = based_inputs(1, 2, 700, 16, 64, seed=3200)
    q = np.zeros_like(k)
    y, z = run(q, k, v, 0.25)
    vf = v.astype(np.uint32) << 16
    vf = vf.view(np.float32).astype(np.float64)
    mean = np.cumsum(vf, axis=2) / np.arange(1, 701)[:, None]
    assert np.max(np.abs(y - mean)) <= MAX_DY
    assert np.max(np.abs(z - np.arange(1, 701)) / np.arange(1, 701)) <= Z_REL


def test_deterministic():
    q, k, v = based_inputs(2, 2, 1500, 16, 64, seed=3300)
    a = run(q, k, v, 0.25)
    b = run(q, k, v, 0.25)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_many_sequences():
    """More sequences than SMs (several waves of CTAs), ragged length."""
    q, k, v = based_inputs(4, 100, 333, 16, 64, seed=3400)
    full_check(q, k, v, 0.25, "400 sequences")


def test_boundary_errors_with_real_buffers():
    q = torch.zeros((1, 1, 256, 16), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(v)
    z = torch.empty((1, 1, 256), device="cuda")
    s = torch.cuda.current_stream()
    assert pkg.attn_based_fwd(q, q, v, y, z, 1, 1, 256, 32, 64, 0.25, s) == pkg.ATTN_ERR_UNSUPPORTED
    assert pkg.attn_based_fwd(q, q, v, y, z, 1, 1, 256, 16, 128, 0.25, s) == pkg.ATTN_ERR_UNSUPPORTED
    assert pkg.attn_based_fwd(q, q, v, v, z, 1, 1, 256, 16, 64, 0.25, s) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_based_fwd(q.data_ptr() + 2, q, v, y, z, 1, 1, 255, 16, 64, 0.25, s) == pkg.ATTN_ERR_INVALID_ARG
    assert pkg.attn_last_status(s) == pkg.ATTN_OK


def test_based_fwd_wrapper_side_stream():
    q, k, v = based_inputs(1, 2, 512, 16, 64, seed=3500)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        y, z = pkg.based_fwd(to_dev(q), to_dev(k), to_dev(v))
    st.synchronize()
    y_ref, z_ref = oracle.based_fwd(q, k, v, 0.25)
    check(o_to_f64(y), z.cpu().numpy().astype(np.float64), y_ref, z_ref, "based_fwd() on a side stream")
