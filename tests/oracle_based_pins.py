"""Pins for the Based linear-attention oracle: facts fixed outside its own code.

Each ``check_*`` takes an oracle object (``oracle.Oracle``) and raises
``AssertionError`` when the oracle disagrees with the fact it checks.

The definition (Based, Arora et al. 2024; the pages name the kernel only):
causal linear attention with the second-order Taylor kernel
a_ij = 1 + s_ij + s_ij^2 / 2, s_ij = scale * q_i . k_j, output
y_i = sum_{j<=i} a_ij v_j / z_i with z_i = sum_{j<=i} a_ij.  The facts:

* exact rational arithmetic (``fractions``) on tiny inputs: the definition
  evaluated with no rounding at all;
* the linear-attention recurrence: an independent numpy restatement through
  an explicit feature map phi(x) = [1, x sqrt(scale), vec(x x^T) scale / sqrt 2]
  (1 + F + F^2 features) and running sums of phi(k_j) v_j^T and phi(k_j) --
  the form Based computes in -- equals the quadratic definition;
* closed forms: zero queries or identical keys (prefix means of V), the first
  row, a single feature with known dot products;
* invariants: y_i is a convex combination of v_0..v_i, z_i >= (i + 1) / 2,
  causality (later keys do not move earlier rows), (batch, head) independence,
  and the sampled-row entry point equals the full one.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from tiled_attention_forward_fa2_gb300.inputs import bf16_bits_to_f64, f64_to_bf16_bits, make_qkv, normal_bf16_bits


def _close(a, b, tol, what, rel=False):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.abs(a - b)
    if rel:
        err = err / np.maximum(np.abs(b), 1e-300)
    m = float(err.max()) if err.size else 0.0
    assert np.all(np.isfinite(a)) and m <= tol, f"{what}: max {'rel ' if rel else ''}|diff| = {m:.3e} > {tol:.1e}"


def based_inputs(B, H, N, F, D, seed, q_std=1.0):
    """q, k [B,H,N,F] and v [B,H,N,D] bf16 bits from the seeded generator."""
    q = normal_bf16_bits(B * H * N * F, seed, 0, q_std).reshape(B, H, N, F)
    k = normal_bf16_bits(B * H * N * F, seed, 1).reshape(B, H, N, F)
    v = normal_bf16_bits(B * H * N * D, seed, 2).reshape(B, H, N, D)
    return q, k, v


def _frac(bits):
    return [[Fraction(float(x)) for x in row] for row in bf16_bits_to_f64(bits)]


# ---------------------------------------------------------------- definition

def check_based_exact_rational(orc):
    """Tiny problems evaluated exactly with fractions: every input is a binary
    rational, so is the scale, and the definition has no transcendental step."""
    for scale in (0.25, 0.3):
        q, k, v = based_inputs(1, 2, 6, 3, 2, seed=21, q_std=1.5)
        y, z = orc.based_fwd(q, k, v, scale)
        sc = Fraction(scale)
        for h in range(2):
            Q, K, V = _frac(q[0, h]), _frac(k[0, h]), _frac(v[0, h])
            for i in range(6):
                zz = Fraction(0)
                yy = [Fraction(0), Fraction(0)]
                for j in range(i + 1):
                    s = sc * sum(Q[i][a] * K[j][a] for a in range(3))
                    w = 1 + s + s * s / 2
                    zz += w
                    for d in range(2):
                        yy[d] += w * V[j][d]
                _close(z[0, h, i], float(zz), 1e-15, f"z exact (h={h}, i={i}, scale={scale})", rel=True)
                for d in range(2):
                    ref = float(yy[d] / zz)
                    assert abs(y[0, h, i, d] - ref) <= 1e-15 * max(1.0, abs(ref)), \
                        f"y exact (h={h}, i={i}, d={d}): {y[0, h, i, d]!r} vs {ref!r}"


def _phi(x, scale):
    """Explicit second-order Taylor feature map of exp(scale * x.y): 1 + F + F^2 features."""
    n, F = x.shape
    quad = (x[:, :, None] * x[:, None, :]).reshape(n, F * F) * (scale / np.sqrt(2.0))
    return np.concatenate([np.ones((n, 1)), x * np.sqrt(scale), quad], axis=1)


def check_based_recurrent_form(orc):
    """The running-state (linear attention) form equals the quadratic definition."""
    B, H, N, F, D = 2, 2, 300, 16, 64
    scale = 1.0 / np.sqrt(F)
    q, k, v = based_inputs(B, H, N, F, D, seed=22)
    y, z = orc.based_fwd(q, k, v, scale)
    qf, kf, vf = bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)
    for b in range(B):
        for h in range(H):
            pq, pk = _phi(qf[b, h], scale), _phi(kf[b, h], scale)
            state = np.zeros((pq.shape[1], D))
            zeta = np.zeros(pq.shape[1])
            yr = np.empty((N, D))
            zr = np.empty(N)
            for i in range(N):
                state += np.outer(pk[i], vf[b, h, i])
                zeta += pk[i]
                zr[i] = pq[i] @ zeta
                yr[i] = (pq[i] @ state) / zr[i]
            _close(z[b, h], zr, 1e-11, f"z recurrent (b={b}, h={h})", rel=True)
            _close(y[b, h], yr, 1e-11, f"y recurrent (b={b}, h={h})")


# ---------------------------------------------------------------- closed forms

def _prefix_mean(vf):
    return np.cumsum(vf, axis=-2) / np.arange(1, vf.shape[-2] + 1)[:, None]


def check_based_zero_queries(orc):
    """q = 0: every weight is 1, so y_i is the mean of v_0..v_i and z_i = i + 1."""
    _, k, v = based_inputs(1, 2, 130, 16, 32, seed=23)
    q = np.zeros_like(k)
    y, z = orc.based_fwd(q, k, v, 0.25)
    _close(z, np.broadcast_to(np.arange(1, 131, dtype=np.float64), z.shape), 0.0, "z with q = 0")
    _close(y, _prefix_mean(bf16_bits_to_f64(v)), 1e-14, "y with q = 0")


def check_based_identical_keys(orc):
    """All keys equal: the weights of row i are all a_i = 1 + s_i + s_i^2/2, so y_i is
    the prefix mean of V and z_i = (i + 1) a_i."""
    q, k, v = based_inputs(1, 1, 90, 8, 16, seed=24, q_std=2.0)
    k = np.broadcast_to(k[:, :, :1], k.shape).copy()
    scale = 0.35
    y, z = orc.based_fwd(q, k, v, scale)
    s = scale * (bf16_bits_to_f64(q)[0, 0] @ bf16_bits_to_f64(k)[0, 0, 0])
    a = 1.0 + s + 0.5 * s * s
    _close(z[0, 0], np.arange(1, 91) * a, 1e-13, "z with identical keys", rel=True)
    _close(y, _prefix_mean(bf16_bits_to_f64(v)), 1e-13, "y with identical keys")


def check_based_first_row(orc):
    """Row 0 sees only key 0: y_0 = v_0, z_0 = 1 + s + s^2/2."""
    q, k, v = based_inputs(2, 3, 7, 16, 24, seed=25)
    y, z = orc.based_fwd(q, k, v, 0.25)
    qf, kf = bf16_bits_to_f64(q), bf16_bits_to_f64(k)
    s = 0.25 * np.einsum("bhf,bhf->bh", qf[:, :, 0], kf[:, :, 0])
    _close(z[:, :, 0], 1.0 + s + 0.5 * s * s, 1e-15, "z_0", rel=True)
    _close(y[:, :, 0], bf16_bits_to_f64(v)[:, :, 0], 2e-15, "y_0 = v_0 (up to the rounding of w v / w)")


def check_based_known_weights(orc):
    """One feature, keys with chosen dot products: the weights are the Taylor
    polynomial at those values (distinguishes 1 + s + s^2/2 from any other
    quadratic), and y follows from them."""
    vals = np.array([0.0, 1.0, -2.0, 3.0, 0.5])
    k = np.zeros((1, 1, 5, 8))
    k[0, 0, :, 0] = vals
    q = np.zeros((1, 1, 5, 8))
    q[0, 0, :, 0] = 2.0
    v = np.zeros((1, 1, 5, 4))
    v[0, 0, :, 0] = 1.0
    v[0, 0, :, 1] = np.arange(5)
    qb, kb, vb = f64_to_bf16_bits(q), f64_to_bf16_bits(k), f64_to_bf16_bits(v)
    for scale in (0.5, 0.125):
        y, z = orc.based_fwd(qb, kb, vb, scale)
        s = scale * 2.0 * vals
        w = 1.0 + s + 0.5 * s * s
        _close(z[0, 0], np.cumsum(w), 1e-15, f"z with known weights (scale={scale})", rel=True)
        _close(y[0, 0, :, 0], 1.0, 1e-15, "y of a constant column")
        _close(y[0, 0, :, 1], np.cumsum(w * np.arange(5)) / np.cumsum(w), 1e-15, "y of a ramp column")


# ---------------------------------------------------------------- invariants

def check_based_convex_combination(orc):
    """Positive weights: every y_id lies within [min, max] of v_0d..v_id; z_i >= (i+1)/2."""
    q, k, v = based_inputs(1, 3, 200, 16, 16, seed=26, q_std=3.0)
    y, z = orc.based_fwd(q, k, v, 0.25)
    vf = bf16_bits_to_f64(v)
    lo = np.minimum.accumulate(vf, axis=2)
    hi = np.maximum.accumulate(vf, axis=2)
    assert np.all(y >= lo - 1e-12) and np.all(y <= hi + 1e-12), "y outside the hull of the visible values"
    assert np.all(z >= 0.5 * np.arange(1, 201) - 1e-12), "z below (i + 1) / 2"


def check_based_causality(orc):
    """Keys and values after position i do not change rows up to i."""
    q, k, v = based_inputs(1, 2, 96, 16, 32, seed=27)
    y, z = orc.based_fwd(q, k, v, 0.25)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 60:] = normal_bf16_bits(k2[:, :, 60:].size, 99, 1).reshape(k2[:, :, 60:].shape)
    v2[:, :, 60:] = normal_bf16_bits(v2[:, :, 60:].size, 99, 2).reshape(v2[:, :, 60:].shape)
    y2, z2 = orc.based_fwd(q, k2, v2, 0.25)
    _close(y2[:, :, :60], y[:, :, :60], 0.0, "rows before the change")
    _close(z2[:, :, :60], z[:, :, :60], 0.0, "z before the change")
    assert np.max(np.abs(y2[:, :, 60:] - y[:, :, 60:])) > 1e-3, "later rows ignored the change"


def check_based_head_independence_and_rows(orc):
    """Each (b, h) slice equals a B = H = 1 run on it; sampled rows equal full rows."""
    q, k, v = based_inputs(2, 3, 40, 16, 8, seed=28)
    y, z = orc.based_fwd(q, k, v, 0.25)
    for b in range(2):
        for h in range(3):
            y1, z1 = orc.based_fwd(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], 0.25)
            _close(y1[0, 0], y[b, h], 0.0, f"slice ({b}, {h})")
            _close(z1[0, 0], z[b, h], 0.0, f"slice z ({b}, {h})")
    bh = np.array([0, 5, 3, 2], np.int64)
    ri = np.array([0, 39, 17, 5], np.int64)
    yr, zr = orc.based_rows(q, k, v, 0.25, bh, ri)
    _close(yr, y.reshape(6, 40, 8)[bh, ri], 0.0, "sampled rows")
    _close(zr, z.reshape(6, 40)[bh, ri], 0.0, "sampled z")


ALL_BASED_CHECKS = [
    check_based_exact_rational,
    check_based_recurrent_form,
    check_based_zero_queries,
    check_based_identical_keys,
    check_based_first_row,
    check_based_known_weights,
    check_based_convex_combination,
    check_based_causality,
    check_based_head_independence_and_rows,
]
