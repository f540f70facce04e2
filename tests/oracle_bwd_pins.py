"""Pins for the backward oracle: facts fixed outside its own code.

* finite differences of the forward (central, fp64) along random directions;
* a library routine: torch autograd through scaled_dot_product_attention in fp64;
* closed forms and invariants of the softmax chain rule: identical keys give
  dQ = 0; the key gradients of a head sum to zero (softmax is unchanged when
  every key moves by the same vector); D_i equals dO_i . O_i; with dO = 1 the
  value gradient of key j is the column sum of P;
* the sampled functions (dQ of chosen rows, dK and dV of chosen keys, used at
  sizes the full backward cannot reach) agree with the pinned full backward.
"""
from __future__ import annotations

import math

import numpy as np

from tiled_attention_forward_fa2_gb300.inputs import bf16_bits_to_f64, make_qkv

TIGHT = 1e-12


def _close(a, b, tol, what):
    err = float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0
    assert np.all(np.isfinite(a)) and err <= tol, f"{what}: max |diff| = {err:.3e} > {tol:.1e}"


def check_bwd_finite_differences(orc):
    rng = np.random.default_rng(7)
    for (Nq, Nk, causal) in [(9, 13, False), (13, 13, True), (5, 11, True)]:
        B, H, D = 1, 2, 8
        q = rng.standard_normal((B, H, Nq, D))
        k = rng.standard_normal((B, H, Nk, D))
        v = rng.standard_normal((B, H, Nk, D))
        do = rng.standard_normal((B, H, Nq, D))
        scale = 0.4
        g = orc.attn_bwd_f64(q, k, v, do, causal, scale)
        loss = lambda q_, k_, v_: float(np.sum(do * orc.attn_bwd_f64(q_, k_, v_, do, causal, scale)["o"]))  # noqa: E731
        eps = 1e-5
        for name, x, grad in (("q", q, g["dq"]), ("k", k, g["dk"]), ("v", v, g["dv"])):
            e = rng.standard_normal(x.shape)
            args = {"q": q, "k": k, "v": v}
            plus = dict(args, **{name: x + eps * e})
            minus = dict(args, **{name: x - eps * e})
            fd = (loss(plus["q"], plus["k"], plus["v"]) - loss(minus["q"], minus["k"], minus["v"])) / (2 * eps)
            an = float(np.sum(grad * e))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(an)), f"d{name} (Nq={Nq}, Nk={Nk}, causal={causal}): fd {fd} vs {an}"


def check_bwd_matches_torch_autograd(orc):
    import torch

    for (Nq, Nk, causal, D) in [(40, 40, True, 16), (33, 70, False, 32), (20, 50, True, 8)]:
        q, _, _ = make_qkv(1, 2, Nq, D, seed=400 + Nq)
        _, k, v = make_qkv(1, 2, Nk, D, seed=401 + Nk)
        do, _, _ = make_qkv(1, 2, Nq, D, seed=402 + Nq)
        scale = float(np.float32(1.0 / math.sqrt(D)))
        g = orc.attn_bwd(q, k, v, do, causal, scale)
        Q, K, V = (torch.from_numpy(bf16_bits_to_f64(x)).requires_grad_(True) for x in (q, k, v))
        mask = torch.ones(Nq, Nk, dtype=torch.bool)
        if causal:
            mask = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
        out = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
        out.backward(torch.from_numpy(bf16_bits_to_f64(do)))
        _close(g["dq"], Q.grad.numpy(), TIGHT, f"dQ vs torch autograd (Nq={Nq}, Nk={Nk})")
        _close(g["dk"], K.grad.numpy(), TIGHT, f"dK vs torch autograd (Nq={Nq}, Nk={Nk})")
        _close(g["dv"], V.grad.numpy(), TIGHT, f"dV vs torch autograd (Nq={Nq}, Nk={Nk})")


def check_bwd_identical_keys_give_zero_dq(orc):
    q, k, v = make_qkv(1, 2, 30, 16, seed=410)
    do, _, _ = make_qkv(1, 2, 30, 16, seed=411)
    k = np.broadcast_to(k[:, :, :1], k.shape).copy()
    for causal in (False, True):
        g = orc.attn_bwd(q, k, v, do, causal, 0.3)
        _close(g["dq"], 0.0, TIGHT, "identical keys: dQ = 0")


def check_bwd_key_gradients_sum_to_zero(orc):
    q, _, _ = make_qkv(2, 2, 25, 8, seed=412)
    _, k, v = make_qkv(2, 2, 31, 8, seed=413)
    do, _, _ = make_qkv(2, 2, 25, 8, seed=414)
    for causal in (False, True):
        g = orc.attn_bwd(q, k, v, do, causal, 0.5)
        _close(g["dk"].sum(axis=2), 0.0, 1e-11, "sum over keys of dK = 0")


def check_bwd_delta_is_do_dot_o(orc):
    q, k, v = make_qkv(1, 3, 27, 16, seed=415)
    do, _, _ = make_qkv(1, 3, 27, 16, seed=416)
    for causal in (False, True):
        g = orc.attn_bwd(q, k, v, do, causal, 0.25)
        _close(g["delta"], np.sum(bf16_bits_to_f64(do) * g["o"], axis=-1), TIGHT, "D = dO . O")


def check_bwd_unit_upstream_gives_column_sums(orc):
    q, k, v = make_qkv(1, 2, 22, 8, seed=417)
    ones = np.full(q.shape, 0x3F80, dtype=np.uint16)  # bf16 1.0
    for causal in (False, True):
        g = orc.attn_bwd(q, k, v, ones, causal, 0.35)
        _, _, p = orc.attn_probs(q, k, v, causal, 0.35)
        _close(g["dv"], np.broadcast_to(p.sum(axis=2)[..., None], g["dv"].shape), TIGHT, "dO = 1: dV = column sums of P")


def check_bwd_sampled_outputs_match_full(orc):
    """The sampled functions (dQ rows; dK, dV of chosen keys) against the full,
    pinned backward, square and rectangular, causal or not, ragged tiles."""
    rng = np.random.default_rng(17)
    for (B, H, Nq, Nk, D, causal) in ((1, 2, 70, 70, 16, True), (2, 1, 33, 90, 8, True), (1, 2, 50, 40, 12, False)):
        q = make_qkv(B, H, Nq, D, seed=80 + Nq)[0]
        _, k, v = make_qkv(B, H, Nk, D, seed=81 + Nk)
        do = make_qkv(B, H, Nq, D, seed=82)[1]
        scale = 0.4
        full = orc.attn_bwd(q, k, v, do, causal, scale)
        bh = rng.integers(0, B * H, 40)
        ri = rng.integers(0, Nq, 40)
        dq, delta = orc.attn_bwd_rows(q, k, v, do, causal, scale, bh, ri)
        _close(dq, full["dq"].reshape(B * H, Nq, D)[bh, ri], TIGHT, "sampled dQ rows")
        _close(delta, full["delta"].reshape(B * H, Nq)[bh, ri], TIGHT, "sampled D")
        for h in range(B * H):
            kj = rng.integers(0, Nk, 25)
            dk, dv = orc.attn_bwd_keys(q, k, v, do, causal, scale, h, kj)
            _close(dk, full["dk"].reshape(B * H, Nk, D)[h, kj], TIGHT, "sampled dK")
            _close(dv, full["dv"].reshape(B * H, Nk, D)[h, kj], TIGHT, "sampled dV")


ALL_BWD_CHECKS = [
    check_bwd_finite_differences,
    check_bwd_matches_torch_autograd,
    check_bwd_identical_keys_give_zero_dq,
    check_bwd_key_gradients_sum_to_zero,
    check_bwd_delta_is_do_dot_o,
    check_bwd_unit_upstream_gives_column_sums,
    check_bwd_sampled_outputs_match_full,
]
