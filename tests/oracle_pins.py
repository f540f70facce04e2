"""Pins for the CPU oracle: facts fixed by the pages and by mathematics.

Each ``check_*`` takes an oracle object (``oracle.Oracle``) and raises
``AssertionError`` when the oracle disagrees with the fact it checks.  The
facts come from outside the oracle's own code:

* the softmax definition (null-ptr.tistory.com "development" softmax post,
  "Original softmax"): rows of the probability matrix sum to one;
* the FlashAttention claim ("[GPU] Deep Learning for HPC", section "Flash
  Attention"): tiling the score matrix and keeping only running statistics
  gives the same result -- checked against an independent numpy restatement of
  the tiled online-softmax recurrence;
* closed forms: identical keys, zero queries, a one-hot dominant logit, the
  first causal row, a common logit shift;
* invariants: joint key/value permutation, (batch, head) independence;
* a library routine: torch's scaled_dot_product_attention in fp64 on the CPU;
* brute force: a 50-digit ``decimal`` evaluation on tiny inputs.

``tests/test_oracle_mutants.py`` plants plausible mistakes in copies of the
oracle's C source and shows that each one fails at least one of these checks.
"""
from __future__ import annotations

import decimal
import math

import numpy as np

from tiled_attention_forward_fa2_gb300.inputs import bf16_bits_to_f64, f64_to_bf16_bits, make_qkv

TIGHT = 1e-12


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert np.all(np.isfinite(a)) and err <= tol, f"{what}: max |diff| = {err:.3e} > {tol:.1e}"


def _vis_counts(N, causal):
    i = np.arange(N)
    return (i + 1) if causal else np.full(N, N)


# ---------------------------------------------------------------- definition

def check_prob_rows_sum_to_one(orc):
    for causal in (False, True):
        q, k, v = make_qkv(2, 2, 37, 16, seed=11)
        _, _, p = orc.attn_probs(q, k, v, causal, 0.25)
        _close(p.sum(axis=-1), 1.0, TIGHT, f"sum_j p_ij (causal={causal})")
        assert np.all(p >= 0.0)
        if causal:
            upper = np.triu(np.ones((37, 37), dtype=bool), k=1)
            assert np.all(p[..., upper] == 0.0), "causal: a key after the query got weight"


def check_o_is_p_times_v(orc):
    q, k, v = make_qkv(1, 3, 29, 8, seed=12)
    for causal in (False, True):
        o, _, p = orc.attn_probs(q, k, v, causal, 0.3)
        _close(o, np.einsum("bhij,bhjd->bhid", p, bf16_bits_to_f64(v)), TIGHT, "O = P V")


# ---------------------------------------------------------- method's claim

def online_softmax_attention(q, k, v, causal, scale, block):
    """Independent numpy restatement of the tiled online-softmax forward.

    Keys are visited ``block`` at a time; each row keeps a running maximum m,
    a running sum l and an unnormalised accumulator, rescaled by exp(m_old -
    m_new) whenever the maximum grows.  Nothing from the oracle is reused.
    """
    Q, K, V = bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)
    B, H, N, D = Q.shape
    O = np.zeros_like(Q)
    LSE = np.zeros((B, H, N))
    rows = np.arange(N)[:, None]
    for b in range(B):
        for h in range(H):
            m = np.full(N, -np.inf)
            l = np.zeros(N)
            acc = np.zeros((N, D))
            for j0 in range(0, N, block):
                j1 = min(N, j0 + block)
                s = scale * (Q[b, h] @ K[b, h, j0:j1].T)
                if causal:
                    s = np.where(np.arange(j0, j1)[None, :] > rows, -np.inf, s)
                m_new = np.maximum(m, s.max(axis=1))
                alpha = np.exp(m - m_new)
                pt = np.exp(s - m_new[:, None])
                l = alpha * l + pt.sum(axis=1)
                acc = alpha[:, None] * acc + pt @ V[b, h, j0:j1]
                m = m_new
            O[b, h] = acc / l[:, None]
            LSE[b, h] = m + np.log(l)
    return O, LSE


def check_online_equals_two_pass(orc):
    cases = [
        (1, 2, 300, 64, False, 1.0, 128),
        (1, 2, 300, 64, True, 1.0, 128),
        (2, 1, 257, 128, True, 4.0, 64),
        (1, 1, 200, 128, False, 4.0, 37),
    ]
    for B, H, N, D, causal, qstd, block in cases:
        q, k, v = make_qkv(B, H, N, D, seed=21 + N, q_std=qstd)
        scale = float(np.float32(1.0 / math.sqrt(D)))
        o, lse = orc.attn_fwd(q, k, v, causal, scale)
        o2, lse2 = online_softmax_attention(q, k, v, causal, scale, block)
        _close(o, o2, TIGHT, f"O online vs two-pass {B,H,N,D,causal}")
        _close(lse, lse2, TIGHT, f"LSE online vs two-pass {B,H,N,D,causal}")


# ------------------------------------------------------------- closed forms

def check_identical_keys(orc):
    B, H, N, D = 1, 2, 40, 16
    q, k, v = make_qkv(B, H, N, D, seed=31)
    k = np.broadcast_to(k[:, :, :1, :], k.shape).copy()
    V = bf16_bits_to_f64(v)
    for causal in (False, True):
        scale = 0.125
        o, lse = orc.attn_fwd(q, k, v, causal, scale)
        n = _vis_counts(N, causal)
        mean_v = np.cumsum(V, axis=2) / np.arange(1, N + 1)[None, None, :, None] if causal else \
            np.broadcast_to(V.mean(axis=2, keepdims=True), V.shape)
        _close(o, mean_v, TIGHT, "identical keys: O = mean of visible V rows")
        c = scale * np.einsum("bhid,bhd->bhi", bf16_bits_to_f64(q), bf16_bits_to_f64(k[:, :, 0, :]))
        _close(lse, c + np.log(n)[None, None, :], TIGHT, "identical keys: LSE = s + ln n")


def check_zero_queries(orc):
    B, H, N, D = 2, 1, 33, 8
    _, k, v = make_qkv(B, H, N, D, seed=32)
    q = np.zeros_like(k)
    V = bf16_bits_to_f64(v)
    for causal in (False, True):
        o, lse = orc.attn_fwd(q, k, v, causal, 0.7)
        n = _vis_counts(N, causal)
        _close(lse, np.broadcast_to(np.log(n), lse.shape), TIGHT, "Q = 0: LSE = ln n")
        ref = np.cumsum(V, axis=2) / n[None, None, :, None] if causal else \
            np.broadcast_to(V.mean(axis=2, keepdims=True), V.shape)
        _close(o, ref, TIGHT, "Q = 0: O = mean of visible V rows")


def check_one_hot_dominant_logit(orc):
    B, H, N, D, t = 1, 1, 64, 64, 9
    _, _, v = make_qkv(B, H, N, D, seed=33)
    sixteen = f64_to_bf16_bits(np.array([16.0]))[0]
    q = np.zeros((B, H, N, D), dtype=np.uint16)
    k = np.zeros((B, H, N, D), dtype=np.uint16)
    q[..., 0] = sixteen
    k[0, 0, t, 0] = sixteen
    V = bf16_bits_to_f64(v)[0, 0]
    scale = 0.125  # s_it = 16 * 16 / 8 = 32, every other logit 0
    big = math.exp(32.0)
    for causal in (False, True):
        o, lse = orc.attn_fwd(q, k, v, causal, scale)
        for i in range(N):
            n = i + 1 if causal else N
            if causal and i < t:
                ref_o = V[: i + 1].mean(axis=0)
                ref_l = math.log(i + 1)
            else:
                rest = V[:n].sum(axis=0) - V[t]
                ref_o = (big * V[t] + rest) / (big + (n - 1))
                ref_l = 32.0 + math.log1p((n - 1) * math.exp(-32.0))
            _close(o[0, 0, i], ref_o, TIGHT, f"one-hot row {i}: O")
            _close(lse[0, 0, i], ref_l, TIGHT, f"one-hot row {i}: LSE")
            if n > 1 and (not causal or i >= t):
                _close(o[0, 0, i], V[t], 1e-11 * max(1.0, np.abs(V).max()), "one-hot selects V_t")


def check_causal_first_row(orc):
    q, k, v = make_qkv(2, 3, 50, 32, seed=34)
    scale = 0.2
    o, lse = orc.attn_fwd(q, k, v, True, scale)
    V = bf16_bits_to_f64(v)
    assert np.array_equal(o[:, :, 0, :], V[:, :, 0, :]), "causal row 0 must copy V_0 exactly"
    s00 = scale * np.einsum("bhd,bhd->bh", bf16_bits_to_f64(q)[:, :, 0], bf16_bits_to_f64(k)[:, :, 0])
    _close(lse[:, :, 0], s00, TIGHT, "causal row 0: LSE = s_00")


def check_logit_shift(orc):
    B, H, N, D = 1, 2, 70, 32
    q, k, v = make_qkv(B, H, N, D, seed=35)
    k0 = k.copy()
    k0[..., D - 1] = 0
    k8 = k.copy()
    k8[..., D - 1] = f64_to_bf16_bits(np.array([8.0]))[0]
    scale = 0.25
    for causal in (False, True):
        o0, l0 = orc.attn_fwd(q, k0, v, causal, scale)
        o8, l8 = orc.attn_fwd(q, k8, v, causal, scale)
        shift = scale * bf16_bits_to_f64(q)[..., D - 1] * 8.0
        _close(o8, o0, TIGHT, "common logit shift leaves O unchanged")
        _close(l8 - l0, shift, TIGHT, "common logit shift moves LSE by the shift")


# --------------------------------------------------------------- invariants

def check_key_permutation(orc):
    q, k, v = make_qkv(1, 2, 90, 16, seed=36)
    perm = np.random.default_rng(5).permutation(90)
    o, lse = orc.attn_fwd(q, k, v, False, 0.25)
    o2, lse2 = orc.attn_fwd(q, k[:, :, perm], v[:, :, perm], False, 0.25)
    _close(o2, o, TIGHT, "key/value permutation: O")
    _close(lse2, lse, TIGHT, "key/value permutation: LSE")


def check_bh_independence(orc):
    q, k, v = make_qkv(2, 3, 24, 8, seed=37)
    for causal in (False, True):
        o, lse = orc.attn_fwd(q, k, v, causal, 0.35)
        for b in range(2):
            for h in range(3):
                sl = (slice(b, b + 1), slice(h, h + 1))
                o1, l1 = orc.attn_fwd(q[sl], k[sl], v[sl], causal, 0.35)
                assert np.array_equal(o1[0, 0], o[b, h]) and np.array_equal(l1[0, 0], lse[b, h]), \
                    f"slice ({b},{h}) differs from its stand-alone run"


def check_rows_match_full(orc):
    q, k, v = make_qkv(2, 2, 130, 64, seed=38)
    for causal in (False, True):
        o, lse = orc.attn_fwd(q, k, v, causal, 0.125)
        bh = np.array([0, 3, 1, 2, 3], dtype=np.int64)
        ri = np.array([0, 129, 64, 127, 1], dtype=np.int64)
        o_r, l_r = orc.attn_rows(q, k, v, causal, 0.125, bh, ri)
        of, lf = o.reshape(4, 130, 64), lse.reshape(4, 130)
        assert np.array_equal(o_r, of[bh, ri]) and np.array_equal(l_r, lf[bh, ri])


# ------------------------------------------------------- library / brute force

def check_matches_torch_sdpa(orc):
    import torch

    for (B, H, N, D, causal, qstd) in [(2, 3, 65, 32, False, 1.0), (1, 2, 100, 64, True, 4.0),
                                        (1, 1, 7, 128, True, 1.0)]:
        q, k, v = make_qkv(B, H, N, D, seed=40 + N, q_std=qstd)
        scale = float(np.float32(1.0 / math.sqrt(D)))
        o, lse = orc.attn_fwd(q, k, v, causal, scale)
        Q, K, V = (torch.from_numpy(bf16_bits_to_f64(x)) for x in (q, k, v))
        with torch.no_grad():
            o_t = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=causal, scale=scale)
            s = scale * (Q @ K.transpose(-1, -2))
            if causal:
                s = s.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
            lse_t = torch.logsumexp(s, dim=-1)
        _close(o, o_t.numpy(), TIGHT, "O vs torch SDPA (fp64)")
        _close(lse, lse_t.numpy(), TIGHT, "LSE vs torch logsumexp (fp64)")


def decimal_attention(q, k, v, causal, scale, digits=50):
    """50-digit brute force of the definition, for tiny inputs."""
    ctx = decimal.Context(prec=digits)
    Dec = decimal.Decimal
    Q, K, V = bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v)
    B, H, N, D = Q.shape
    Nk = K.shape[2]
    sc = Dec(float(scale))
    O = np.zeros((B, H, N, D))
    LSE = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                n = max(0, min(Nk, i + 1 + Nk - N)) if causal else Nk
                if n == 0:
                    LSE[b, h, i] = -np.inf
                    continue
                s = []
                for j in range(n):
                    acc = Dec(0)
                    for d in range(D):
                        acc = ctx.add(acc, ctx.multiply(Dec(float(Q[b, h, i, d])), Dec(float(K[b, h, j, d]))))
                    s.append(ctx.multiply(sc, acc))
                e = [ctx.exp(x) for x in s]
                z = Dec(0)
                for x in e:
                    z = ctx.add(z, x)
                for d in range(D):
                    acc = Dec(0)
                    for j in range(n):
                        acc = ctx.add(acc, ctx.multiply(e[j], Dec(float(V[b, h, j, d]))))
                    O[b, h, i, d] = float(ctx.divide(acc, z))
                LSE[b, h, i] = float(ctx.ln(z))
    return O, LSE


def check_decimal_brute_force(orc):
    for (B, H, N, D, causal, qstd, seed) in [(1, 2, 8, 4, False, 1.0, 51), (2, 1, 8, 4, True, 1.0, 52),
                                              (1, 1, 6, 3, False, 4.0, 53), (1, 1, 5, 2, True, 4.0, 54)]:
        q, k, v = make_qkv(B, H, N, D, seed=seed, q_std=qstd)
        scale = float(np.float32(1.0 / math.sqrt(D)))
        o, lse = orc.attn_fwd(q, k, v, causal, scale)
        o_d, lse_d = decimal_attention(q, k, v, causal, scale)
        _close(o, o_d, 1e-14, "O vs 50-digit brute force")
        _close(lse, lse_d, 1e-14, "LSE vs 50-digit brute force")


# ------------------------------------------------ queries and keys of different lengths

def check_causal_suffix_is_bottom_right(orc):
    """A causal query block that ends with the keys sees exactly what the same rows
    of the square causal problem see: rows N-Nq.. of causal(Q, K, V) equal
    causal(Q[N-Nq:], K, V).  This pins the bottom-right alignment on the square case."""
    B, H, N, D = 1, 2, 90, 16
    q, k, v = make_qkv(B, H, N, D, seed=61)
    o_sq, l_sq = orc.attn_fwd(q, k, v, True, 0.3)
    for nq in (1, 7, 37, 90):
        o_r, l_r = orc.attn_fwd(q[:, :, N - nq:], k, v, True, 0.3)
        assert np.array_equal(o_r, o_sq[:, :, N - nq:]) and np.array_equal(l_r, l_sq[:, :, N - nq:]), \
            f"causal Nq={nq}, Nk={N}: not the last rows of the square problem"


def check_full_rows_depend_on_their_query_only(orc):
    """Without the mask each query row is independent: any block of queries gives
    the same rows as the square problem that contains it."""
    B, H, N, D = 1, 2, 70, 8
    q, k, v = make_qkv(B, H, N, D, seed=62)
    o_sq, l_sq = orc.attn_fwd(q, k, v, False, 0.25)
    for a, b in ((0, 1), (5, 40), (69, 70)):
        o_r, l_r = orc.attn_fwd(q[:, :, a:b], k, v, False, 0.25)
        assert np.array_equal(o_r, o_sq[:, :, a:b]) and np.array_equal(l_r, l_sq[:, :, a:b])


def check_more_queries_than_keys_causal(orc):
    """Causal with Nq > Nk: the first Nq - Nk queries see no key (O = 0, LSE = -inf);
    the others are the square causal problem on the last Nk queries."""
    B, H, Nq, Nk, D = 1, 2, 50, 30, 8
    q, _, _ = make_qkv(B, H, Nq, D, seed=63)
    _, k, v = make_qkv(B, H, Nk, D, seed=64)
    o, lse = orc.attn_fwd(q, k, v, True, 0.4)
    assert np.all(o[:, :, : Nq - Nk] == 0.0) and np.all(np.isneginf(lse[:, :, : Nq - Nk]))
    o_sq, l_sq = orc.attn_fwd(q[:, :, Nq - Nk:], k, v, True, 0.4)
    assert np.array_equal(o[:, :, Nq - Nk:], o_sq) and np.array_equal(lse[:, :, Nq - Nk:], l_sq)


def check_rectangular_against_torch_mask(orc):
    import torch

    for (Nq, Nk, causal) in [(33, 100, True), (100, 33, False), (1, 77, True), (64, 64, True)]:
        B, H, D = 1, 2, 32
        q, _, _ = make_qkv(B, H, Nq, D, seed=70 + Nq)
        _, k, v = make_qkv(B, H, Nk, D, seed=71 + Nk)
        scale = float(np.float32(1.0 / math.sqrt(D)))
        o, lse = orc.attn_fwd(q, k, v, causal, scale)
        Q, K, V = (torch.from_numpy(bf16_bits_to_f64(x)) for x in (q, k, v))
        visible = torch.ones(Nq, Nk, dtype=torch.bool)
        if causal:
            visible = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
        with torch.no_grad():
            o_t = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=visible, scale=scale)
            lse_t = torch.logsumexp((scale * (Q @ K.transpose(-1, -2))).masked_fill(~visible, float("-inf")), dim=-1)
        _close(o, o_t.numpy(), TIGHT, f"O vs torch SDPA with mask (Nq={Nq}, Nk={Nk})")
        _close(lse, lse_t.numpy(), TIGHT, f"LSE vs torch logsumexp (Nq={Nq}, Nk={Nk})")


def check_rectangular_decimal(orc):
    for (Nq, Nk, causal, seed) in [(3, 8, True, 81), (8, 3, False, 82), (6, 4, True, 83)]:
        q, _, _ = make_qkv(1, 1, Nq, 4, seed=seed)
        _, k, v = make_qkv(1, 1, Nk, 4, seed=seed + 100)
        o, lse = orc.attn_fwd(q, k, v, causal, 0.5)
        o_d, lse_d = decimal_attention(q, k, v, causal, 0.5)
        fin = np.isfinite(lse_d)
        _close(o, o_d, 1e-14, f"O vs 50-digit brute force (Nq={Nq}, Nk={Nk})")
        assert np.array_equal(np.isfinite(lse), fin)
        _close(lse[fin], lse_d[fin], 1e-14, f"LSE vs 50-digit brute force (Nq={Nq}, Nk={Nk})")


ALL_CHECKS = [
    check_prob_rows_sum_to_one,
    check_o_is_p_times_v,
    check_online_equals_two_pass,
    check_identical_keys,
    check_zero_queries,
    check_one_hot_dominant_logit,
    check_causal_first_row,
    check_logit_shift,
    check_key_permutation,
    check_bh_independence,
    check_rows_match_full,
    check_matches_torch_sdpa,
    check_decimal_brute_force,
    check_causal_suffix_is_bottom_right,
    check_full_rows_depend_on_their_query_only,
    check_more_queries_than_keys_causal,
    check_rectangular_against_torch_mask,
    check_rectangular_decimal,
]
