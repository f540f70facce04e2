"""Seeded synthetic inputs for the attention forward.

This module only draws numbers: it holds none of the attention arithmetic.  The
tests, the bench and the CPU oracle's callers all take their Q, K and V from
here, so both sides of every parity check see the same bf16 bytes.

Generator (defined here so it is identical on x86-64 and aarch64):

* raw 64-bit words come from numpy's Philox-4x64 counter-based bit generator,
  keyed by ``(seed, stream)``; its output is pure integer arithmetic;
* word ``w`` becomes a uniform ``u = ((w >> 11) + 0.5) * 2**-53`` in (0, 1);
* consecutive uniform pairs ``(u1, u2)`` become two standard normals by the
  Box-Muller transform ``sqrt(-2 ln u1) * (cos 2 pi u2, sin 2 pi u2)``;
* each normal is multiplied by ``std``, rounded to fp32 (nearest-even), then to
  bf16 (nearest-even on the fp32 bits).

Streams: Q = 0, K = 1, V = 2.  Arrays come back as ``uint16`` bf16 bit patterns
in [B, H, N, D] row-major order (D innermost), the layout of the C ABI.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

STREAM_Q, STREAM_K, STREAM_V = 0, 1, 2


def normal_bf16_bits(n: int, seed: int, stream: int, std: float = 1.0) -> np.ndarray:
    """``n`` bf16 bit patterns of N(0, std^2) draws (see the module docstring)."""
    if n == 0:
        return np.zeros(0, dtype=np.uint16)
    m = n + (n & 1)
    bg = np.random.Philox(key=np.array([seed, stream], dtype=np.uint64))
    raw = bg.random_raw(m)
    u = ((raw >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = (2.0 * np.pi) * u2
    z = np.empty(m, dtype=np.float64)
    z[0::2] = r * np.cos(t)
    z[1::2] = r * np.sin(t)
    f = (z[:n] * std).astype(np.float32).view(np.uint32)
    return ((f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64 (bf16 is the top half of fp32)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (nearest-even) -> bf16 (nearest-even) bit patterns; used to build exact test tensors."""
    f = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)
    return ((f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def make_qkv(B: int, H: int, N: int, D: int, seed: int, q_std: float = 1.0):
    """Q, K, V as bf16 bit arrays of shape [B, H, N, D]; Q ~ N(0, q_std^2), K, V ~ N(0, 1)."""
    shape = (B, H, N, D)
    n = B * H * N * D
    q = normal_bf16_bits(n, seed, STREAM_Q, q_std).reshape(shape)
    k = normal_bf16_bits(n, seed, STREAM_K, 1.0).reshape(shape)
    v = normal_bf16_bits(n, seed, STREAM_V, 1.0).reshape(shape)
    return q, k, v


@dataclass(frozen=True)
class Workload:
    """One named problem: shapes, mask, seed and the spread of Q.

    N is the query length; Nk the key length (0 means Nk = N).
    """
    name: str
    B: int
    H: int
    N: int
    D: int
    causal: bool
    seed: int
    q_std: float = 1.0
    Nk: int = 0

    @property
    def n_keys(self) -> int:
        return self.Nk or self.N

    @property
    def scale(self) -> float:
        """The softmax scale 1/sqrt(D), as the fp32 value both sides use."""
        return float(np.float32(1.0 / np.sqrt(self.D)))

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs: 4*B*H*D times the visible (query, key) pairs:
        N*Nk, or N*(Nk-N) + N^2/2 with the (bottom-right) causal mask -- for
        N = Nk, 4*B*H*N^2*D halved when causal."""
        nq, nk = float(self.N), float(self.n_keys)
        pairs = nq * (nk - nq) + 0.5 * nq * nq if self.causal else nq * nk
        return 4.0 * self.B * self.H * pairs * self.D

    def qkv(self):
        if self.n_keys == self.N:
            return make_qkv(self.B, self.H, self.N, self.D, self.seed, self.q_std)
        shape_q = (self.B, self.H, self.N, self.D)
        shape_kv = (self.B, self.H, self.n_keys, self.D)
        q = normal_bf16_bits(self.B * self.H * self.N * self.D, self.seed, STREAM_Q, self.q_std).reshape(shape_q)
        k = normal_bf16_bits(self.B * self.H * self.n_keys * self.D, self.seed, STREAM_K, 1.0).reshape(shape_kv)
        v = normal_bf16_bits(self.B * self.H * self.n_keys * self.D, self.seed, STREAM_V, 1.0).reshape(shape_kv)
        return q, k, v


# The problem sizes the method is measured on: a tiny case, a short-sequence case
# with and without the causal mask, a long-sequence throughput case, a very long
# causal case whose queries are spread 4x wider (large logits), and a many-head
# short-sequence causal case.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("b1h1n256d64", 1, 1, 256, 64, False, 1001),
        Workload("b2h8n1024d64", 2, 8, 1024, 64, False, 1002),
        Workload("b2h8n1024d64_causal", 2, 8, 1024, 64, True, 1002),
        Workload("b4h16n4096d128", 4, 16, 4096, 128, False, 1003),
        Workload("b1h16n16384d128_causal_q4", 1, 16, 16384, 128, True, 1004, 4.0),
        Workload("b16h32n512d64_causal", 16, 32, 512, 64, True, 1005),
        # A block of 512 new queries against a key/value cache of 8192 positions
        # (causal, aligned at the end of the cache).
        Workload("b8h16nq512nk8192d128_causal", 8, 16, 512, 128, True, 1006, Nk=8192),
    ]
}


@dataclass(frozen=True)
class BasedWorkload:
    """One Based linear-attention problem: q, k [B, H, N, F], v [B, H, N, D], causal.

    F is the feature dimension of q and k (16 in Based) and D the value head
    dimension; scale = 1/sqrt(F).  Streams as for attention (Q = 0, K = 1, V = 2).
    """
    name: str
    B: int
    H: int
    N: int
    F: int
    D: int
    seed: int
    q_std: float = 1.0

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / np.sqrt(self.F)))

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.N

    def qkv(self):
        q = normal_bf16_bits(self.B * self.H * self.N * self.F, self.seed, STREAM_Q, self.q_std)
        k = normal_bf16_bits(self.B * self.H * self.N * self.F, self.seed, STREAM_K, 1.0)
        v = normal_bf16_bits(self.B * self.H * self.N * self.D, self.seed, STREAM_V, 1.0)
        return (q.reshape(self.B, self.H, self.N, self.F), k.reshape(self.B, self.H, self.N, self.F),
                v.reshape(self.B, self.H, self.N, self.D))


# Based problem sizes: feature dimension 16 and value head dimension 64 (the
# Based layer's shape); a small case with a ragged last chunk, and a long-
# sequence throughput case (B*H = 256 sequences of 4096 tokens).
BASED_WORKLOADS = {
    w.name: w
    for w in [
        BasedWorkload("based_b1h2n300f16d64", 1, 2, 300, 16, 64, 2001),
        BasedWorkload("based_b16h16n4096f16d64", 16, 16, 4096, 16, 64, 2002),
    ]
}
