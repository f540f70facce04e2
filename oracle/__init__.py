"""CPU oracles for the attention forward and the Based linear-attention forward
-- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls it, and it shares no code
with that path: its arithmetic lives in ``attn_oracle.c``, ``attn_oracle_bwd.c``
and ``based_oracle.c`` (plain C, fp64), built with gcc into
``oracle/lib/liboracle_attn.so``.

Every function takes Q as ``uint16`` bf16 bit patterns shaped [B, H, Nq, D] and
K, V shaped [B, H, Nk, D] (Nk = Nq for self-attention; the layout of the C
ABI) and returns float64 results.  Causal masking is aligned at the
bottom-right corner: key j is visible to query i iff j <= i + Nk - Nq.

Pins for every function here live in ``tests/oracle_pins.py``,
``tests/oracle_bwd_pins.py`` and ``tests/oracle_based_pins.py`` (closed forms,
invariants, independent restatements -- the tiled online softmax, the linear
attention recurrence over an explicit Taylor feature map -- a library routine
and exact or 50-digit brute force).  The one part left unpinned is the GPU's
own fp32/bf16 rounding, which nothing fixes beyond the stated tolerances.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attn_oracle.c")
SOURCE_BWD = os.path.join(_HERE, "attn_oracle_bwd.c")
SOURCE_BASED = os.path.join(_HERE, "based_oracle.c")
SOURCES = [SOURCE, SOURCE_BWD, SOURCE_BASED]
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "liboracle_attn.so")
_lock = threading.Lock()
_default = None


def compile_source(src, out: str) -> str:
    """gcc the C oracle source(s) ``src`` into the shared library ``out`` (OpenMP when available)."""
    srcs = [src] if isinstance(src, str) else list(src)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, *srcs, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build ``oracle/lib/liboracle_attn.so`` if it is missing or stale; returns its path."""
    if not force and os.path.exists(_LIB) and all(os.path.getmtime(_LIB) >= os.path.getmtime(f) for f in SOURCES):
        return _LIB
    return compile_source(SOURCES, _LIB)


def _bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16 or a.ndim != 4:
        raise TypeError("expected uint16 bf16 bit patterns shaped [B, H, N, D]")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one compiled copy of ``attn_oracle.c``."""

    def __init__(self, libpath: str):
        lib = ctypes.CDLL(libpath)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_attn_fwd_qk.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64, I, ctypes.c_double, I]
        lib.oracle_attn_rows_qk.argtypes = [P, P, P, I64, I64, I64, I64, I, ctypes.c_double, P, P, I64, P, P, I]
        lib.oracle_attn_probs_qk.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I64, I, ctypes.c_double]
        lib.oracle_threads.argtypes = [I]
        for f in (lib.oracle_attn_fwd_qk, lib.oracle_attn_rows_qk, lib.oracle_attn_probs_qk, lib.oracle_threads):
            f.restype = I
        self.has_bwd = hasattr(lib, "oracle_attn_bwd")
        if self.has_bwd:
            args = [P] * 10 + [I64, I64, I64, I64, I64, I, ctypes.c_double, I]
            lib.oracle_attn_bwd.argtypes = args
            lib.oracle_attn_bwd_f64.argtypes = args
            lib.oracle_attn_bwd.restype = I
            lib.oracle_attn_bwd_f64.restype = I
            lib.oracle_attn_bwd_rows.argtypes = [P, P, P, P, I64, I64, I64, I64, I, ctypes.c_double, P, P, I64, P,
                                                 P, I]
            lib.oracle_attn_bwd_keys.argtypes = [P, P, P, P, I64, I64, I64, I64, I, ctypes.c_double, I64, P, I64,
                                                 P, P, I]
            lib.oracle_attn_bwd_rows.restype = I
            lib.oracle_attn_bwd_keys.restype = I
        self.has_based = hasattr(lib, "oracle_based_fwd")
        if self.has_based:
            lib.oracle_based_fwd.argtypes = [P, P, P, P, P, I64, I64, I64, I64, ctypes.c_double, I]
            lib.oracle_based_rows.argtypes = [P, P, P, I64, I64, I64, I64, ctypes.c_double, P, P, I64, P, P, I]
            lib.oracle_based_fwd.restype = I
            lib.oracle_based_rows.restype = I
        self._lib = lib
        self.path = libpath

    @staticmethod
    def _based_shapes(q, k, v):
        if not (q.shape == k.shape and q.shape[:3] == v.shape[:3]):
            raise ValueError("q, k [B,H,N,F] and v [B,H,N,D] expected")
        B, H, N, F = q.shape
        return B, H, N, F, v.shape[3]

    def based_fwd(self, q, k, v, scale: float, nthreads: int = 0):
        """Based linear attention (causal, second-order Taylor kernel) by its plain
        definition: (Y [B,H,N,D] float64, Z [B,H,N] float64)."""
        q, k, v = _bits(q), _bits(k), _bits(v)
        B, H, N, F, D = self._based_shapes(q, k, v)
        y = np.empty((B, H, N, D), dtype=np.float64)
        z = np.empty((B, H, N), dtype=np.float64)
        rc = self._lib.oracle_based_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(z), B * H, N, F, D, float(scale),
                                        int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_based_fwd failed")
        return y, z

    def based_rows(self, q, k, v, scale: float, bh_idx, row_idx, nthreads: int = 0):
        """Y and Z for the rows (bh_idx[r], row_idx[r]) only: shapes [R, D] and [R]."""
        q, k, v = _bits(q), _bits(k), _bits(v)
        B, H, N, F, D = self._based_shapes(q, k, v)
        bh = np.ascontiguousarray(bh_idx, dtype=np.int64)
        ri = np.ascontiguousarray(row_idx, dtype=np.int64)
        if bh.shape != ri.shape or bh.ndim != 1:
            raise ValueError("bh_idx and row_idx must be 1-D and of one length")
        y = np.empty((bh.shape[0], D), dtype=np.float64)
        z = np.empty((bh.shape[0],), dtype=np.float64)
        rc = self._lib.oracle_based_rows(_ptr(q), _ptr(k), _ptr(v), B * H, N, F, D, float(scale), _ptr(bh), _ptr(ri),
                                         bh.shape[0], _ptr(y), _ptr(z), int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_based_rows failed (bad index?)")
        return y, z

    def threads(self, nthreads: int = 0) -> int:
        """OpenMP threads a call with ``nthreads`` uses (0 means all available)."""
        return self._lib.oracle_threads(nthreads)

    @staticmethod
    def _shapes(q, k, v):
        if not (k.shape == v.shape and q.shape[:2] == k.shape[:2] and q.shape[3] == k.shape[3]):
            raise ValueError("q [B,H,Nq,D], k and v [B,H,Nk,D] expected")
        B, H, Nq, D = q.shape
        return B, H, Nq, k.shape[2], D

    def attn_fwd(self, q, k, v, causal: bool, scale: float, nthreads: int = 0):
        """(O [B,H,Nq,D] float64, LSE [B,H,Nq] float64) by the two-pass definition."""
        q, k, v = _bits(q), _bits(k), _bits(v)
        B, H, Nq, Nk, D = self._shapes(q, k, v)
        o = np.empty((B, H, Nq, D), dtype=np.float64)
        lse = np.empty((B, H, Nq), dtype=np.float64)
        rc = self._lib.oracle_attn_fwd_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, D,
                                          int(bool(causal)), float(scale), int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_attn_fwd failed")
        return o, lse

    def attn_rows(self, q, k, v, causal: bool, scale: float, bh_idx, row_idx, nthreads: int = 0):
        """O and LSE for the rows (bh_idx[r], row_idx[r]) only: shapes [R, D] and [R]."""
        q, k, v = _bits(q), _bits(k), _bits(v)
        B, H, Nq, Nk, D = self._shapes(q, k, v)
        bh = np.ascontiguousarray(bh_idx, dtype=np.int64)
        ri = np.ascontiguousarray(row_idx, dtype=np.int64)
        if bh.shape != ri.shape or bh.ndim != 1:
            raise ValueError("bh_idx and row_idx must be 1-D and of one length")
        R = bh.shape[0]
        o = np.empty((R, D), dtype=np.float64)
        lse = np.empty((R,), dtype=np.float64)
        rc = self._lib.oracle_attn_rows_qk(_ptr(q), _ptr(k), _ptr(v), B * H, Nq, Nk, D, int(bool(causal)),
                                        float(scale), _ptr(bh), _ptr(ri), R, _ptr(o), _ptr(lse),
                                        int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_attn_rows failed (bad index?)")
        return o, lse

    def attn_probs(self, q, k, v, causal: bool, scale: float):
        """(O, LSE, P [B,H,Nq,Nk]) for small problems; P is the softmax matrix."""
        q, k, v = _bits(q), _bits(k), _bits(v)
        B, H, Nq, Nk, D = self._shapes(q, k, v)
        o = np.empty((B, H, Nq, D), dtype=np.float64)
        lse = np.empty((B, H, Nq), dtype=np.float64)
        p = np.empty((B, H, Nq, Nk), dtype=np.float64)
        rc = self._lib.oracle_attn_probs_qk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(p),
                                            B, H, Nq, Nk, D, int(bool(causal)), float(scale))
        if rc != 0:
            raise RuntimeError("oracle_attn_probs failed")
        return o, lse, p


def _bwd_call(fn, q, k, v, do, causal, scale, nthreads):
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if not (k.shape == v.shape and q.shape == do.shape and q.shape[:2] == k.shape[:2] and k.shape[3] == D):
        raise ValueError("q, do [B,H,Nq,D] and k, v [B,H,Nk,D] expected")
    out = {n: np.empty(sh, dtype=np.float64) for n, sh in
           (("dq", q.shape), ("dk", k.shape), ("dv", k.shape), ("delta", (B, H, Nq)), ("o", q.shape), ("lse", (B, H, Nq)))}
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]),
            _ptr(out["delta"]), _ptr(out["o"]), _ptr(out["lse"]), B, H, Nq, Nk, D, int(bool(causal)), float(scale),
            int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle backward failed")
    return out


def _bwd_methods(cls):
    def attn_bwd(self, q, k, v, do, causal: bool, scale: float, nthreads: int = 0):
        """Gradients of sum(dO * O) from bf16 bit inputs: dict dq, dk, dv, delta, o, lse (float64)."""
        q, k, v, do = _bits(q), _bits(k), _bits(v), _bits(do)
        return _bwd_call(self._lib.oracle_attn_bwd, q, k, v, do, causal, scale, nthreads)

    def attn_bwd_f64(self, q, k, v, do, causal: bool, scale: float, nthreads: int = 0):
        """Same from float64 inputs (for finite-difference checks)."""
        arr = [np.ascontiguousarray(x, dtype=np.float64) for x in (q, k, v, do)]
        return _bwd_call(self._lib.oracle_attn_bwd_f64, *arr, causal, scale, nthreads)

    def attn_bwd_rows(self, q, k, v, do, causal: bool, scale: float, bh_idx, row_idx, nthreads: int = 0):
        """dQ rows [R, D] and D [R] for the query rows (bh_idx[r], row_idx[r]) only."""
        q, k, v, do = _bits(q), _bits(k), _bits(v), _bits(do)
        B, H, Nq, Nk, D = self._shapes(q, k, v)
        bh = np.ascontiguousarray(bh_idx, dtype=np.int64)
        ri = np.ascontiguousarray(row_idx, dtype=np.int64)
        if bh.shape != ri.shape or bh.ndim != 1 or do.shape != q.shape:
            raise ValueError("bh_idx, row_idx 1-D of one length; do shaped like q")
        dq = np.empty((bh.shape[0], D), dtype=np.float64)
        delta = np.empty((bh.shape[0],), dtype=np.float64)
        rc = self._lib.oracle_attn_bwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B * H, Nq, Nk, D,
                                            int(bool(causal)), float(scale), _ptr(bh), _ptr(ri), bh.shape[0],
                                            _ptr(dq), _ptr(delta), int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_attn_bwd_rows failed (bad index?)")
        return dq, delta

    def attn_bwd_keys(self, q, k, v, do, causal: bool, scale: float, bh: int, key_idx, nthreads: int = 0):
        """dK and dV rows [R, D] for the keys key_idx[r] of slice bh (b * H + h) only."""
        q, k, v, do = _bits(q), _bits(k), _bits(v), _bits(do)
        B, H, Nq, Nk, D = self._shapes(q, k, v)
        kj = np.ascontiguousarray(key_idx, dtype=np.int64)
        if kj.ndim != 1 or do.shape != q.shape:
            raise ValueError("key_idx 1-D; do shaped like q")
        dk = np.empty((kj.shape[0], D), dtype=np.float64)
        dv = np.empty((kj.shape[0], D), dtype=np.float64)
        rc = self._lib.oracle_attn_bwd_keys(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B * H, Nq, Nk, D,
                                            int(bool(causal)), float(scale), int(bh), _ptr(kj), kj.shape[0],
                                            _ptr(dk), _ptr(dv), int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_attn_bwd_keys failed (bad index?)")
        return dk, dv

    cls.attn_bwd = attn_bwd
    cls.attn_bwd_f64 = attn_bwd_f64
    cls.attn_bwd_rows = attn_bwd_rows
    cls.attn_bwd_keys = attn_bwd_keys
    return cls


_bwd_methods(Oracle)


def attn_bwd(q, k, v, do, causal: bool, scale: float, nthreads: int = 0):
    return default().attn_bwd(q, k, v, do, causal, scale, nthreads)


def attn_bwd_rows(q, k, v, do, causal: bool, scale: float, bh_idx, row_idx, nthreads: int = 0):
    return default().attn_bwd_rows(q, k, v, do, causal, scale, bh_idx, row_idx, nthreads)


def attn_bwd_keys(q, k, v, do, causal: bool, scale: float, bh: int, key_idx, nthreads: int = 0):
    return default().attn_bwd_keys(q, k, v, do, causal, scale, bh, key_idx, nthreads)


def default() -> Oracle:
    """The oracle built from ``attn_oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def threads(nthreads: int = 0) -> int:
    return default().threads(nthreads)


def attn_fwd(q, k, v, causal: bool, scale: float, nthreads: int = 0):
    return default().attn_fwd(q, k, v, causal, scale, nthreads)


def attn_rows(q, k, v, causal: bool, scale: float, bh_idx, row_idx, nthreads: int = 0):
    return default().attn_rows(q, k, v, causal, scale, bh_idx, row_idx, nthreads)


def attn_probs(q, k, v, causal: bool, scale: float):
    return default().attn_probs(q, k, v, causal, scale)


def based_fwd(q, k, v, scale: float, nthreads: int = 0):
    return default().based_fwd(q, k, v, scale, nthreads)


def based_rows(q, k, v, scale: float, bh_idx, row_idx, nthreads: int = 0):
    return default().based_rows(q, k, v, scale, bh_idx, row_idx, nthreads)
