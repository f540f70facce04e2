"""ctypes binding of the C ABI in include/attn.h -- argument marshalling only.

Every step of the forward runs in the CUDA library; if the library is missing
this module raises instead of computing anything another way.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4

_lock = threading.Lock()
_lib = None


def load(path: str) -> ctypes.CDLL:
    """Load a build of the library at ``path`` and declare its C signatures."""
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    sigs = {
        "attn_fwd": ([P, P, P, P, P, I64, I64, I64, I64, I, ctypes.c_float, P], I),
        "attn_last_status": ([P], I),
        "attn_status_string": ([I], ctypes.c_char_p),
        "attn_set_tuning": ([I, I, I, I64], I),
        "attn_fwd_flops": ([I64, I64, I64, I64, I], ctypes.c_double),
        "attn_fwd_qk": ([P, P, P, P, P, I64, I64, I64, I64, I64, I, ctypes.c_float, P], I),
        "attn_fwd_qk_flops": ([I64, I64, I64, I64, I64, I], ctypes.c_double),
        "attn_bwd": ([P] * 10 + [I64, I64, I64, I64, I, ctypes.c_float, P], I),
        "attn_bwd_qk": ([P] * 10 + [I64, I64, I64, I64, I64, I, ctypes.c_float, P], I),
        "attn_bwd_qk_flops": ([I64, I64, I64, I64, I64, I], ctypes.c_double),
        "attn_fwd_from_host": ([P] * 10 + [I64, I64, I64, I64, I64, I, ctypes.c_float, P], I),
        "attn_fwd_from_host_static": ([P] * 5 + [I64, I64, I64, I64, I64, I, ctypes.c_float, P], I),
        "attn_fwd_kernel_name": ([I64, I64, I64, I64, I64, I], ctypes.c_char_p),
        "attn_fwd_ld": ([P, P, P, P, P, I64, I64, I64, I64, I64, I64, I, ctypes.c_float, P], I),
        "attn_bwd_ld": ([P] * 10 + [I64, I64, I64, I64, I64, I64, I, ctypes.c_float, P], I),
        "attn_based_fwd": ([P, P, P, P, P, I64, I64, I64, I64, I64, ctypes.c_float, P], I),
        "attn_based_fwd_flops": ([I64, I64, I64, I64, I64], ctypes.c_double),
        "attn_test_withhold_kv": ([I], I),  # test build only
    }
    for name, (args, res) in sigs.items():
        if hasattr(lib, name):
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
    return lib


def library() -> ctypes.CDLL:
    """The loaded production CUDA library (built by ``build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = load(LIB)
    return _lib


def _addr(x) -> int | None:
    """A device/host address from a torch tensor, an int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def attn_fwd(q, k, v, o, lse, B: int, H: int, N: int, D: int, causal: bool, scale: float, stream) -> int:
    """Call ``attn_fwd``; tensors or raw addresses; ``stream`` a handle int or a torch stream."""
    s = stream if (stream is None or isinstance(stream, int)) else stream.cuda_stream
    return library().attn_fwd(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H), int(N),
                              int(D), int(bool(causal)), float(scale), s)


def attn_last_status(stream) -> int:
    s = stream if (stream is None or isinstance(stream, int)) else stream.cuda_stream
    return library().attn_last_status(s)


def attn_status_string(status: int) -> str:
    return library().attn_status_string(int(status)).decode()


def attn_set_tuning(unit: int = 0, grid: int = 0, pipe_chunks: int = 0, wait_limit_cycles: int = 0) -> int:
    """Call ``attn_set_tuning`` (process-wide overrides; all zero = automatic)."""
    return library().attn_set_tuning(int(unit), int(grid), int(pipe_chunks), int(wait_limit_cycles))


def attn_fwd_flops(B: int, H: int, N: int, D: int, causal: bool) -> float:
    return library().attn_fwd_flops(int(B), int(H), int(N), int(D), int(bool(causal)))


def attn_fwd_qk(q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int, D: int, causal: bool, scale: float,
                stream) -> int:
    """Call ``attn_fwd_qk`` (queries and keys of different lengths, bottom-right causal)."""
    s = stream if (stream is None or isinstance(stream, int)) else stream.cuda_stream
    return library().attn_fwd_qk(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), int(B), int(H), int(Nq),
                                 int(Nk), int(D), int(bool(causal)), float(scale), s)


def attn_fwd_qk_flops(B: int, H: int, Nq: int, Nk: int, D: int, causal: bool) -> float:
    return library().attn_fwd_qk_flops(int(B), int(H), int(Nq), int(Nk), int(D), int(bool(causal)))


def _stream(stream):
    return stream if (stream is None or isinstance(stream, int)) else stream.cuda_stream


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, delta, B: int, H: int, N: int, D: int, causal: bool,
             scale: float, stream) -> int:
    """Call ``attn_bwd`` (gradients of sum(dO * O) for the square forward)."""
    a = [_addr(x) for x in (q, k, v, o, lse, dout, dq, dk, dv, delta)]
    return library().attn_bwd(*a, int(B), int(H), int(N), int(D), int(bool(causal)), float(scale), _stream(stream))


def attn_bwd_qk(q, k, v, o, lse, dout, dq, dk, dv, delta, B: int, H: int, Nq: int, Nk: int, D: int, causal: bool,
                scale: float, stream) -> int:
    """Call ``attn_bwd_qk`` (queries and keys of different lengths)."""
    a = [_addr(x) for x in (q, k, v, o, lse, dout, dq, dk, dv, delta)]
    return library().attn_bwd_qk(*a, int(B), int(H), int(Nq), int(Nk), int(D), int(bool(causal)), float(scale),
                                 _stream(stream))


def attn_bwd_qk_flops(B: int, H: int, Nq: int, Nk: int, D: int, causal: bool) -> float:
    return library().attn_bwd_qk_flops(int(B), int(H), int(Nq), int(Nk), int(D), int(bool(causal)))


def attn_fwd_from_host(q_host, k_host, v_host, o_host, lse_host, q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int,
                       D: int, causal: bool, scale: float, stream) -> int:
    """Call ``attn_fwd_from_host`` (host inputs and outputs, copies overlapped with the kernels)."""
    a = [_addr(x) for x in (q_host, k_host, v_host, o_host, lse_host, q, k, v, o, lse)]
    return library().attn_fwd_from_host(*a, int(B), int(H), int(Nq), int(Nk), int(D), int(bool(causal)),
                                        float(scale), _stream(stream))


def attn_fwd_from_host_static(q_host, k_host, v_host, o_host, lse_host, B: int, H: int, Nq: int, Nk: int, D: int,
                              causal: bool, scale: float, stream) -> int:
    """Call ``attn_fwd_from_host_static`` (host inputs and outputs staged through the library's fixed device array)."""
    a = [_addr(x) for x in (q_host, k_host, v_host, o_host, lse_host)]
    return library().attn_fwd_from_host_static(*a, int(B), int(H), int(Nq), int(Nk), int(D), int(bool(causal)),
                                               float(scale), _stream(stream))


def attn_fwd_kernel_name(B: int, H: int, Nq: int, Nk: int, D: int, causal: bool):
    """The kernel instance ``attn_fwd_qk`` would launch for these sizes (None if it would reject them)."""
    name = library().attn_fwd_kernel_name(int(B), int(H), int(Nq), int(Nk), int(D), int(bool(causal)))
    return None if name is None else name.decode()


def attn_based_fwd(q, k, v, y, z, B: int, H: int, N: int, F: int, D: int, scale: float, stream) -> int:
    """Call ``attn_based_fwd`` (Based linear attention; tensors or raw addresses)."""
    a = [_addr(x) for x in (q, k, v, y, z)]
    return library().attn_based_fwd(*a, int(B), int(H), int(N), int(F), int(D), float(scale), _stream(stream))


def attn_based_fwd_flops(B: int, H: int, N: int, F: int, D: int) -> float:
    return library().attn_based_fwd_flops(int(B), int(H), int(N), int(F), int(D))


def attn_fwd_ld(q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int, D: int, ld: int, causal: bool, scale: float,
                stream) -> int:
    """Call ``attn_fwd_ld`` (rows ``ld`` elements apart; any head dim up to 256)."""
    a = [_addr(x) for x in (q, k, v, o, lse)]
    return library().attn_fwd_ld(*a, int(B), int(H), int(Nq), int(Nk), int(D), int(ld), int(bool(causal)),
                                 float(scale), _stream(stream))


def attn_bwd_ld(q, k, v, o, lse, dout, dq, dk, dv, delta, B: int, H: int, Nq: int, Nk: int, D: int, ld: int,
                causal: bool, scale: float, stream) -> int:
    """Call ``attn_bwd_ld`` (rows ``ld`` elements apart; any head dim up to 128)."""
    a = [_addr(x) for x in (q, k, v, o, lse, dout, dq, dk, dv, delta)]
    return library().attn_bwd_ld(*a, int(B), int(H), int(Nq), int(Nk), int(D), int(ld), int(bool(causal)),
                                 float(scale), _stream(stream))
