"""GB300 (sm_103a) fused attention forward: O = softmax(scale * Q K^T [+causal]) V and LSE.

``attn_fwd`` and friends are the C ABI of include/attn.h under the same names;
``fwd`` is the convenience call on torch tensors.  PyTorch only provides device
memory and the stream; the arithmetic runs in the package's CUDA library.
"""
from __future__ import annotations

import math

from ._binding import (  # noqa: F401
    ATTN_ERR_CUDA,
    ATTN_ERR_INVALID_ARG,
    ATTN_ERR_TIMEOUT,
    ATTN_ERR_UNSUPPORTED,
    ATTN_OK,
    attn_based_fwd,
    attn_based_fwd_flops,
    attn_bwd,
    attn_bwd_ld,
    attn_bwd_qk,
    attn_bwd_qk_flops,
    attn_fwd,
    attn_fwd_flops,
    attn_fwd_from_host,
    attn_fwd_from_host_static,
    attn_fwd_kernel_name,
    attn_fwd_ld,
    attn_fwd_qk,
    attn_fwd_qk_flops,
    attn_last_status,
    attn_set_tuning,
    attn_status_string,
    library,
)


class AttnError(RuntimeError):
    def __init__(self, status: int):
        super().__init__(attn_status_string(status))
        self.status = status


def fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, stream=None):
    """Fused forward on contiguous bf16 CUDA tensors q [B, H, Nq, D], k, v [B, H, Nk, D].

    Returns ``(o, lse)``: o bf16 [B, H, Nq, D], lse fp32 [B, H, Nq].  With
    ``causal`` and Nq != Nk the mask is aligned at the bottom-right.  ``scale``
    defaults to 1/sqrt(D).  Runs on ``stream`` (default: torch's current
    stream) without synchronising.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [B, H, N, D]")
    if not (k.shape == v.shape and q.shape[:2] == k.shape[:2] and q.shape[3] == k.shape[3]):
        raise ValueError("q must be [B, H, Nq, D] and k, v [B, H, Nk, D]")
    B, H, N, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    if Nk == N:
        st = attn_fwd(q, k, v, out, lse, B, H, N, D, causal, scale, stream)
    else:
        st = attn_fwd_qk(q, k, v, out, lse, B, H, N, Nk, D, causal, scale, stream)
    if st != ATTN_OK:
        raise AttnError(st)
    return out, lse


def bwd(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, stream=None):
    """Backward of ``fwd``: returns ``(dq, dk, dv, delta)`` for contiguous bf16 CUDA tensors."""
    import torch

    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = attn_bwd_qk(q, k, v, o, lse, do, dq, dk, dv, delta, B, H, Nq, Nk, D, causal, scale, stream)
    if st != ATTN_OK:
        raise AttnError(st)
    return dq, dk, dv, delta


def fwd_from_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, device_buffers=None,
                  stream=None):
    """Forward for bf16 CPU tensors q [B, H, Nq, D], k, v [B, H, Nk, D] (pin them for overlapped copies).

    ``device_buffers`` = (q, k, v, o, lse) CUDA tensors of the same shapes (o like q,
    lse fp32 [B, H, Nq]) are the staging area; allocated on the current device when
    omitted.  Returns ``(out, lse)`` CPU tensors, filled once ``stream`` (default:
    torch's current stream) has been synchronised.  Keep q, k, v (and the device
    buffers) alive until then: the copies run asynchronously, and torch's
    pinned-memory cache may hand a freed block to another tensor at once.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CPU tensor [B, H, N, D]")
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    pin = q.is_pinned()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=pin)
    if device_buffers is None:
        dev = torch.device("cuda", torch.cuda.current_device())
        device_buffers = (torch.empty(q.shape, dtype=torch.bfloat16, device=dev),
                          torch.empty(k.shape, dtype=torch.bfloat16, device=dev),
                          torch.empty(v.shape, dtype=torch.bfloat16, device=dev),
                          torch.empty(q.shape, dtype=torch.bfloat16, device=dev),
                          torch.empty((B, H, Nq), dtype=torch.float32, device=dev))
    qd, kd, vd, od, ld = device_buffers
    if stream is None:
        stream = torch.cuda.current_stream(qd.device)
    st = attn_fwd_from_host(q, k, v, out, lse, qd, kd, vd, od, ld, B, H, Nq, Nk, D, causal, scale, stream)
    if st != ATTN_OK:
        raise AttnError(st)
    return out, lse


def based_fwd(q, k, v, scale: float | None = None, out=None, z=None, stream=None):
    """Based linear attention on contiguous bf16 CUDA tensors q, k [B, H, N, F], v [B, H, N, D].

    Returns ``(y, z)``: y bf16 [B, H, N, D], z fp32 [B, H, N] (the normaliser).
    ``scale`` defaults to 1/sqrt(F).  Runs on ``stream`` (default: torch's
    current stream) without synchronising.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if not (q.shape == k.shape and q.shape[:3] == v.shape[:3]):
        raise ValueError("q, k must be [B, H, N, F] and v [B, H, N, D]")
    B, H, N, F = q.shape
    D = v.shape[3]
    if scale is None:
        scale = 1.0 / math.sqrt(F)
    if out is None:
        out = torch.empty_like(v)
    if z is None:
        z = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    st = attn_based_fwd(q, k, v, out, z, B, H, N, F, D, scale, stream)
    if st != ATTN_OK:
        raise AttnError(st)
    return out, z
