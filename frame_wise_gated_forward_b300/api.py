"""Python entry points of the frame-wise GDN forward (thin wrappers over the C ABI).

    out, state = frame_forward(q, k, v, alpha, beta, state_in=None)
    out, state = frame_step(q, k, v, alpha, beta, state)      # one latent frame
    out, state = frame_forward_host(q, k, v, alpha, beta, state_in=None)  # host tensors

Shapes (see include/gdn.h): q, k bf16 [B, F, N, H, dk]; v bf16 [B, F, N, H, dv];
alpha fp32 [B, F, H]; beta fp32 [B, F, N, H]; state fp32 [B, H, dv, dk].
For frame_step drop the F axis.  Tensors must be contiguous CUDA tensors on
the current device; calls run on torch's current CUDA stream.
"""
from __future__ import annotations

import torch

from ._lib import GDNError, check, load


def _stream_handle(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _dev(t, name, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def frame_forward(q, k, v, alpha, beta, state_in=None, *, out=None, state_out=None, stream=None):
    """Whole-sequence forward.  Returns (out bf16 [B,F,N,H,dv], state_out fp32 [B,H,dv,dk])."""
    lib = load()
    B, F, N, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, F, N, H, dv), dtype=torch.bfloat16, device=q.device)
    if state_out is None:
        state_out = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    args = [
        _dev(q, "q", torch.bfloat16, (B, F, N, H, dk)),
        _dev(k, "k", torch.bfloat16, (B, F, N, H, dk)),
        _dev(v, "v", torch.bfloat16, (B, F, N, H, dv)),
        _dev(alpha, "alpha", torch.float32, (B, F, H)),
        _dev(beta, "beta", torch.float32, (B, F, N, H)),
        None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
        _dev(out, "out", torch.bfloat16, (B, F, N, H, dv)),
        _dev(state_out, "state_out", torch.float32, (B, H, dv, dk)),
    ]
    check(lib.gdn_frame_forward(*args, B, H, F, N, dk, dv, _stream_handle(stream)), "gdn_frame_forward")
    return out, state_out


def frame_step(q, k, v, alpha, beta, state_in=None, *, out=None, state_out=None, stream=None):
    """One latent frame on a resident state.  q, k [B,N,H,dk]; v [B,N,H,dv];
    alpha [B,H]; beta [B,N,H].  state_out may be the same tensor as state_in."""
    lib = load()
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=q.device)
    if state_out is None:
        state_out = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    args = [
        _dev(q, "q", torch.bfloat16, (B, N, H, dk)),
        _dev(k, "k", torch.bfloat16, (B, N, H, dk)),
        _dev(v, "v", torch.bfloat16, (B, N, H, dv)),
        _dev(alpha, "alpha", torch.float32, (B, H)),
        _dev(beta, "beta", torch.float32, (B, N, H)),
        None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
        _dev(out, "out", torch.bfloat16, (B, N, H, dv)),
        _dev(state_out, "state_out", torch.float32, (B, H, dv, dk)),
    ]
    check(lib.gdn_frame_step(*args, B, H, N, dk, dv, _stream_handle(stream)), "gdn_frame_step")
    return out, state_out


def frame_forward_host(q, k, v, alpha, beta, state_in=None, *, out=None, state_out=None, device=None):
    """End-to-end call on HOST tensors: copies the inputs to the device, runs
    gdn_frame_forward, copies out and the final state back (pinned host
    tensors make the copies asynchronous).  Returns host tensors."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    nb = q.is_pinned()
    dq, dk_, dv_ = (t.to(device, non_blocking=nb) for t in (q, k, v))
    da, db = alpha.to(device, non_blocking=nb), beta.to(device, non_blocking=nb)
    ds = None if state_in is None else state_in.to(device, non_blocking=nb)
    o, s = frame_forward(dq, dk_, dv_, da, db, ds)
    if out is None:
        out = torch.empty(o.shape, dtype=o.dtype, pin_memory=nb)
    if state_out is None:
        state_out = torch.empty(s.shape, dtype=s.dtype, pin_memory=nb)
    out.copy_(o, non_blocking=nb)
    state_out.copy_(s, non_blocking=nb)
    torch.cuda.current_stream().synchronize()
    return out, state_out


def workspace_bytes(B, H, F, N, dk, dv) -> int:
    return int(load().gdn_workspace_bytes(B, H, F, N, dk, dv))


def step_workspace_bytes(B, H, N, dk, dv) -> int:
    return int(load().gdn_step_workspace_bytes(B, H, N, dk, dv))


def sync_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded an error."""
    check(load().gdn_sync_status(_stream_handle(stream)), "gdn_sync_status")


def set_wait_limit_ns(ns: int) -> None:
    load().gdn_set_wait_limit_ns(int(ns))


def selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Launch the bounded-wait self-test; returns the status gdn_sync_status reports."""
    lib = load()
    check(lib.gdn_selftest_wait_timeout(int(limit_ns), _stream_handle(stream)), "gdn_selftest_wait_timeout")
    return int(lib.gdn_sync_status(_stream_handle(stream)))


__all__ = ["frame_forward", "frame_step", "frame_forward_host", "workspace_bytes",
           "step_workspace_bytes", "sync_status", "set_wait_limit_ns", "selftest_wait_timeout",
           "GDNError"]
