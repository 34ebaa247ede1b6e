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

import ctypes

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


def frame_forward(q, k, v, alpha, beta, state_in=None, *, out=None, state_out=None, stream=None,
                  reverse=False):
    """Whole-sequence forward.  Returns (out bf16 [B,F,N,H,dv], state_out fp32 [B,H,dv,dk]).
    reverse=True scans the frames from the last to the first (bidirectional stage)."""
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
    fn = lib.gdn_frame_forward_reverse if reverse else lib.gdn_frame_forward
    check(fn(*args, B, H, F, N, dk, dv, _stream_handle(stream)), "gdn_frame_forward")
    return out, state_out


def frame_forward_gated(q, k, v, a_logit, b_logit, alpha_scale, state_in=None, *, out=None, state_out=None,
                        stream=None):
    """Forward on raw q/k and gate logits: q and k are L2-normalized per (token,
    head), beta = sigmoid(b_logit), alpha = exp(-softplus(a_logit) * alpha_scale),
    all inside the kernels.  Shapes as frame_forward."""
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
        _dev(a_logit, "a_logit", torch.float32, (B, F, H)),
        _dev(b_logit, "b_logit", torch.float32, (B, F, N, H)),
    ]
    rest = [None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
            _dev(out, "out", torch.bfloat16, (B, F, N, H, dv)),
            _dev(state_out, "state_out", torch.float32, (B, H, dv, dk))]
    check(lib.gdn_frame_forward_gated(*args, float(alpha_scale), *rest, B, H, F, N, dk, dv, _stream_handle(stream)),
          "gdn_frame_forward_gated")
    return out, state_out


def frame_step_gated(q, k, v, a_logit, b_logit, alpha_scale, state_in=None, *, out=None, state_out=None,
                     stream=None):
    """One frame on a resident state with the folded prologue (see frame_forward_gated).
    q, k [B,N,H,dk]; v [B,N,H,dv]; a_logit [B,H]; b_logit [B,N,H]."""
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
        _dev(a_logit, "a_logit", torch.float32, (B, H)),
        _dev(b_logit, "b_logit", torch.float32, (B, N, H)),
    ]
    rest = [None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
            _dev(out, "out", torch.bfloat16, (B, N, H, dv)),
            _dev(state_out, "state_out", torch.float32, (B, H, dv, dk))]
    check(lib.gdn_frame_step_gated(*args, float(alpha_scale), *rest, B, H, N, dk, dv, _stream_handle(stream)),
          "gdn_frame_step_gated")
    return out, state_out


def frame_forward_save(q, k, v, alpha, beta, state_in=None, *, out=None, state_out=None, saved_A=None,
                       saved_S=None, stream=None):
    """frame_forward that also writes the activations its backward needs:
    returns (out, state_out, saved_A, saved_S) with saved_A bf16 [B,F,H,dk,dk]
    (A_f of every frame) and saved_S bf16 [B,F,H,dv,dk] (the state after every
    frame); pass them to frame_backward_saved."""
    lib = load()
    B, F, N, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    if out is None:
        out = torch.empty((B, F, N, H, dv), dtype=torch.bfloat16, device=dev)
    if state_out is None:
        state_out = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev)
    if saved_A is None:
        saved_A = torch.empty((B, F, H, dk, dk), dtype=torch.bfloat16, device=dev)
    if saved_S is None:
        saved_S = torch.empty((B, F, H, dv, dk), dtype=torch.bfloat16, device=dev)
    args = [
        _dev(q, "q", torch.bfloat16, (B, F, N, H, dk)),
        _dev(k, "k", torch.bfloat16, (B, F, N, H, dk)),
        _dev(v, "v", torch.bfloat16, (B, F, N, H, dv)),
        _dev(alpha, "alpha", torch.float32, (B, F, H)),
        _dev(beta, "beta", torch.float32, (B, F, N, H)),
        None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
        _dev(out, "out", torch.bfloat16, (B, F, N, H, dv)),
        _dev(state_out, "state_out", torch.float32, (B, H, dv, dk)),
        _dev(saved_A, "saved_A", torch.bfloat16, (B, F, H, dk, dk)),
        _dev(saved_S, "saved_S", torch.bfloat16, (B, F, H, dv, dk)),
    ]
    check(lib.gdn_frame_forward_save(*args, B, H, F, N, dk, dv, _stream_handle(stream)), "gdn_frame_forward_save")
    return out, state_out, saved_A, saved_S


def frame_backward_saved(q, k, v, alpha, beta, state_in, saved_A, saved_S, d_out, d_state_out=None, *,
                         want_d_state_in=True, stream=None):
    """frame_backward from the activations of frame_forward_save (no
    recompute of phase 1 and the forward scan); the same gradients."""
    return frame_backward(q, k, v, alpha, beta, state_in, d_out, d_state_out, want_d_state_in=want_d_state_in,
                          stream=stream, _saved=(saved_A, saved_S))


def frame_backward(q, k, v, alpha, beta, state_in, d_out, d_state_out=None, *, want_d_state_in=True,
                   stream=None, _saved=None):
    """Gradients of frame_forward: returns (dq, dk, dv, d_alpha, d_beta,
    d_state_in) for upstream d_out [B,F,N,H,dv] (bf16) and d_state_out
    [B,H,dv,dk] (fp32, None = 0).  Shapes and dtypes as the inputs."""
    lib = load()
    B, F, N, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    dq = torch.empty((B, F, N, H, dk), dtype=torch.bfloat16, device=dev)
    dkk = torch.empty((B, F, N, H, dk), dtype=torch.bfloat16, device=dev)
    dvv = torch.empty((B, F, N, H, dv), dtype=torch.bfloat16, device=dev)
    d_alpha = torch.empty((B, F, H), dtype=torch.float32, device=dev)
    d_beta = torch.empty((B, F, N, H), dtype=torch.float32, device=dev)
    d_s0 = torch.empty((B, H, dv, dk), dtype=torch.float32, device=dev) if want_d_state_in else None
    args = [
        _dev(q, "q", torch.bfloat16, (B, F, N, H, dk)),
        _dev(k, "k", torch.bfloat16, (B, F, N, H, dk)),
        _dev(v, "v", torch.bfloat16, (B, F, N, H, dv)),
        _dev(alpha, "alpha", torch.float32, (B, F, H)),
        _dev(beta, "beta", torch.float32, (B, F, N, H)),
        None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
        _dev(d_out, "d_out", torch.bfloat16, (B, F, N, H, dv)),
        None if d_state_out is None else _dev(d_state_out, "d_state_out", torch.float32, (B, H, dv, dk)),
        dq.data_ptr(), dkk.data_ptr(), dvv.data_ptr(), d_alpha.data_ptr(), d_beta.data_ptr(),
        None if d_s0 is None else d_s0.data_ptr(),
    ]
    if _saved is None:
        check(lib.gdn_frame_backward(*args, B, H, F, N, dk, dv, _stream_handle(stream)), "gdn_frame_backward")
    else:
        sa = _dev(_saved[0], "saved_A", torch.bfloat16, (B, F, H, dk, dk))
        ss = _dev(_saved[1], "saved_S", torch.bfloat16, (B, F, H, dv, dk))
        check(lib.gdn_frame_backward_saved(*args[:6], sa, ss, *args[6:], B, H, F, N, dk, dv, _stream_handle(stream)),
              "gdn_frame_backward_saved")
    return dq, dkk, dvv, d_alpha, d_beta, d_s0


def _bytes8(t):
    """e4m3 tensors are passed as their bytes (torch.float8_e4m3fn or uint8)."""
    if isinstance(t, torch.Tensor) and t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8)
    return t


def frame_forward_fp8(q, k, v, q_scale, k_scale, v_scale, alpha, beta, state_in=None, *, out=None,
                      state_out=None, stream=None):
    """Forward on 8-bit inputs: q, k [B,F,N,H,dk] and v [B,F,N,H,dv] as OCP
    FP8 E4M3 (torch.float8_e4m3fn, or uint8 holding the codes), each with one
    fp32 scale (value = scale * e4m3).  out bf16, state fp32 as frame_forward."""
    lib = load()
    q, k, v = _bytes8(q), _bytes8(k), _bytes8(v)
    B, F, N, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, F, N, H, dv), dtype=torch.bfloat16, device=q.device)
    if state_out is None:
        state_out = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    args = [
        _dev(q, "q", torch.uint8, (B, F, N, H, dk)),
        _dev(k, "k", torch.uint8, (B, F, N, H, dk)),
        _dev(v, "v", torch.uint8, (B, F, N, H, dv)),
        float(q_scale), float(k_scale), float(v_scale),
        _dev(alpha, "alpha", torch.float32, (B, F, H)),
        _dev(beta, "beta", torch.float32, (B, F, N, H)),
        None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
        _dev(out, "out", torch.bfloat16, (B, F, N, H, dv)),
        _dev(state_out, "state_out", torch.float32, (B, H, dv, dk)),
    ]
    check(lib.gdn_frame_forward_fp8(*args, B, H, F, N, dk, dv, _stream_handle(stream)), "gdn_frame_forward_fp8")
    return out, state_out


def frame_step_fp8(q, k, v, q_scale, k_scale, v_scale, alpha, beta, state_in=None, *, out=None, state_out=None,
                   stream=None):
    """One frame on a resident state with 8-bit inputs (see frame_forward_fp8).
    q, k [B,N,H,dk]; v [B,N,H,dv]; alpha [B,H]; beta [B,N,H]."""
    lib = load()
    q, k, v = _bytes8(q), _bytes8(k), _bytes8(v)
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=q.device)
    if state_out is None:
        state_out = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
    args = [
        _dev(q, "q", torch.uint8, (B, N, H, dk)),
        _dev(k, "k", torch.uint8, (B, N, H, dk)),
        _dev(v, "v", torch.uint8, (B, N, H, dv)),
        float(q_scale), float(k_scale), float(v_scale),
        _dev(alpha, "alpha", torch.float32, (B, H)),
        _dev(beta, "beta", torch.float32, (B, N, H)),
        None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
        _dev(out, "out", torch.bfloat16, (B, N, H, dv)),
        _dev(state_out, "state_out", torch.float32, (B, H, dv, dk)),
    ]
    check(lib.gdn_frame_step_fp8(*args, B, H, N, dk, dv, _stream_handle(stream)), "gdn_frame_step_fp8")
    return out, state_out


def frame_forward_nvfp4(q4, k4, v4, q_sf, k_sf, v_sf, q_gs, k_gs, v_gs, alpha, beta, state_in=None, *,
                        out=None, state_out=None, stream=None):
    """Forward on NVFP4 inputs: q4, k4 uint8 [B,F,N,H,dk/2] and v4 [B,F,N,H,dv/2]
    (two E2M1 codes per byte, lower-indexed element in the low nibble), block
    scales q_sf, k_sf uint8 [B,F,N,H,dk/16] and v_sf [B,F,N,H,dv/16] (E4M3),
    per-tensor fp32 scales q_gs, k_gs, v_gs.  dk, dv in {64, 128}."""
    lib = load()
    B, F, N, H, hk = q4.shape
    dk, dv = 2 * hk, 2 * v4.shape[-1]
    if out is None:
        out = torch.empty((B, F, N, H, dv), dtype=torch.bfloat16, device=q4.device)
    if state_out is None:
        state_out = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q4.device)
    args = [
        _dev(q4, "q4", torch.uint8, (B, F, N, H, dk // 2)),
        _dev(k4, "k4", torch.uint8, (B, F, N, H, dk // 2)),
        _dev(v4, "v4", torch.uint8, (B, F, N, H, dv // 2)),
        _dev(q_sf, "q_sf", torch.uint8, (B, F, N, H, dk // 16)),
        _dev(k_sf, "k_sf", torch.uint8, (B, F, N, H, dk // 16)),
        _dev(v_sf, "v_sf", torch.uint8, (B, F, N, H, dv // 16)),
        float(q_gs), float(k_gs), float(v_gs),
        _dev(alpha, "alpha", torch.float32, (B, F, H)),
        _dev(beta, "beta", torch.float32, (B, F, N, H)),
        None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
        _dev(out, "out", torch.bfloat16, (B, F, N, H, dv)),
        _dev(state_out, "state_out", torch.float32, (B, H, dv, dk)),
    ]
    check(lib.gdn_frame_forward_nvfp4(*args, B, H, F, N, dk, dv, _stream_handle(stream)), "gdn_frame_forward_nvfp4")
    return out, state_out


def frame_step_nvfp4(q4, k4, v4, q_sf, k_sf, v_sf, q_gs, k_gs, v_gs, alpha, beta, state_in=None, *, out=None,
                     state_out=None, stream=None):
    """One frame on a resident state with NVFP4 inputs (see frame_forward_nvfp4).
    q4, k4 [B,N,H,dk/2]; v4 [B,N,H,dv/2]; scales [B,N,H,d/16]; alpha [B,H]; beta [B,N,H]."""
    lib = load()
    B, N, H, hk = q4.shape
    dk, dv = 2 * hk, 2 * v4.shape[-1]
    if out is None:
        out = torch.empty((B, N, H, dv), dtype=torch.bfloat16, device=q4.device)
    if state_out is None:
        state_out = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q4.device)
    args = [
        _dev(q4, "q4", torch.uint8, (B, N, H, dk // 2)),
        _dev(k4, "k4", torch.uint8, (B, N, H, dk // 2)),
        _dev(v4, "v4", torch.uint8, (B, N, H, dv // 2)),
        _dev(q_sf, "q_sf", torch.uint8, (B, N, H, dk // 16)),
        _dev(k_sf, "k_sf", torch.uint8, (B, N, H, dk // 16)),
        _dev(v_sf, "v_sf", torch.uint8, (B, N, H, dv // 16)),
        float(q_gs), float(k_gs), float(v_gs),
        _dev(alpha, "alpha", torch.float32, (B, H)),
        _dev(beta, "beta", torch.float32, (B, N, H)),
        None if state_in is None else _dev(state_in, "state_in", torch.float32, (B, H, dv, dk)),
        _dev(out, "out", torch.bfloat16, (B, N, H, dv)),
        _dev(state_out, "state_out", torch.float32, (B, H, dv, dk)),
    ]
    check(lib.gdn_frame_step_nvfp4(*args, B, H, N, dk, dv, _stream_handle(stream)), "gdn_frame_step_nvfp4")
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


def frame_forward_timed(q, k, v, alpha, beta, state_in, out, state_out, events, stream=None):
    """gdn_frame_forward that also records four torch.cuda.Event objects
    (already recorded once, so their CUDA handles exist) before phase 1,
    before phase 2, before phase 3 and after phase 3."""
    lib = load()
    B, F, N, H, dk = q.shape
    dv = v.shape[-1]
    handles = (ctypes.c_void_p * 4)(*[int(e.cuda_event) for e in events])
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
    check(lib.gdn_frame_forward_timed(*args, B, H, F, N, dk, dv, _stream_handle(stream), handles),
          "gdn_frame_forward_timed")
    return out, state_out


def _host(t, name, dtype, shape):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}")
    return t.data_ptr()


def frame_forward_host(q, k, v, alpha, beta, state_in=None, *, out=None, state_out=None, stream=None):
    """End-to-end call on HOST tensors through gdn_frame_forward_host: the
    library copies the inputs to the device, runs the forward and copies out
    and the final state back before returning.  Page-locked (pinned) tensors
    give full-speed copies.  Returns host tensors (out, state_out)."""
    lib = load()
    B, F, N, H, dk = q.shape
    dv = v.shape[-1]
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, F, N, H, dv), dtype=torch.bfloat16, pin_memory=pin)
    if state_out is None:
        state_out = torch.empty((B, H, dv, dk), dtype=torch.float32, pin_memory=pin)
    args = [
        _host(q, "q", torch.bfloat16, (B, F, N, H, dk)),
        _host(k, "k", torch.bfloat16, (B, F, N, H, dk)),
        _host(v, "v", torch.bfloat16, (B, F, N, H, dv)),
        _host(alpha, "alpha", torch.float32, (B, F, H)),
        _host(beta, "beta", torch.float32, (B, F, N, H)),
        None if state_in is None else _host(state_in, "state_in", torch.float32, (B, H, dv, dk)),
        _host(out, "out", torch.bfloat16, (B, F, N, H, dv)),
        _host(state_out, "state_out", torch.float32, (B, H, dv, dk)),
    ]
    check(lib.gdn_frame_forward_host(*args, B, H, F, N, dk, dv, _stream_handle(stream)),
          "gdn_frame_forward_host")
    return out, state_out


def set_contract_pairs(on: bool) -> None:
    """Phase 1 on head pairs where the shape allows it (True, the default) or
    one head at a time (False); identical results."""
    load().gdn_set_contract_pairs(1 if on else 0)


def set_host_chunk_frames(frames: int) -> None:
    """Frames per chunk of frame_forward_host's copy/compute pipeline (0: automatic)."""
    load().gdn_set_host_chunk_frames(int(frames))


def workspace_bytes(B, H, F, N, dk, dv) -> int:
    return int(load().gdn_workspace_bytes(B, H, F, N, dk, dv))


def step_workspace_bytes(B, H, N, dk, dv) -> int:
    return int(load().gdn_step_workspace_bytes(B, H, N, dk, dv))


def sync_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded an error."""
    check(load().gdn_sync_status(_stream_handle(stream)), "gdn_sync_status")


def set_fused_scan(mode) -> None:
    """Run the scan and the output pass as one cooperative launch (True or 1,
    the default; 16, 32 or 64 to force the state rows per scan CTA) or as two
    launches (False or 0).  Results are identical."""
    if mode is True:
        mode = 1
    load().gdn_set_fused_scan(int(mode))


def set_contract_split(max_split: int) -> None:
    """Phase-1 work plan: 0 (default) splits the items left over after the
    last full round of the grid into token ranges only when they have at
    least 32 chunks of 64 tokens; 1 never splits; k > 1 always splits them
    into up to k ranges."""
    load().gdn_set_contract_split(int(max_split))


def set_fused_step(on: bool) -> None:
    """One-launch step for frames of up to 1024 tokens (True, the default) or
    the three-phase path (False)."""
    load().gdn_set_fused_step(1 if on else 0)


def set_single_pass(on: bool, contract_ctas: int = 0, ring_frames: int = 0) -> None:
    """Whole forward as one launch (True, the default: one scan CTA per head,
    contraction and output CTAs on the other SMs, frames handed on through
    L2-resident rings) or phase 1 then phases 2+3 (False).  contract_ctas and
    ring_frames > 0 fix the contraction CTA count and the ring depth."""
    load().gdn_set_single_pass(1 if on else 0, int(contract_ctas), int(ring_frames))


def forward_schedule(B, H, F, N, dk, dv) -> int:
    """2: single pass; 1: phase 1 then fused scan/output; 0: three launches."""
    return int(load().gdn_forward_schedule(B, H, F, N, dk, dv))


def scan_schedule(B, H, dv) -> int:
    """+R: fused scan/output with R state rows per scan CTA; -R: two launches."""
    return int(load().gdn_scan_schedule(B, H, dv))


def last_timeout() -> dict:
    """Where the first bounded wait that ran out gave up (and clear it):
    site code, block, thread, value seen, value awaited (site 0: none)."""
    import ctypes
    info = (ctypes.c_int * 5)()
    check(load().gdn_debug_last_timeout(info), "gdn_debug_last_timeout")
    return dict(zip(("site", "block", "thread", "seen", "awaited"), list(info)))


def set_wait_limit_ns(ns: int) -> None:
    load().gdn_set_wait_limit_ns(int(ns))


def selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    """Launch the bounded-wait self-test; returns the status gdn_sync_status reports."""
    lib = load()
    check(lib.gdn_selftest_wait_timeout(int(limit_ns), _stream_handle(stream)), "gdn_selftest_wait_timeout")
    return int(lib.gdn_sync_status(_stream_handle(stream)))


__all__ = ["frame_forward", "frame_forward_save", "frame_backward_saved", "frame_forward_nvfp4", "frame_step_nvfp4", "frame_forward_gated", "frame_step_gated", "frame_step", "frame_forward_timed", "frame_forward_host", "workspace_bytes",
           "step_workspace_bytes", "sync_status", "set_fused_scan", "scan_schedule", "set_single_pass",
           "forward_schedule", "set_wait_limit_ns", "selftest_wait_timeout",
           "GDNError"]
