"""fp64 CPU oracle for the frame-wise Gated DeltaNet forward and its backward.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library and never imports the product package.

The arithmetic lives in ``gdn_oracle.c`` (plain loops, fp64); this module only
builds it with gcc, loads it with ctypes and marshals numpy/torch arrays.

What it computes (SANA-WM article, "The Architecture": a recurrent layer that
processes one whole latent frame per step with a fixed-size state matrix, a
decay gate and a delta-rule correction; wispaper summary, "Methodology" 1:
frames scanned one by one), per (batch, head):

    S_f = alpha_f * S_{f-1} (I - K_f^T B_f K_f) + V_f^T B_f K_f
    O_f = Q_f S_f^T

Every function here is pinned by ``tests/test_oracle.py`` against properties
that the definition and the mathematics fix (token-level gated delta rule at
N=1, closed forms, exact delta writes, linearity, a brute-force unrolled
product, permutation invariance, split/resume, contraction).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

MODE_GDN = 0
MODE_NODELTA = 1
MODE_REVERSE = 2

_lib = None


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``liboracle.so`` beside it (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_gdn_frame_forward.argtypes = [
            p, p, p, p, p, p, p, p, p, p, ctypes.c_int64, p,
            i, i, i, i, i, i, i, i]
        lib.oracle_gdn_frame_forward.restype = ctypes.c_int
        lib.oracle_gdn_frame_forward_f64.argtypes = [
            p, p, p, p, p, p, p, p, p, p, ctypes.c_int64, p,
            i, i, i, i, i, i, i, i]
        lib.oracle_gdn_frame_forward_f64.restype = ctypes.c_int
        lib.oracle_gdn_frame_backward_f64.argtypes = [p] * 14 + [i] * 7
        lib.oracle_gdn_frame_backward_f64.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _bits16(x) -> np.ndarray:
    """bf16 values -> contiguous uint16 bit patterns (torch bf16 tensor, or
    a numpy uint16 array that already holds bf16 bits)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype != torch.bfloat16:
                raise TypeError("oracle expects bf16 q/k/v tensors")
            return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError("oracle expects bf16 bit patterns (uint16)")
    return a


def _f32(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().to(torch.float32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def frame_forward(q, k, v, alpha, beta, state_in=None, *, B, H, F, N, dk, dv,
                  want_out=True, want_states=False, sample_tokens=None,
                  mode=MODE_GDN, n_threads=0):
    """Run the fp64 oracle.

    q, k: bf16 [B,F,N,H,dk]; v: bf16 [B,F,N,H,dv]; alpha fp32 [B,F,H];
    beta fp32 [B,F,N,H]; state_in fp32 [B,H,dv,dk] or None (zero state).
    Returns a dict with ``state`` fp64 [B,H,dv,dk], and optionally ``out``
    fp64 [B,F,N,H,dv], ``states`` fp64 [B,H,F,dv,dk] (state after each frame),
    ``sample_out`` fp64 [S,H,dv] for the flat token indices ``sample_tokens``.
    """
    lib = _load()
    kb, vb = _bits16(k), _bits16(v)
    qb = _bits16(q) if q is not None else None
    al, be = _f32(alpha), _f32(beta)
    s0 = _f32(state_in) if state_in is not None else None
    if kb.size != B * F * N * H * dk or vb.size != B * F * N * H * dv:
        raise ValueError("k/v size does not match B,F,N,H,d")
    if qb is not None and qb.size != B * F * N * H * dk:
        raise ValueError("q size does not match B,F,N,H,dk")
    if al.size != B * F * H or be.size != B * F * N * H:
        raise ValueError("alpha/beta size mismatch")
    if s0 is not None and s0.size != B * H * dv * dk:
        raise ValueError("state_in size mismatch")
    state = np.empty((B, H, dv, dk), dtype=np.float64)
    out = np.empty((B, F, N, H, dv), dtype=np.float64) if want_out else None
    states = np.empty((B, H, F, dv, dk), dtype=np.float64) if want_states else None
    if sample_tokens is not None:
        st = np.ascontiguousarray(sample_tokens, dtype=np.int64)
        sout = np.zeros((st.size, H, dv), dtype=np.float64)
    else:
        st, sout = None, None
    rc = lib.oracle_gdn_frame_forward(
        _ptr(qb), _ptr(kb), _ptr(vb), _ptr(al), _ptr(be), _ptr(s0),
        _ptr(out), _ptr(state), _ptr(states),
        _ptr(st), 0 if st is None else int(st.size), _ptr(sout),
        B, H, F, N, dk, dv, int(mode), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_gdn_frame_forward failed with code {rc}")
    res = {"state": state}
    if out is not None:
        res["out"] = out
    if states is not None:
        res["states"] = states
    if sout is not None:
        res["sample_out"] = sout
    return res


def prologue(q_raw, k_raw, a_logit, b_logit, alpha_scale):
    """The per-token prologue that gdn_frame_forward_gated folds into its
    kernels, in fp64 by its definition:
        q / max(|q|, 1e-12),  k / max(|k|, 1e-12)   (norm over the head dim)
        beta  = sigmoid(b_logit) = 1 / (1 + exp(-b))
        alpha = exp(-softplus(a_logit) * alpha_scale),  softplus(a) = log(1 + exp(a))
    Takes bf16 torch tensors (or fp64 arrays) for q/k and fp32 logits; returns
    fp64 numpy arrays (q, k, alpha, beta)."""
    def f64(x):
        try:
            import torch
            if isinstance(x, torch.Tensor):
                return x.detach().cpu().to(torch.float64).numpy()
        except ImportError:  # pragma: no cover
            pass
        return np.asarray(x, dtype=np.float64)
    q, k = f64(q_raw), f64(k_raw)
    qn = q / np.maximum(np.sqrt((q * q).sum(-1, keepdims=True)), 1e-12)
    kn = k / np.maximum(np.sqrt((k * k).sum(-1, keepdims=True)), 1e-12)
    b = f64(b_logit)
    a = f64(a_logit)
    beta = 1.0 / (1.0 + np.exp(-b))
    softplus = np.logaddexp(0.0, a)
    alpha = np.exp(-softplus * float(alpha_scale))
    return qn, kn, alpha, beta


def decode_e4m3(codes) -> np.ndarray:
    """OCP FP8 E4M3 codes (uint8) -> fp64 values, from the format's definition:
    bit 7 sign s, bits 6..3 exponent e (bias 7), bits 2..0 mantissa m;
        e == 0:              (-1)^s * (m / 8) * 2^-6        (zero and subnormals)
        e == 15 and m == 7:  NaN                             (no infinities)
        otherwise:           (-1)^s * (1 + m / 8) * 2^(e - 7)
    Accepts a uint8 numpy array or torch tensor (uint8 or float8_e4m3fn)."""
    try:
        import torch
        if isinstance(codes, torch.Tensor):
            t = codes.detach().cpu()
            if t.dtype != torch.uint8:
                t = t.view(torch.uint8)
            codes = t.numpy()
    except ImportError:  # pragma: no cover
        pass
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 15
    m = c & 7
    sign = np.where(s == 1, -1.0, 1.0)
    val = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = sign * val
    return np.where((e == 15) & (m == 7), np.nan, val)


def frame_forward_fp8(q8, k8, v8, q_scale, k_scale, v_scale, alpha, beta, state_in=None, *, B, H, F, N,
                      dk, dv, **kw):
    """The forward on 8-bit inputs: every element's value is scale * e4m3(code)
    (one fp32 scale per tensor), then exactly frame_forward_f64 on those values."""
    q = None if q8 is None else decode_e4m3(q8) * float(q_scale)
    k = decode_e4m3(k8) * float(k_scale)
    v = decode_e4m3(v8) * float(v_scale)
    return frame_forward_f64(q, k, v, alpha, beta, state_in, B=B, H=H, F=F, N=N, dk=dk, dv=dv, **kw)


def decode_e2m1(codes) -> np.ndarray:
    """FP4 E2M1 codes (0..15, the low 4 bits of each value) -> fp64 values,
    from the format's definition: bit 3 sign s, bits 2..1 exponent e (bias 1),
    bit 0 mantissa m;
        e == 0:     (-1)^s * (m / 2)                  (zero and the one subnormal)
        otherwise:  (-1)^s * (1 + m / 2) * 2^(e - 1)
    No infinities and no NaN (the largest magnitude is 6)."""
    c = np.asarray(codes).astype(np.int64) & 15
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    val = np.where(e == 0, m / 2.0, (1.0 + m / 2.0) * np.exp2(e.astype(np.float64) - 1.0))
    return np.where(s == 1, -val, val)


def _bytes(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            t = x.detach().cpu()
            if t.dtype != torch.uint8:
                t = t.view(torch.uint8)
            return t.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.uint8)


def decode_nvfp4(packed, scales, global_scale) -> np.ndarray:
    """NVFP4 tensor -> fp64 values [..., d].

    packed: uint8 [..., d/2], element 2i in the low nibble of byte i and element
    2i+1 in the high nibble (E2M1 codes); scales: E4M3 codes [..., d/16], one
    per 16 consecutive elements; global_scale: one fp32 per tensor.
        x[..., i] = global_scale * e4m3(scales[..., i // 16]) * e2m1(code i)"""
    p = _bytes(packed).astype(np.int64)
    codes = np.stack([p & 15, p >> 4], axis=-1).reshape(*p.shape[:-1], 2 * p.shape[-1])
    sc = decode_e4m3(_bytes(scales))
    if sc.shape[-1] * 16 != codes.shape[-1]:
        raise ValueError("one scale per 16 elements")
    return decode_e2m1(codes) * np.repeat(sc, 16, axis=-1) * float(global_scale)


def frame_forward_nvfp4(q4, k4, v4, q_sf, k_sf, v_sf, q_gs, k_gs, v_gs, alpha, beta, state_in=None, *,
                        B, H, F, N, dk, dv, **kw):
    """The forward on NVFP4 inputs: each of q, k, v decoded by decode_nvfp4
    (E2M1 elements, E4M3 scales per 16 elements along the head dimension, one
    fp32 scale per tensor), then exactly frame_forward_f64 on those values."""
    q = None if q4 is None else decode_nvfp4(q4, q_sf, q_gs)
    k = decode_nvfp4(k4, k_sf, k_gs)
    v = decode_nvfp4(v4, v_sf, v_gs)
    return frame_forward_f64(q, k, v, alpha, beta, state_in, B=B, H=H, F=F, N=N, dk=dk, dv=dv, **kw)


def frame_forward_f64(q, k, v, alpha, beta, state_in=None, *, B, H, F, N, dk, dv,
                      want_out=True, want_states=False, sample_tokens=None,
                      mode=MODE_GDN, n_threads=0):
    """frame_forward on fp64 inputs (any array-likes; v may be a bf16 torch tensor)."""
    lib = _load()

    def f64(x):
        if x is None:
            return None
        try:
            import torch
            if isinstance(x, torch.Tensor):
                return x.detach().cpu().to(torch.float64).contiguous().numpy()
        except ImportError:  # pragma: no cover
            pass
        return np.ascontiguousarray(x, dtype=np.float64)
    qa, ka, va, al, be, s0 = (f64(t) for t in (q, k, v, alpha, beta, state_in))
    if ka.size != B * F * N * H * dk or va.size != B * F * N * H * dv or al.size != B * F * H \
            or be.size != B * F * N * H or (qa is not None and qa.size != B * F * N * H * dk) \
            or (s0 is not None and s0.size != B * H * dv * dk):
        raise ValueError("input sizes do not match B,F,N,H,dk,dv")
    state = np.empty((B, H, dv, dk), dtype=np.float64)
    out = np.empty((B, F, N, H, dv), dtype=np.float64) if want_out else None
    states = np.empty((B, H, F, dv, dk), dtype=np.float64) if want_states else None
    if sample_tokens is not None:
        st = np.ascontiguousarray(sample_tokens, dtype=np.int64)
        sout = np.zeros((st.size, H, dv), dtype=np.float64)
    else:
        st, sout = None, None
    rc = lib.oracle_gdn_frame_forward_f64(
        _ptr(qa), _ptr(ka), _ptr(va), _ptr(al), _ptr(be), _ptr(s0),
        _ptr(out), _ptr(state), _ptr(states),
        _ptr(st), 0 if st is None else int(st.size), _ptr(sout),
        B, H, F, N, dk, dv, int(mode), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_gdn_frame_forward_f64 failed with code {rc}")
    res = {"state": state}
    if out is not None:
        res["out"] = out
    if states is not None:
        res["states"] = states
    if sout is not None:
        res["sample_out"] = sout
    return res


def frame_backward(q, k, v, alpha, beta, state_in, d_out, d_state_out=None, *, B, H, F, N, dk, dv,
                   n_threads=0):
    """Reverse-mode derivatives of the forward (fp64; gdn_oracle.c,
    backward_head).  Inputs are any arrays (bf16/fp32 torch tensors or
    numpy), converted to fp64 exactly; d_out [B,F,N,H,dv]; d_state_out
    [B,H,dv,dk] or None (zero).  Returns a dict of fp64 arrays: dq, dk, dv,
    d_alpha [B,F,H], d_beta [B,F,N,H], d_state_in [B,H,dv,dk]."""
    lib = _load()

    def f64(x):
        if x is None:
            return None
        try:
            import torch
            if isinstance(x, torch.Tensor):
                return x.detach().cpu().to(torch.float64).contiguous().numpy()
        except ImportError:  # pragma: no cover
            pass
        return np.ascontiguousarray(x, dtype=np.float64)
    qa, ka, va, al, be, s0, do, dsf = (f64(t) for t in (q, k, v, alpha, beta, state_in, d_out, d_state_out))
    T = B * F * N
    if (qa.size != T * H * dk or ka.size != T * H * dk or va.size != T * H * dv or al.size != B * F * H
            or be.size != T * H or do.size != T * H * dv
            or (s0 is not None and s0.size != B * H * dv * dk)
            or (dsf is not None and dsf.size != B * H * dv * dk)):
        raise ValueError("input sizes do not match B,F,N,H,dk,dv")
    res = {"dq": np.empty((B, F, N, H, dk)), "dk": np.empty((B, F, N, H, dk)), "dv": np.empty((B, F, N, H, dv)),
           "d_alpha": np.empty((B, F, H)), "d_beta": np.empty((B, F, N, H)),
           "d_state_in": np.empty((B, H, dv, dk))}
    rc = lib.oracle_gdn_frame_backward_f64(
        _ptr(qa), _ptr(ka), _ptr(va), _ptr(al), _ptr(be), _ptr(s0), _ptr(do), _ptr(dsf),
        _ptr(res["dq"]), _ptr(res["dk"]), _ptr(res["dv"]), _ptr(res["d_alpha"]), _ptr(res["d_beta"]),
        _ptr(res["d_state_in"]), B, H, F, N, dk, dv, int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle_gdn_frame_backward_f64 failed with code {rc}")
    return res
