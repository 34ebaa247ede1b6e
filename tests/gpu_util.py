"""Helpers shared by the GPU parity tests (CUDA path vs the fp64 oracle)."""
import numpy as np
import torch

import oracle
from frame_wise_gated_forward_b300 import api, build

# Tolerances of the frame-wise GDN forward with bf16 inputs and fp32
# accumulation: max|O - O_ref| / max|O_ref| and the same for the final state.
TOL_OUT = 2e-2
TOL_STATE = 1e-2


def ensure_built():
    build.build()


def to_dev(x):
    return {k: v.cuda() for k, v in x.items()}


def rel_err(a, ref):
    a = np.asarray(a, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max()
    return float(np.abs(a - ref).max() / (den if den > 0 else 1.0))


def oracle_run(x, B, H, F, N, dk, dv, zero_state=False, **kw):
    return oracle.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"],
                                None if zero_state else x["state_in"],
                                B=B, H=H, F=F, N=N, dk=dk, dv=dv, **kw)


def gpu_forward(xd, zero_state=False, **kw):
    out, st = api.frame_forward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"],
                                None if zero_state else xd["state_in"], **kw)
    api.sync_status()
    return out, st


def sample_tokens(B, F, N, n_random=1500, seed=0):
    """Flat token indices (b*F + f)*N + n: every frame's first and last token,
    the whole last frame's ragged 128-token tail, and random tokens."""
    g = np.random.default_rng(seed)
    idx = set()
    for b in range(B):
        for f in range(F):
            base = (b * F + f) * N
            idx.update([base, base + N - 1, base + N // 2])
        last = (b * F + F - 1) * N
        idx.update(range(last + (N // 128) * 128, last + N))
    idx.update(g.integers(0, B * F * N, size=n_random).tolist())
    return np.array(sorted(idx), dtype=np.int64)


def random_inputs(B, H, F, N, dk, dv, seed, s0_std=0.1):
    """Generic seeded inputs with the workloads' distributions at any shape."""
    from frame_wise_gated_forward_b300 import inputs
    return inputs.draw(B, H, F, N, dk, dv, seed, s0_std)
