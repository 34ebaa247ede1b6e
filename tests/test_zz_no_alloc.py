"""GPU test of gdn_frame_step_noalloc, the allocation-free step.

Some callers cannot allocate device memory when they advance a resident
state: an interactive rollout that reserved nearly all device memory for its
models up front, or a runtime whose allocator must not be entered from this
code path.  gdn_frame_step_noalloc serves them: when the step runs as
several kernels it keeps their workspace in one fixed device array inside the
library instead of a pool allocation.

The tests turn the one-launch step off (which needs no workspace at all), so
that the calls really run the three-phase step on the fixed array, and
restore it afterwards whatever happens.  They call the entry point through
the C ABI twice in a row on consecutive frames (the second call reuses the
array the first call left its contents in), with a call of a smaller shape in
between (stale contents in another layout must not leak into the next call),
and compare every frame with gdn_frame_step and with the fp64 oracle.  The
file is named to be collected last; it passes alone or after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from frame_wise_gated_forward_b300 import inputs
from frame_wise_gated_forward_b300._lib import load
from gpu_util import TOL_OUT, TOL_STATE, ensure_built, rel_err

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call(fn, x, f, s_in, out, s_out, B, H, N, d):
    args = [x["q"][:, f].contiguous(), x["k"][:, f].contiguous(), x["v"][:, f].contiguous(),
            x["alpha"][:, f].contiguous(), x["beta"][:, f].contiguous()]
    return fn(*[_ptr(a) for a in args], _ptr(s_in), _ptr(out), _ptr(s_out), B, H, N, d, d, _stream())


def test_noalloc_step_matches_step_and_oracle_on_two_calls_in_a_row():
    ensure_built()
    lib = load()
    B, H, N, d = 1, 16, 880, 128
    xc = inputs.draw(B, H, 2, N, d, d, seed=77, s0_std=0.1)
    ref = oracle.frame_forward(xc["q"], xc["k"], xc["v"], xc["alpha"], xc["beta"], xc["state_in"],
                               B=B, H=H, F=2, N=N, dk=d, dv=d, want_states=True)
    x = {k: v.cuda() for k, v in xc.items()}
    # a smaller shape run on the same array between the two frames
    ys = inputs.draw(1, 3, 1, 100, 64, 64, seed=78, s0_std=0.1)
    refs = oracle.frame_forward(ys["q"], ys["k"], ys["v"], ys["alpha"], ys["beta"], ys["state_in"],
                                B=1, H=3, F=1, N=100, dk=64, dv=64)
    y = {k: v.cuda() for k, v in ys.items()}
    s_ref = x["state_in"].clone()
    s_na = x["state_in"].clone()
    lib.gdn_set_fused_step(0)
    try:
        assert lib.gdn_step_workspace_bytes(B, H, N, d, d) <= (32 << 20)
        for f in range(2):
            o_ref = torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda")
            o_na = torch.full((B, N, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
            assert _call(lib.gdn_frame_step, x, f, s_ref, o_ref, s_ref, B, H, N, d) == 0
            assert _call(lib.gdn_frame_step_noalloc, x, f, s_na, o_na, s_na, B, H, N, d) == 0
            assert lib.gdn_sync_status(_stream()) == 0
            # the same kernels and work plan on another workspace: the same bits
            assert torch.equal(o_na, o_ref) and torch.equal(s_na, s_ref), f
            eo = rel_err(o_na.float().cpu().numpy(), ref["out"][:, f])
            es = rel_err(s_na.cpu().numpy(), ref["states"][:, :, f])
            print(f"noalloc frame {f}: err_O={eo:.3e} err_S={es:.3e}")
            assert eo <= TOL_OUT and es <= TOL_STATE, (f, eo, es)
            if f == 0:
                o_s = torch.full((1, 100, 3, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
                s_s = torch.empty((1, 3, 64, 64), dtype=torch.float32, device="cuda")
                assert _call(lib.gdn_frame_step_noalloc, y, 0, y["state_in"], o_s, s_s, 1, 3, 100, 64) == 0
                assert lib.gdn_sync_status(_stream()) == 0
                assert rel_err(o_s.float().cpu().numpy(), refs["out"][:, 0]) <= TOL_OUT
                assert rel_err(s_s.cpu().numpy(), refs["state"]) <= TOL_STATE
    finally:
        lib.gdn_set_fused_step(1)


def test_noalloc_step_rejects_shapes_beyond_its_scratch():
    """With the one-launch step off a shape whose workspace exceeds the fixed
    array is refused before any launch; with it on (no workspace) the same
    shape runs."""
    ensure_built()
    lib = load()
    B, H, N, d = 4, 72, 1100, 128        # 288 heads: 36+ MiB of workspace
    q = torch.zeros((B, N, H, d), dtype=torch.bfloat16, device="cuda")
    k, v, out = torch.zeros_like(q), torch.zeros_like(q), torch.zeros_like(q)
    alpha = torch.ones((B, H), device="cuda")
    beta = torch.zeros((B, N, H), device="cuda")
    lib.gdn_set_fused_step(0)
    try:
        rc = lib.gdn_frame_step_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), None, _ptr(out),
                                        None, B, H, N, d, d, _stream())
    finally:
        lib.gdn_set_fused_step(1)
    assert rc == 10  # GDN_ERR_TOO_LARGE, nothing launched
    assert lib.gdn_step_workspace_bytes(B, H, N, d, d) > (32 << 20)
    rc = lib.gdn_frame_step_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), None, _ptr(out), None,
                                    B, H, N, d, d, _stream())
    assert rc == 0 and lib.gdn_sync_status(_stream()) == 0
    assert np.isfinite(out.float().cpu().numpy()).all()
