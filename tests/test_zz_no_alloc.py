"""GPU test of gdn_frame_step_noalloc, the allocation-free step.

Some callers cannot allocate device memory when they advance a resident
state (for example an interactive rollout that reserved nearly all device
memory for its models up front).  gdn_frame_step_noalloc serves them: it runs
the step path with its workspace in a fixed device array inside the library
instead of a pool allocation.  This test calls it through the C ABI twice in a
row (two consecutive frames, so the second call reuses the scratch holding the
first call's contents) and checks each result against gdn_frame_step.  The
file is named to be collected last, and passes alone or after other tests.
"""
import ctypes

import pytest
import torch

from frame_wise_gated_forward_b300 import inputs
from frame_wise_gated_forward_b300._lib import load
from gpu_util import TOL_OUT, TOL_STATE, ensure_built, rel_err

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(fn, x, f, s_in, out, s_out, B, H, N, d):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [x["q"][:, f].contiguous(), x["k"][:, f].contiguous(), x["v"][:, f].contiguous(),
            x["alpha"][:, f].contiguous(), x["beta"][:, f].contiguous()]
    return fn(*[_ptr(a) for a in args], _ptr(s_in), _ptr(out), _ptr(s_out), B, H, N, d, d, stream)


def test_noalloc_step_matches_step_on_two_calls_in_a_row():
    ensure_built()
    lib = load()
    B, H, N, d = 1, 16, 880, 128
    x = {k: v.cuda() for k, v in inputs.draw(B, H, 2, N, d, d, seed=77, s0_std=0.1).items()}
    s_ref = x["state_in"].clone()
    s_na = x["state_in"].clone()
    for f in range(2):
        o_ref = torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda")
        o_na = torch.full((B, N, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call(lib.gdn_frame_step, x, f, s_ref, o_ref, s_ref, B, H, N, d) == 0
        assert _call(lib.gdn_frame_step_noalloc, x, f, s_na, o_na, s_na, B, H, N, d) == 0
        assert lib.gdn_sync_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
        eo = rel_err(o_na.float().cpu().numpy(), o_ref.float().cpu().numpy())
        es = rel_err(s_na.cpu().numpy(), s_ref.cpu().numpy())
        assert eo <= TOL_OUT and es <= TOL_STATE, (f, eo, es)


def test_noalloc_step_rejects_shapes_beyond_its_scratch():
    """With the one-launch step off the call runs on the fixed scratch array,
    and a shape whose workspace exceeds it is refused before any launch."""
    ensure_built()
    lib = load()
    lib.gdn_set_fused_step(0)
    B, H, N, d = 4, 72, 1100, 128        # 288 heads: 36+ MiB of workspace
    q = torch.zeros((B, N, H, d), dtype=torch.bfloat16, device="cuda")
    k, v, out = torch.zeros_like(q), torch.zeros_like(q), torch.zeros_like(q)
    alpha = torch.ones((B, H), device="cuda")
    beta = torch.zeros((B, N, H), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.gdn_frame_step_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), None, _ptr(out), None,
                                    B, H, N, d, d, stream)
    lib.gdn_set_fused_step(1)
    assert rc == 10  # GDN_ERR_TOO_LARGE, nothing launched
    assert lib.gdn_step_workspace_bytes(B, H, N, d, d) > (32 << 20)
    # the one-launch step needs no scratch: the same shape runs
    rc = lib.gdn_frame_step_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), None, _ptr(out), None,
                                    B, H, N, d, d, stream)
    assert rc == 0 and lib.gdn_sync_status(stream) == 0
