"""GPU parity of gdn_frame_backward against the fp64 backward oracle.

The oracle's backward (oracle/gdn_oracle.c, backward_head) is pinned on the
CPU against central differences and autograd.  Here the CUDA backward gets
the same seeded inputs and upstream gradients.  Bar, per gradient:
max|g - g_ref| / max|g_ref| <= 2e-2 -- the same class of error as the
forward's outputs: bf16 inputs, bf16 per-frame state and state-gradient
images as MMA operands, fp32 accumulation, bf16 rounding of dq, dk, dv.
"""
import numpy as np
import pytest
import torch

import oracle
from frame_wise_gated_forward_b300 import api, inputs
from gpu_util import ensure_built, rel_err

pytestmark = pytest.mark.gpu
TOL_GRAD = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def case(B, H, F, N, dk, dv, seed, s0_std=0.1, with_dsf=True):
    x = inputs.draw(B, H, F, N, dk, dv, seed=seed, s0_std=s0_std)
    g = torch.Generator().manual_seed(seed + 1000)
    d_out = torch.randn((B, F, N, H, dv), generator=g).to(torch.bfloat16)
    d_sf = torch.randn((B, H, dv, dk), generator=g) * 0.1 if with_dsf else None
    return x, d_out, d_sf


def run_both(x, d_out, d_sf, dims):
    B, H, F, N, dk, dv = dims
    ref = oracle.frame_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"], d_out, d_sf,
                                B=B, H=H, F=F, N=N, dk=dk, dv=dv)
    xd = {k: v.cuda() for k, v in x.items()}
    got = api.frame_backward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["state_in"], d_out.cuda(),
                             None if d_sf is None else d_sf.cuda())
    api.sync_status()
    names = ("dq", "dk", "dv", "d_alpha", "d_beta", "d_state_in")
    return ref, dict(zip(names, got)), names


@pytest.mark.parametrize("dims", [
    (1, 2, 3, 16, 32, 32),       # one chunk and one tile per frame
    (1, 2, 4, 100, 64, 64),      # ragged N, d = 64 (one 64-column box)
    (2, 2, 3, 130, 128, 128),    # two batch rows, ragged second tile
    (1, 3, 3, 64, 64, 128),      # dk != dv
    (1, 2, 2, 200, 128, 48),     # dv not a multiple of 32
])
def test_backward_full_compare(dims):
    x, d_out, d_sf = case(*dims, seed=21)
    ref, got, names = run_both(x, d_out, d_sf, dims)
    errs = {n: rel_err(got[n].float().cpu().numpy(), ref[n]) for n in names}
    print(dims, {n: f"{e:.2e}" for n, e in errs.items()})
    for n in names:
        assert np.isfinite(got[n].float().cpu().numpy()).all(), n
        assert errs[n] <= TOL_GRAD, (n, errs[n])


def test_backward_sixty_second_shapes():
    """16 frames of the 60 s workload's shape (H=16, N=880, d=128), zero S_0,
    no upstream state gradient; then the same call again gives the same bits."""
    dims = (1, 16, 16, 880, 128, 128)
    x, d_out, _ = case(*dims, seed=22, s0_std=0.0, with_dsf=False)
    ref, got, names = run_both(x, d_out, None, dims)
    errs = {n: rel_err(got[n].float().cpu().numpy(), ref[n]) for n in names}
    print(dims, {n: f"{e:.2e}" for n, e in errs.items()})
    for n in names:
        assert errs[n] <= TOL_GRAD, (n, errs[n])
    xd = {k: v.cuda() for k, v in x.items()}
    again = api.frame_backward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["state_in"], d_out.cuda())
    api.sync_status()
    for n, t in zip(names, again):
        assert torch.equal(t, got[n]), n


def test_backward_rejects_bad_arguments():
    from frame_wise_gated_forward_b300._lib import load
    lib = load()
    B, H, F, N, d = 1, 2, 2, 64, 64
    x = {k: v.cuda() for k, v in inputs.draw(B, H, F, N, d, d, seed=3).items()}
    d_out = torch.zeros_like(x["q"])
    outs = [torch.empty_like(x["q"]), torch.empty_like(x["q"]), torch.empty_like(x["q"]),
            torch.empty_like(x["alpha"]), torch.empty_like(x["beta"]), torch.empty_like(x["state_in"])]
    p = [t.data_ptr() for t in outs]
    s = torch.cuda.current_stream().cuda_stream

    def call(dq=p[0], dk=p[1], dv=p[2], da=p[3], db=p[4], ds=p[5], q=x["q"].data_ptr()):
        return lib.gdn_frame_backward(q, x["k"].data_ptr(), x["v"].data_ptr(), x["alpha"].data_ptr(),
                                      x["beta"].data_ptr(), x["state_in"].data_ptr(), d_out.data_ptr(), None,
                                      dq, dk, dv, da, db, ds, B, H, F, N, d, d, s)
    assert call(dq=None) == 1
    assert call(dk=x["k"].data_ptr()) == 8       # a gradient written over an input
    assert call(dv=p[0]) == 8                    # two gradients on one buffer
    assert call(dq=p[0] + 2) == 4                # misaligned
    assert call() == 0
    assert lib.gdn_sync_status(s) == 0


@pytest.mark.parametrize("dims", [
    (2, 2, 3, 130, 128, 128),    # two batch rows, ragged second tile
    (1, 3, 3, 64, 64, 128),      # dk != dv
    (1, 16, 16, 880, 128, 128),  # 16 frames of the 60 s shape
])
def test_forward_save_and_backward_from_saved_activations(dims):
    """gdn_frame_forward_save gives the forward's results plus A_f and the
    per-frame state images; gdn_frame_backward_saved from them gives the same
    bits as the backward that recomputes them, and matches the oracle."""
    B, H, F, N, dk, dv = dims
    x, d_out, d_sf = case(*dims, seed=23)
    xd = {k: v.cuda() for k, v in x.items()}
    api.set_single_pass(False)
    try:
        o_ref, s_ref = api.frame_forward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["state_in"])
    finally:
        api.set_single_pass(True)
    o, s, sa, ss = api.frame_forward_save(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["state_in"])
    api.sync_status()
    assert torch.equal(o, o_ref) and torch.equal(s, s_ref)
    st = oracle.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"], B=B, H=H, F=F, N=N,
                              dk=dk, dv=dv, want_out=False, want_states=True)["states"]     # [B, H, F, dv, dk]
    assert rel_err(ss.float().permute(0, 2, 1, 3, 4).cpu().numpy(), st) <= 1e-2
    dd = d_out.cuda()
    dsf = d_sf.cuda()
    g_re = api.frame_backward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["state_in"], dd, dsf)
    g_sv = api.frame_backward_saved(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["state_in"], sa, ss, dd,
                                    dsf)
    api.sync_status()
    names = ("dq", "dk", "dv", "d_alpha", "d_beta", "d_state_in")
    for n, a, b in zip(names, g_re, g_sv):
        assert torch.equal(a, b), n
    ref = oracle.frame_backward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"], d_out, d_sf,
                                B=B, H=H, F=F, N=N, dk=dk, dv=dv)
    for n, t in zip(names, g_sv):
        assert rel_err(t.float().cpu().numpy(), ref[n]) <= TOL_GRAD, n
