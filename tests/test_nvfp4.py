"""GPU parity of the NVFP4 entry points (gdn_frame_forward_nvfp4,
gdn_frame_step_nvfp4) against the fp64 oracle on the decoded inputs.

q, k and v are NVFP4 (E2M1 codes, an E4M3 scale per 16 elements along the
head dimension, one fp32 scale per tensor), drawn by inputs.draw_nvfp4 from the
same fp32 draws as the bf16 workloads.  The oracle decodes them by the formats'
definitions (pinned on the CPU) and runs the recurrence in fp64; the kernels
decode in shared memory.  The bar is the bf16 path's: 2e-2 on outputs, 1e-2
on the final state.
"""
import numpy as np
import pytest
import torch

import oracle
from frame_wise_gated_forward_b300 import api, inputs
from frame_wise_gated_forward_b300._lib import GDNError, load
from gpu_util import TOL_OUT, TOL_STATE, ensure_built, rel_err, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def ref_nvfp4(x, B, H, F, N, dk, dv, **kw):
    return oracle.frame_forward_nvfp4(x["q4"], x["k4"], x["v4"], x["q_sf"], x["k_sf"], x["v_sf"], x["q_gs"],
                                      x["k_gs"], x["v_gs"], x["alpha"], x["beta"], x["state_in"],
                                      B=B, H=H, F=F, N=N, dk=dk, dv=dv, **kw)


def dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def gpu_nvfp4(xd, state=True):
    out, st = api.frame_forward_nvfp4(xd["q4"], xd["k4"], xd["v4"], xd["q_sf"], xd["k_sf"], xd["v_sf"], xd["q_gs"],
                                      xd["k_gs"], xd["v_gs"], xd["alpha"], xd["beta"],
                                      xd["state_in"] if state else None)
    api.sync_status()
    return out, st


@pytest.fixture(params=["single", "multi"])
def schedule(request):
    api.set_single_pass(request.param == "single")
    yield request.param
    api.set_single_pass(True)


@pytest.mark.parametrize("shape", [
    (1, 2, 4, 100, 64, 64),       # ragged chunk and tile, one 64-column box
    (1, 8, 9, 880, 64, 64),       # one 9-frame window at d = 64
    (1, 4, 5, 300, 128, 128),     # ragged last chunk and tile at d = 128
    (2, 3, 4, 200, 64, 128),      # dk != dv, two batch rows
    (1, 2, 3, 130, 128, 64),      # dk != dv the other way
])
def test_nvfp4_forward_matches_oracle(shape, schedule):
    B, H, F, N, dk, dv = shape
    x = inputs.draw_nvfp4(B, H, F, N, dk, dv, seed=61, s0_std=0.1)
    ref = ref_nvfp4(x, B, H, F, N, dk, dv)
    out, st = gpu_nvfp4(dev(x))
    eo = rel_err(out.float().cpu().numpy(), ref["out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"nvfp4 {shape} [{schedule}]: err_O={eo:.3e} err_S={es:.3e}")
    assert np.isfinite(out.float().cpu().numpy()).all()
    assert eo <= TOL_OUT and es <= TOL_STATE


def test_nvfp4_sixty_second_sequence():
    """The full 60 s shape (H=16, F=121, N=880, d=128), final state whole and
    sampled outputs; the same call again gives the same bits."""
    w = inputs.WORKLOADS["seq60s"]
    x = inputs.draw_nvfp4(w.B, w.H, w.F, w.N, w.dk, w.dv, seed=0)
    toks = sample_tokens(w.B, w.F, w.N)
    ref = ref_nvfp4(x, w.B, w.H, w.F, w.N, w.dk, w.dv, want_out=False, sample_tokens=toks)
    xd = dev(x)
    out, st = gpu_nvfp4(xd, state=False)
    flat = out.view(-1, w.H, w.dv)[torch.as_tensor(toks, device="cuda")].float().cpu().numpy()
    eo = rel_err(flat, ref["sample_out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"nvfp4 seq60s: err_O(sampled {toks.size})={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE
    out2, st2 = gpu_nvfp4(xd, state=False)
    assert torch.equal(out, out2) and torch.equal(st, st2)


def test_nvfp4_step_rollout():
    """Six frames through gdn_frame_step_nvfp4 on a resident state against the
    oracle's whole sequence."""
    B, H, F, N, d = 1, 4, 6, 300, 128
    x = inputs.draw_nvfp4(B, H, F, N, d, d, seed=62, s0_std=0.1)
    ref = ref_nvfp4(x, B, H, F, N, d, d)
    xd = dev(x)
    state = xd["state_in"].clone()
    outs = []
    for f in range(F):
        o, _ = api.frame_step_nvfp4(*[xd[k][:, f].contiguous() for k in ("q4", "k4", "v4", "q_sf", "k_sf", "v_sf")],
                                    xd["q_gs"], xd["k_gs"], xd["v_gs"], xd["alpha"][:, f].contiguous(),
                                    xd["beta"][:, f].contiguous(), state, state_out=state)
        outs.append(o)
    api.sync_status()
    out = torch.stack(outs, dim=1)
    eo = rel_err(out.float().cpu().numpy(), ref["out"])
    es = rel_err(state.cpu().numpy(), ref["state"])
    print(f"nvfp4 step rollout: err_O={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE


def test_nvfp4_argument_errors_and_beta_range():
    lib = load()
    B, H, F, N, d = 1, 2, 2, 64, 64
    x = dev(inputs.draw_nvfp4(B, H, F, N, d, d, seed=63))
    out = torch.empty((B, F, N, H, d), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call(q_sf=None, dk=d, dv=d, beta=None):
        q_sf = x["q_sf"].data_ptr() if q_sf is None else q_sf
        beta = x["beta"] if beta is None else beta
        return lib.gdn_frame_forward_nvfp4(x["q4"].data_ptr(), x["k4"].data_ptr(), x["v4"].data_ptr(), q_sf,
                                           x["k_sf"].data_ptr(), x["v_sf"].data_ptr(), x["q_gs"], x["k_gs"],
                                           x["v_gs"], x["alpha"].data_ptr(), beta.data_ptr(), None, out.data_ptr(),
                                           None, B, H, F, N, dk, dv, s)
    assert call(dk=32, dv=32) == 3                  # head sizes 64 or 128 only
    assert call(q_sf=x["q_sf"].data_ptr() + 4) == 4  # scales 16-byte aligned
    assert call(q_sf=out.data_ptr()) == 8           # a scale array under the output
    assert call() == 0 and lib.gdn_sync_status(s) == 0
    bad = x["beta"].clone()
    bad[0, 1, 3, 1] = 600.0                         # beyond [0, 512]
    assert call(beta=bad) == 0
    assert lib.gdn_sync_status(s) == 11             # GDN_ERR_RANGE, reported once
    assert call() == 0 and lib.gdn_sync_status(s) == 0
    with pytest.raises(GDNError):
        api.frame_forward_nvfp4(x["q4"][..., :16].contiguous(), x["k4"][..., :16].contiguous(),
                                x["v4"][..., :16].contiguous(), x["q_sf"][..., :2].contiguous(),
                                x["k_sf"][..., :2].contiguous(), x["v_sf"][..., :2].contiguous(),
                                x["q_gs"], x["k_gs"], x["v_gs"], x["alpha"], x["beta"])
