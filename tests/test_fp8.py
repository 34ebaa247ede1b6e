"""GPU parity of the 8-bit-input entry points (gdn_frame_forward_fp8,
gdn_frame_step_fp8) against the fp64 oracle on the decoded inputs.

q, k and v are OCP FP8 E4M3 codes with one fp32 scale per tensor, drawn by
inputs.draw_fp8 (the same draws as the bf16 workloads, quantized instead of
rounded).  The oracle decodes the codes by the format's definition and runs
the same recurrence in fp64; the kernels decode them in shared memory.  The
bar is the bf16 path's: max|O - O_ref| / max|O_ref| <= 2e-2 and <= 1e-2 for
the final state.
"""
import numpy as np
import pytest
import torch

import oracle
from frame_wise_gated_forward_b300 import api, inputs
from gpu_util import TOL_OUT, TOL_STATE, ensure_built, rel_err, sample_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def ref_fp8(x, B, H, F, N, dk, dv, **kw):
    return oracle.frame_forward_fp8(x["q8"], x["k8"], x["v8"], x["q_scale"], x["k_scale"], x["v_scale"],
                                    x["alpha"], x["beta"], x["state_in"], B=B, H=H, F=F, N=N, dk=dk, dv=dv, **kw)


def dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def gpu_fp8(xd):
    out, st = api.frame_forward_fp8(xd["q8"], xd["k8"], xd["v8"], xd["q_scale"], xd["k_scale"], xd["v_scale"],
                                    xd["alpha"], xd["beta"], xd["state_in"])
    api.sync_status()
    return out, st


@pytest.mark.parametrize("shape", [
    (1, 2, 4, 16, 32, 32),      # tiny: one chunk, columns past d zero-filled by TMA
    (1, 8, 9, 880, 64, 64),     # one 9-frame window at d = 64
    (1, 4, 5, 300, 128, 128),   # ragged last chunk and tile
    (2, 3, 4, 200, 64, 128),    # dk != dv
    (1, 2, 3, 130, 128, 48),    # dv not a multiple of 32
])
def test_fp8_forward_full_compare(shape):
    B, H, F, N, dk, dv = shape
    x = inputs.draw_fp8(B, H, F, N, dk, dv, seed=11, s0_std=0.1)
    ref = ref_fp8(x, B, H, F, N, dk, dv)
    out, st = gpu_fp8(dev(x))
    eo = rel_err(out.float().cpu().numpy(), ref["out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"fp8 {shape}: err_O={eo:.3e} err_S={es:.3e}")
    assert np.isfinite(out.float().cpu().numpy()).all()
    assert eo <= TOL_OUT and es <= TOL_STATE


def test_fp8_forward_full_size_sampled():
    """The 60 s sequence (H=16, F=121, N=880, d=128) with 8-bit inputs."""
    B, H, F, N, d = 1, 16, 121, 880, 128
    x = inputs.draw_fp8(B, H, F, N, d, d, seed=0)
    toks = sample_tokens(B, F, N)
    ref = ref_fp8(x, B, H, F, N, d, d, want_out=False, sample_tokens=toks)
    out, st = gpu_fp8(dev(x))
    flat = out.view(-1, H, d)[torch.as_tensor(toks, device=out.device)].float().cpu().numpy()
    eo = rel_err(flat, ref["sample_out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"fp8 seq60s: err_O(sampled {toks.size})={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE
    out2, st2 = gpu_fp8(dev(x))
    assert torch.equal(out, out2) and torch.equal(st, st2)


def test_fp8_steps_match_forward_oracle():
    """Frame-by-frame 8-bit steps on a resident state follow the oracle's
    whole-sequence forward."""
    B, H, F, N, d = 1, 4, 6, 300, 128
    x = inputs.draw_fp8(B, H, F, N, d, d, seed=13, s0_std=0.1)
    ref = ref_fp8(x, B, H, F, N, d, d)
    xd = dev(x)
    state = xd["state_in"].clone()
    outs = torch.empty((B, F, N, H, d), dtype=torch.bfloat16, device="cuda")
    for f in range(F):
        api.frame_step_fp8(xd["q8"][:, f].contiguous(), xd["k8"][:, f].contiguous(), xd["v8"][:, f].contiguous(),
                           x["q_scale"], x["k_scale"], x["v_scale"], xd["alpha"][:, f].contiguous(),
                           xd["beta"][:, f].contiguous(), state, out=outs[:, f], state_out=state)
    api.sync_status()
    eo = rel_err(outs.float().cpu().numpy(), ref["out"])
    es = rel_err(state.cpu().numpy(), ref["state"])
    print(f"fp8 steps: err_O={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE


def test_fp8_accepts_float8_tensors_and_rejects_bf16():
    B, H, F, N, d = 1, 2, 2, 64, 64
    x = dev(inputs.draw_fp8(B, H, F, N, d, d, seed=3))
    o1, s1 = api.frame_forward_fp8(x["q8"].view(torch.float8_e4m3fn), x["k8"].view(torch.float8_e4m3fn),
                                   x["v8"].view(torch.float8_e4m3fn), x["q_scale"], x["k_scale"], x["v_scale"],
                                   x["alpha"], x["beta"], x["state_in"])
    o2, s2 = gpu_fp8(x)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    with pytest.raises(TypeError):
        api.frame_forward_fp8(x["q8"].to(torch.bfloat16), x["k8"], x["v8"], 1.0, 1.0, 1.0, x["alpha"], x["beta"])


@pytest.mark.parametrize("bad", [-0.25, 20000.0, float("nan")])
def test_fp8_reports_beta_out_of_range(bad):
    """The 8-bit contraction scales k and v by sqrt(beta) in f16, so it takes
    beta in [0, 16384]; one value outside is reported as GDN_ERR_RANGE (11)
    by gdn_sync_status, and the next call runs clean."""
    B, H, F, N, d = 1, 2, 2, 64, 64
    x = dev(inputs.draw_fp8(B, H, F, N, d, d, seed=4))
    beta = x["beta"].clone()
    beta[0, 1, 5, 1] = bad
    api.frame_forward_fp8(x["q8"], x["k8"], x["v8"], x["q_scale"], x["k_scale"], x["v_scale"],
                          x["alpha"], beta, x["state_in"])
    with pytest.raises(api.GDNError) as e:
        api.sync_status()
    assert e.value.code == 11
    gpu_fp8(x)  # clean inputs: no error left behind
