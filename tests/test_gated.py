"""GPU parity of the folded-prologue entry points (gdn_frame_forward_gated,
gdn_frame_step_gated) against the oracle: the prologue in fp64 by its
definition (L2-normalized q and k, beta = sigmoid(b), alpha =
exp(-softplus(a) * c)) followed by the fp64 frame-wise forward."""
import numpy as np
import pytest
import torch

import oracle
from frame_wise_gated_forward_b300 import api, inputs
from gpu_util import TOL_OUT, TOL_STATE, ensure_built, rel_err, sample_tokens

pytestmark = pytest.mark.gpu
ALPHA_SCALE = 0.05


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def oracle_gated(x, B, H, F, N, dk, dv, **kw):
    qn, kn, alpha, beta = oracle.prologue(x["q"], x["k"], x["a_logit"], x["b_logit"], ALPHA_SCALE)
    return oracle.frame_forward_f64(qn, kn, x["v"], alpha, beta, x["state_in"],
                                    B=B, H=H, F=F, N=N, dk=dk, dv=dv, **kw)


@pytest.mark.parametrize("shape", [(1, 2, 4, 16, 32, 32, 2.0), (1, 8, 9, 880, 64, 64, 0.5),
                                   (1, 3, 5, 150, 48, 80, 3.0), (1, 16, 121, 880, 128, 128, 1.0)])
def test_gated_forward(shape):
    B, H, F, N, dk, dv, qk_std = shape
    x = inputs.draw_raw(B, H, F, N, dk, dv, seed=F * 7 + N, qk_std=qk_std, s0_std=0.1)
    full = B * F * N <= 10000
    toks = None if full else sample_tokens(B, F, N)
    ref = oracle_gated(x, B, H, F, N, dk, dv, want_out=full, sample_tokens=toks)
    xd = {k: v.cuda() for k, v in x.items()}
    out, st = api.frame_forward_gated(xd["q"], xd["k"], xd["v"], xd["a_logit"], xd["b_logit"], ALPHA_SCALE,
                                      xd["state_in"])
    api.sync_status()
    if full:
        eo = rel_err(out.float().cpu().numpy(), ref["out"])
    else:
        flat = out.view(-1, H, dv)[torch.as_tensor(toks, device="cuda")].float().cpu().numpy()
        eo = rel_err(flat, ref["sample_out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"gated {shape}: err_O={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE


def test_gated_step_rollout():
    B, H, F, N, d = 1, 16, 6, 880, 128
    x = inputs.draw_raw(B, H, F, N, d, d, seed=5, qk_std=1.5)
    ref = oracle_gated(x, B, H, F, N, d, d, want_states=True)
    xd = {k: v.cuda() for k, v in x.items()}
    st = torch.zeros((B, H, d, d), device="cuda")
    outs = []
    for f in range(F):
        o, _ = api.frame_step_gated(*(xd[n][:, f].contiguous() for n in ("q", "k", "v", "a_logit", "b_logit")),
                                    ALPHA_SCALE, st, state_out=st)
        outs.append(o)
    api.sync_status()
    out = torch.stack(outs, dim=1)
    eo = rel_err(out.float().cpu().numpy(), ref["out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"gated step x{F}: err_O={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE


def test_gated_equals_plain_on_prenormalized_inputs():
    """With unit-norm bf16 q, k the folded prologue only adds the gates: the
    gated call matches the plain call given the same alpha and beta."""
    B, H, F, N, d = 1, 4, 6, 300, 128
    x = inputs.draw(B, H, F, N, d, d, seed=9)
    b = torch.randn((B, F, N, H), generator=torch.Generator().manual_seed(1)) - 5.0
    a = torch.randn((B, F, H), generator=torch.Generator().manual_seed(2))
    beta = torch.sigmoid(b)
    alpha = torch.exp(-torch.nn.functional.softplus(a) * ALPHA_SCALE)
    xd = {k: v.cuda() for k, v in x.items()}
    o1, s1 = api.frame_forward_gated(xd["q"], xd["k"], xd["v"], a.cuda(), b.cuda(), ALPHA_SCALE, None)
    o2, s2 = api.frame_forward(xd["q"], xd["k"], xd["v"], alpha.cuda(), beta.cuda(), None)
    api.sync_status()
    assert rel_err(o1.float().cpu().numpy(), o2.float().cpu().numpy()) <= 1e-2
    assert rel_err(s1.cpu().numpy(), s2.cpu().numpy()) <= 5e-3


@pytest.mark.parametrize("single", [True, False])
def test_gated_contract_pairs_match_single_heads(single):
    """Phase 1 on head pairs with the folded prologue (k normalized, beta =
    sigmoid(b) inside the scalers) gives the same bits as one head at a time,
    over more frames than the single pass's ring holds, and matches the
    oracle."""
    B, H, F, N, d = 1, 16, 14, 880, 128
    x = inputs.draw_raw(B, H, F, N, d, d, seed=77, qk_std=1.0, s0_std=0.1)
    xd = {k: v.cuda() for k, v in x.items()}

    def run():
        o, s = api.frame_forward_gated(xd["q"], xd["k"], xd["v"], xd["a_logit"], xd["b_logit"], ALPHA_SCALE,
                                       xd["state_in"])
        api.sync_status()
        return o, s
    api.set_single_pass(single)
    try:
        api.set_contract_pairs(True)
        o1, s1 = run()
        api.set_contract_pairs(False)
        o2, s2 = run()
    finally:
        api.set_contract_pairs(False)
        api.set_single_pass(True)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    toks = sample_tokens(B, F, N)
    ref = oracle_gated(x, B, H, F, N, d, d, want_out=False, sample_tokens=toks)
    flat = o1.view(-1, H, d)[torch.as_tensor(toks, device="cuda")].float().cpu().numpy()
    assert rel_err(flat, ref["sample_out"]) <= TOL_OUT
    assert rel_err(s1.cpu().numpy(), ref["state"]) <= TOL_STATE
