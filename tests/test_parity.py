"""GPU parity of the CUDA path against the fp64 oracle on the five workloads.

The CUDA path (C ABI, sm_103a kernels) and the oracle get the same seeded
inputs.  Bar: max|O - O_ref| / max|O_ref| <= 2e-2 and the same <= 1e-2 for the
final state S_F, with bf16 inputs and fp32 accumulation.  At the full sizes the
final state is compared whole and the outputs on sampled tokens (every frame's
first/middle/last token, the ragged last tile, random tokens).
"""
import numpy as np
import pytest
import torch

from frame_wise_gated_forward_b300 import api, inputs
from gpu_util import (TOL_OUT, TOL_STATE, ensure_built, gpu_forward, oracle_run, rel_err,
                      sample_tokens, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.fixture(params=["single", "fused", "separate"])
def schedule(request):
    """The whole forward in one launch; or phase 1, then phases 2 and 3 as one
    cooperative launch or as two launches."""
    api.set_single_pass(request.param == "single")
    api.set_fused_scan(request.param != "separate")
    yield request.param
    api.set_single_pass(True)
    api.set_fused_scan(True)


@pytest.mark.parametrize("name", ["tiny", "window9"])
def test_small_workloads_full_compare(name, schedule):
    w = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(w)
    ref = oracle_run(x, w.B, w.H, w.F, w.N, w.dk, w.dv)
    out, st = gpu_forward(to_dev(x))
    eo = rel_err(out.float().cpu().numpy(), ref["out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"{name} [{schedule}]: err_O={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE


@pytest.mark.parametrize("name", ["seq60s", "cfg2"])
def test_full_size_workloads(name, schedule):
    w = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(w)
    toks = sample_tokens(w.B, w.F, w.N)
    ref = oracle_run(x, w.B, w.H, w.F, w.N, w.dk, w.dv, want_out=False, sample_tokens=toks)
    out, st = gpu_forward(to_dev(x))
    flat = out.view(-1, w.H, w.dv)[torch.as_tensor(toks, device=out.device)].float().cpu().numpy()
    eo = rel_err(flat, ref["sample_out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"{name} [{schedule}, sched={api.forward_schedule(w.B, w.H, w.F, w.N, w.dk, w.dv)}]: "
          f"err_O(sampled {toks.size})={eo:.3e} err_S={es:.3e}")
    assert np.isfinite(out.float().cpu().numpy()).all()
    assert eo <= TOL_OUT and es <= TOL_STATE
    # the same call again gives the same bits (no atomics decide any sum)
    out2, st2 = gpu_forward(to_dev(x))
    assert torch.equal(out2, out) and torch.equal(st2, st)
    if w.B == 2:
        # each guidance stream on its own gives exactly its rows of the batch
        # (at 14 chunks per item the contraction splits no item, so every sum
        # is taken in the same order whatever the batch)
        for b in range(2):
            xb = {k: v[b:b + 1].contiguous() for k, v in x.items()}
            ob, sb = gpu_forward(to_dev(xb))
            assert torch.equal(ob, out[b:b + 1]) and torch.equal(sb, st[b:b + 1])


def test_streaming_rollout_121_steps(schedule):
    w = inputs.WORKLOADS["stream121"]
    x = inputs.workload_inputs(w)
    toks = sample_tokens(1, w.F, w.N, n_random=500)
    ref = oracle_run(x, 1, w.H, w.F, w.N, w.dk, w.dv, want_out=False, sample_tokens=toks, want_states=True)
    xd = to_dev(x)
    state = torch.zeros((1, w.H, w.dv, w.dk), dtype=torch.float32, device="cuda")
    outs = torch.empty((1, w.F, w.N, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
    for f in range(w.F):
        api.frame_step(xd["q"][:, f], xd["k"][:, f], xd["v"][:, f], xd["alpha"][:, f], xd["beta"][:, f],
                       state, out=outs[:, f], state_out=state)
    api.sync_status()
    flat = outs.view(-1, w.H, w.dv)[torch.as_tensor(toks, device="cuda")].float().cpu().numpy()
    eo = rel_err(flat, ref["sample_out"])
    es = rel_err(state.cpu().numpy(), ref["state"])
    print(f"stream121 [{schedule}]: err_O={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE


def test_schedules_agree_exactly():
    """Phases 2 and 3 fused or as two launches run the same arithmetic."""
    w = inputs.WORKLOADS["seq60s"]
    x = to_dev(inputs.workload_inputs(w))
    res = {}
    api.set_single_pass(False)
    try:
        for fused in (True, False):
            api.set_fused_scan(fused)
            res[fused] = gpu_forward(x)
    finally:
        api.set_fused_scan(True)
        api.set_single_pass(True)
    assert torch.equal(res[True][0], res[False][0]) and torch.equal(res[True][1], res[False][1])


@pytest.mark.parametrize("contract_ctas,ring", [(0, 0), (20, 4), (100, 0), (0, 121), (1, 4)])
def test_single_pass_role_splits_and_rings(contract_ctas, ring):
    """The single pass with few or many contraction CTAs and shallow or full
    rings (4 frames: every slot reused 30 times) gives the same bits as the
    automatic plan (every item is summed the same way whoever computes it)
    and matches the oracle."""
    w = inputs.WORKLOADS["seq60s"]
    x = inputs.workload_inputs(w)
    xd = to_dev(x)
    api.set_single_pass(True)
    base = gpu_forward(xd)
    api.set_single_pass(True, contract_ctas, ring)
    try:
        assert api.forward_schedule(w.B, w.H, w.F, w.N, w.dk, w.dv) == 2
        out, st = gpu_forward(xd)
    finally:
        api.set_single_pass(True)
    assert torch.equal(out, base[0]) and torch.equal(st, base[1])
    toks = sample_tokens(w.B, w.F, w.N, n_random=300)
    ref = oracle_run(x, w.B, w.H, w.F, w.N, w.dk, w.dv, want_out=False, sample_tokens=toks)
    flat = out.view(-1, w.H, w.dv)[torch.as_tensor(toks, device=out.device)].float().cpu().numpy()
    assert rel_err(flat, ref["sample_out"]) <= TOL_OUT and rel_err(st.cpu().numpy(), ref["state"]) <= TOL_STATE


@pytest.mark.parametrize("name", ["tiny", "window9", "seq60s"])
def test_reverse_direction(name, schedule):
    """Reverse scan (bidirectional stage): frames F-1 .. 0, against the oracle's reverse mode."""
    import oracle
    w = inputs.WORKLOADS[name]
    x = inputs.workload_inputs(w)
    full = w.F * w.N <= 10000
    toks = None if full else sample_tokens(w.B, w.F, w.N)
    ref = oracle_run(x, w.B, w.H, w.F, w.N, w.dk, w.dv, mode=oracle.MODE_REVERSE, want_out=full,
                     sample_tokens=toks)
    xd = to_dev(x)
    out, st = api.frame_forward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["state_in"], reverse=True)
    api.sync_status()
    if full:
        eo = rel_err(out.float().cpu().numpy(), ref["out"])
    else:
        flat = out.view(-1, w.H, w.dv)[torch.as_tensor(toks, device=out.device)].float().cpu().numpy()
        eo = rel_err(flat, ref["sample_out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"{name} reverse [{schedule}]: err_O={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE


@pytest.mark.parametrize("max_split", [1, 3, 12, 0])
def test_contraction_split_plans(max_split):
    """160 items on the grid: one full round of whole items, then 12 items
    left over, split into 3 or 12 token ranges, or whole (1, and the
    automatic plan at 14 chunks per item).  Every plan matches the oracle;
    each is deterministic."""
    B, H, F, N, d = 1, 16, 10, 880, 128
    x = inputs.draw(B, H, F, N, d, d, seed=5, s0_std=0.1)
    ref = oracle_run(x, B, H, F, N, d, d)
    api.set_contract_split(max_split)
    try:
        out, st = gpu_forward(to_dev(x))
        out2, st2 = gpu_forward(to_dev(x))
    finally:
        api.set_contract_split(0)
    eo = rel_err(out.float().cpu().numpy(), ref["out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"max_split={max_split}: err_O={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE
    assert torch.equal(out, out2) and torch.equal(st, st2)


@pytest.mark.parametrize("max_split", [1, 0])
def test_long_frames_split_across_ctas(max_split):
    """One frame of 16 heads with N = 4100 tokens (65 chunks, the last one 4
    tokens): the automatic plan splits every head into 9 token ranges, whose
    boundaries fall inside the frame and one of which ends on the ragged
    chunk.  Matches the oracle either way."""
    B, H, F, N, d = 1, 16, 1, 4100, 128
    x = inputs.draw(B, H, F, N, d, d, seed=6, s0_std=0.1)
    ref = oracle_run(x, B, H, F, N, d, d)
    api.set_contract_split(max_split)
    try:
        out, st = gpu_forward(to_dev(x))
    finally:
        api.set_contract_split(0)
    eo = rel_err(out.float().cpu().numpy(), ref["out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    print(f"N=4100 max_split={max_split}: err_O={eo:.3e} err_S={es:.3e}")
    assert eo <= TOL_OUT and es <= TOL_STATE


@pytest.mark.parametrize("sched", ["single", "multi"])
@pytest.mark.parametrize("shape", [
    (1, 16, 10, 880, 128, 128),   # the 60 s shape's frames: last chunk reaches 16 tokens into the next frame
    (2, 4, 5, 24, 128, 128),      # frames shorter than one chunk, two batch rows
    (1, 2, 3, 8, 128, 128),       # one 8-token group per frame
])
def test_contract_pairs_match_single_heads(shape, sched):
    """Phase 1 on head pairs (two heads' 512 contiguous bytes per token in one
    copy) gives the same bits as one head at a time, and matches the oracle."""
    B, H, F, N, dk, dv = shape
    x = inputs.draw(B, H, F, N, dk, dv, seed=9, s0_std=0.1)
    xd = to_dev(x)
    api.set_single_pass(sched == "single")
    try:
        api.set_contract_pairs(True)
        o1, s1 = gpu_forward(xd)
        api.set_contract_pairs(False)
        o2, s2 = gpu_forward(xd)
    finally:
        api.set_contract_pairs(False)
        api.set_single_pass(True)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    ref = oracle_run(x, B, H, F, N, dk, dv)
    assert rel_err(o1.float().cpu().numpy(), ref["out"]) <= TOL_OUT
    assert rel_err(s1.cpu().numpy(), ref["state"]) <= TOL_STATE
