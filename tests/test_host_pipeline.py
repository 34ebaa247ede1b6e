"""GPU test of the pipelined end-to-end call gdn_frame_forward_host.

The call streams the sequence through the device in chunks of frames,
copying chunk i in while chunk i-1 runs and chunk i-2's outputs go out, and
carries the state on the device from chunk to chunk.  Splitting the frames
and resuming from the carried state is exact, so the result must be
bit-identical to one gdn_frame_forward over the whole sequence on device
buffers, for every chunk size, with and without an initial state, batch rows
> 1 (strided copies) and pinned or pageable host memory.  Also checked
against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from frame_wise_gated_forward_b300 import api, inputs
from gpu_util import TOL_OUT, TOL_STATE, ensure_built, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


@pytest.mark.parametrize("chunk", [0, 1, 2, 4, 9])
@pytest.mark.parametrize("with_state", [True, False])
def test_host_call_is_bit_identical_to_device_call(chunk, with_state):
    B, H, F, N, d = 2, 3, 9, 100, 64
    x = inputs.draw(B, H, F, N, d, d, seed=71, s0_std=0.1)
    s_in = x["state_in"] if with_state else None
    xd = {k: v.cuda() for k, v in x.items()}
    o_dev, s_dev = api.frame_forward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"],
                                     xd["state_in"] if with_state else None)
    api.sync_status()
    hx = {k: v.pin_memory() for k, v in x.items()}
    h_out = torch.empty((B, F, N, H, d), dtype=torch.bfloat16).pin_memory()
    h_st = torch.empty((B, H, d, d), dtype=torch.float32).pin_memory()
    api.set_host_chunk_frames(chunk)
    try:
        api.frame_forward_host(hx["q"], hx["k"], hx["v"], hx["alpha"], hx["beta"],
                               hx["state_in"] if with_state else None, out=h_out, state_out=h_st)
    finally:
        api.set_host_chunk_frames(0)
    assert torch.equal(h_out, o_dev.cpu()) and torch.equal(h_st, s_dev.cpu())
    ref = oracle.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], s_in, B=B, H=H, F=F, N=N, dk=d, dv=d)
    assert rel_err(h_out.float().numpy(), ref["out"]) <= TOL_OUT
    assert rel_err(h_st.numpy(), ref["state"]) <= TOL_STATE


def test_host_call_with_pageable_memory_and_the_sixty_second_shape():
    w = inputs.WORKLOADS["seq60s"]
    x = inputs.workload_inputs(w)
    xd = {k: v.cuda() for k, v in x.items()}
    o_dev, s_dev = api.frame_forward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], None)
    api.sync_status()
    h_out = torch.empty((w.B, w.F, w.N, w.H, w.dv), dtype=torch.bfloat16)   # pageable
    h_st = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32)
    api.frame_forward_host(x["q"], x["k"], x["v"], x["alpha"], x["beta"], None, out=h_out, state_out=h_st)
    assert torch.equal(h_out, o_dev.cpu()) and torch.equal(h_st, s_dev.cpu())
    assert np.isfinite(h_out.float().numpy()).all()
