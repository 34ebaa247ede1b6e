"""GPU edge cases of the CUDA path: ragged frames, every supported head size,
dk != dv, state handling (NULL, in place, split/resume), step vs forward,
batch independence, determinism, guard canaries, error codes and the
bounded-wait self-test."""
import numpy as np
import pytest
import torch

from frame_wise_gated_forward_b300 import api
from frame_wise_gated_forward_b300._lib import GDNError, load
from gpu_util import TOL_OUT, TOL_STATE, ensure_built, gpu_forward, oracle_run, random_inputs, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def check_vs_oracle(B, H, F, N, dk, dv, seed, s0_std=0.1):
    x = random_inputs(B, H, F, N, dk, dv, seed, s0_std)
    ref = oracle_run(x, B, H, F, N, dk, dv)
    out, st = gpu_forward(to_dev(x))
    eo = rel_err(out.float().cpu().numpy(), ref["out"])
    es = rel_err(st.cpu().numpy(), ref["state"])
    assert eo <= TOL_OUT and es <= TOL_STATE, (eo, es)
    return eo, es


@pytest.mark.parametrize("N", [1, 15, 63, 64, 65, 127, 128, 129, 200, 880])
def test_ragged_token_counts(N):
    check_vs_oracle(1, 2, 3, N, 64, 64, seed=N)


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 32), (48, 80), (64, 64), (96, 112), (128, 128),
                                   (128, 64), (64, 128), (112, 48)])
def test_head_sizes(dk, dv):
    check_vs_oracle(1, 3, 4, 150, dk, dv, seed=dk * 1000 + dv)


def test_many_frames_small_heads():
    check_vs_oracle(2, 5, 37, 33, 32, 32, seed=3)


def test_null_state_equals_zero_state():
    x = to_dev(random_inputs(1, 4, 5, 100, 64, 64, seed=4))
    z = torch.zeros_like(x["state_in"])
    o1, s1 = api.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], None)
    o2, s2 = api.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], z)
    api.sync_status()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_in_place_state_and_split_resume_are_exact():
    x = to_dev(random_inputs(1, 4, 9, 130, 128, 128, seed=5))
    o_full, s_full = api.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"])
    st = x["state_in"].clone()
    o_a, _ = api.frame_forward(*(t[:, :4].contiguous() for t in (x["q"], x["k"], x["v"], x["alpha"], x["beta"])),
                               st, state_out=st)
    o_b, _ = api.frame_forward(*(t[:, 4:].contiguous() for t in (x["q"], x["k"], x["v"], x["alpha"], x["beta"])),
                               st, state_out=st)
    api.sync_status()
    assert torch.equal(torch.cat([o_a, o_b], dim=1), o_full)
    assert torch.equal(st, s_full)


def test_step_matches_oracle_and_is_deterministic():
    B, H, N, d = 2, 16, 880, 128
    x = random_inputs(B, H, 1, N, d, d, seed=6)
    ref = oracle_run(x, B, H, 1, N, d, d)
    xd = to_dev(x)
    args = (xd["q"][:, 0].contiguous(), xd["k"][:, 0].contiguous(), xd["v"][:, 0].contiguous(),
            xd["alpha"][:, 0].contiguous(), xd["beta"][:, 0].contiguous(), xd["state_in"])
    o1, s1 = api.frame_step(*args)
    o2, s2 = api.frame_step(*args)
    api.sync_status()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    assert rel_err(o1.float().cpu().numpy(), ref["out"][:, 0]) <= TOL_OUT
    assert rel_err(s1.cpu().numpy(), ref["state"]) <= TOL_STATE


def test_forward_is_deterministic():
    x = to_dev(random_inputs(1, 8, 6, 300, 128, 128, seed=7))
    o1, s1 = gpu_forward(x)
    o2, s2 = gpu_forward(x)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_guard_canaries_untouched():
    B, H, F, N, d = 1, 3, 4, 77, 64
    x = to_dev(random_inputs(B, H, F, N, d, d, seed=8))
    n_out = B * F * N * H * d
    pad = 4096
    buf = torch.full((n_out + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    sbuf = torch.full((B * H * d * d + 2 * pad,), float("nan"), dtype=torch.float32, device="cuda")
    out = buf[pad:pad + n_out].view(B, F, N, H, d)
    st = sbuf[pad:pad + B * H * d * d].view(B, H, d, d)
    api.frame_forward(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["state_in"], out=out, state_out=st)
    api.sync_status()
    assert torch.isnan(buf[:pad].float()).all() and torch.isnan(buf[pad + n_out:].float()).all()
    assert torch.isnan(sbuf[:pad]).all() and torch.isnan(sbuf[pad + B * H * d * d:]).all()
    assert torch.isfinite(out.float()).all() and torch.isfinite(st).all()


def test_error_codes_with_device_tensors():
    lib = load()
    x = to_dev(random_inputs(1, 2, 2, 32, 32, 32, seed=9))
    out = torch.empty((1, 2, 32, 2, 32), dtype=torch.bfloat16, device="cuda")
    base = [x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), x["alpha"].data_ptr(),
            x["beta"].data_ptr(), None, out.data_ptr(), None]
    stream = torch.cuda.current_stream().cuda_stream

    def call(**over):
        a = list(base)
        names = ["q", "k", "v", "alpha", "beta", "s_in", "out", "s_out"]
        for kname, val in over.items():
            a[names.index(kname)] = val
        return lib.gdn_frame_forward(*a, 1, 2, 2, 32, 32, 32, stream)

    assert call() == 0
    assert call(q=base[0] + 2) == 4                       # misaligned bf16 tensor
    assert call(out=base[0]) == 8                         # out aliases q
    host = torch.zeros(1 << 16, dtype=torch.bfloat16)
    assert call(q=host.data_ptr()) == 1                   # host memory is rejected, never launched
    with pytest.raises(GDNError):
        api.frame_forward(x["q"][:, :, :0], x["k"][:, :, :0], x["v"][:, :, :0], x["alpha"],
                          x["beta"][:, :, :0])            # empty frames (N = 0) are rejected
    api.sync_status()


def test_bounded_wait_selftest_reports_timeout_and_context_survives():
    status = api.selftest_wait_timeout(2_000_000)  # 2 ms limit on a barrier nothing completes
    assert status == 7
    api.sync_status()  # cleared
    check_vs_oracle(1, 2, 2, 40, 32, 32, seed=10)
