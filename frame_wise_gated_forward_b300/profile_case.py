"""Run the frame-wise GDN forward (or the step, the 8-bit-input forward or the
backward) a few times on a 60 s-sequence-shaped case with a chosen number of
latent frames, for profilers (ncu) to capture.

    python -m frame_wise_gated_forward_b300.profile_case --frames 31 --iters 2 [--schedule multi] [--pairs 1]

Shapes are those of the 60 s 720p workload (H=16, N=880, d=128) with F
frames; inputs come from the seeded generator.  Prints the event-timed
milliseconds per call.
"""
import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from frame_wise_gated_forward_b300 import api, build, inputs  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--frames", type=int, default=31)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--heads", type=int, default=16)
    ap.add_argument("--tokens", type=int, default=880)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--iters", type=int, default=2)
    ap.add_argument("--mode", choices=["forward", "step", "fp8", "backward"], default="forward",
                    help="gdn_frame_forward, gdn_frame_step (F ignored), gdn_frame_forward_fp8 or "
                         "gdn_frame_backward")
    ap.add_argument("--step", action="store_true", help="same as --mode step")
    ap.add_argument("--schedule", choices=["single", "multi"], default="single",
                    help="the whole forward in one launch, or phase 1 then phases 2+3")
    ap.add_argument("--pairs", type=int, default=0, help="phase 1 on head pairs (1) or single heads (0)")
    a = ap.parse_args()
    mode = "step" if a.step else a.mode
    build.build()
    api.set_single_pass(a.schedule == "single")
    api.set_contract_pairs(bool(a.pairs))
    F = 1 if mode == "step" else a.frames
    B, H, N, d = a.batch, a.heads, a.tokens, a.d
    if mode == "fp8":
        x8 = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inputs.draw_fp8(B, H, F, N, d, d, seed=0).items()}
        call = lambda: api.frame_forward_fp8(x8["q8"], x8["k8"], x8["v8"], x8["q_scale"], x8["k_scale"],  # noqa: E731
                                             x8["v_scale"], x8["alpha"], x8["beta"], None)
    else:
        x = inputs.draw(B, H, F, N, d, d, seed=0, s0_std=0.0)
        xd = {k: v.cuda() for k, v in x.items()}
        if mode == "step":
            args = [xd[k][:, 0].contiguous() for k in ("q", "k", "v", "alpha", "beta")]
            call = lambda: api.frame_step(*args, xd["state_in"])  # noqa: E731
        elif mode == "backward":
            g = torch.Generator().manual_seed(1)
            d_out = torch.randn((B, F, N, H, d), generator=g).to(torch.bfloat16).cuda()
            call = lambda: api.frame_backward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], None,  # noqa: E731
                                              d_out)
        else:
            call = lambda: api.frame_forward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], None)  # noqa: E731
    call()
    api.sync_status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.iters):
        call()
    e1.record()
    api.sync_status()
    print(f"{mode} B={B} H={H} F={F} N={N} d={d}: {e0.elapsed_time(e1) / a.iters:.4f} ms/call")


if __name__ == "__main__":
    main()
