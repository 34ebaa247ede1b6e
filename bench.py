#!/usr/bin/env python3
"""Benchmark of the frame-wise Gated DeltaNet forward on B300.

One step = one gdn_frame_forward call over the 60 s 720p latent sequence
(B=1, H=16, F=121 latent frames x N=880 tokens, dk=dv=128; inputs resident in
HBM).  Prints ONE JSON line (rank 0):

  value       whole-job tokens/s (device time, CUDA events, max over ranks)
  roofline    the dominant kernel's algorithmic bytes / its event-timed
              duration against the measured HBM copy bandwidth
  e2e         the same metric through gdn_frame_forward_host on pinned host
              buffers, host<->device copies inside the timed region
  cpu_baseline  the fp64 CPU oracle on the host cores (rank 0, N=1 only)
  clocks      NVML samples (SM clock, throttle reasons) taken during the
              timed region

--impl reference times the fp64 CPU oracle on the same workload instead
(a bounded sample of frames per step).

Multi-GPU: launch under torchrun; each rank runs its own sequence (weak
scaling, replicas only: no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN fwd tokens/s (121×880 tok, 16 heads, d=128) and % tensor/HBM roofline"
UNIT = "tokens/s"
WORKLOAD = "seq60s"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--reference-budget-s", type=float, default=90.0,
                    help="wall-clock budget of the --impl reference run")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def kernel_costs(w):
    """Bytes and FLOPs of one launch of each kernel of the forward.

    "bytes" are the algorithmic bytes: what the layer itself must move for the
    part of the work the kernel does (q, k, v, beta and alpha read, out
    written, the initial and final state), 16,468 B per token at H = 16,
    d = 128 over the whole path.  The per-frame workspace that a multi-launch
    schedule adds (A_f, U_f written by the contraction and read back, the bf16
    per-frame states) is reported apart as "overhead_bytes": it is a cost of
    the schedule, not work of the layer.
    """
    T = w.B * w.F * w.N            # tokens
    items = w.B * w.F * w.H        # (b, f, h) items
    dk, dv, H = w.dk, w.dv, w.H
    ws_a = items * dk * dk * 2     # A_f bf16
    ws_u = items * dv * dk * 4     # U_f fp32
    ws_s = items * dv * dk * 2     # S_f bf16
    state = w.B * H * dv * dk * 4
    alpha = w.B * w.F * H * 4
    kvb = T * H * (dk + dv) * 2 + T * H * 4        # k, v, beta
    qo = T * H * dk * 2 + T * H * dv * 2           # q in, out
    f_contract = 2 * T * H * dk * (dk + dv)
    f_scan = 2 * items * dv * dk * dk
    f_out = 2 * T * H * dk * dv
    return {
        "k1_contract": {"bytes": kvb, "overhead_bytes": ws_a + ws_u, "flops": f_contract},
        "k2_scan": {"bytes": alpha + 2 * state, "overhead_bytes": ws_a + ws_u + ws_s, "flops": f_scan},
        "k3_output": {"bytes": qo, "overhead_bytes": ws_s, "flops": f_out},
        # scan and output pass in one launch: the per-frame states stay on
        # chip / in L2; A_f and U_f are read back from the workspace
        "k23_scan_output": {"bytes": qo + alpha + 2 * state, "overhead_bytes": ws_a + ws_u,
                            "flops": f_scan + f_out},
        # the whole pass in one launch: every byte is compulsory
        "fwd_single_pass": {"bytes": kvb + qo + alpha + 2 * state, "overhead_bytes": 0,
                            "flops": f_contract + f_scan + f_out},
    }


def path_floor_bytes(w, in_bytes=2):
    """Compulsory HBM bytes of the whole forward: q, k, v read (in_bytes per
    element: 2 bf16, 1 fp8), out written (bf16), beta, alpha, state."""
    T = w.B * w.F * w.N
    return (T * w.H * (2 * w.dk + w.dv) * in_bytes + T * w.H * w.dv * 2 + T * w.H * 4 + w.B * w.F * w.H * 4
            + w.B * w.H * w.dv * w.dk * 4)


# the sources the forward pass's kernels (the single pass and the multi-launch
# schedule) are built from;
# the step and backward kernels live in files of their own, and the one-launch
# step's host launcher is cut out of gdn_api.cu before hashing
FORWARD_SOURCES = ("gdn_api.cu", "gdn_fwd_single.cuh", "gdn_scan_head.cuh", "gdn_k1_contract.cuh", "gdn_k1_pair.cuh",
                   "gdn_k23_fused.cuh", "gdn_k2_scan.cuh", "gdn_k3_output.cuh", "gdn_ptx.cuh")


def forward_part(name, text):
    if name == "gdn_api.cu":
        i = text.find(b"gdn_status launch_step_fused(")
        j = text.find(b"\n}\n", i) if i >= 0 else -1
        if i >= 0 and j >= 0:
            text = text[:i] + text[j + 3:]
    return text


def kernel_source_sha(read=None):
    """Hash of the forward kernels' sources; `read(name)` returns a file's
    bytes (default: the working tree)."""
    d = os.path.join(ROOT, "frame_wise_gated_forward_b300", "csrc")
    read = read or (lambda f: open(os.path.join(d, f), "rb").read())
    h = hashlib.sha256()
    for f in FORWARD_SOURCES:
        h.update(forward_part(f, read(f)))
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """dram bytes per launch of `kernel` from the committed ncu summary, or None
    if absent or taken on a different kernel source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    d = json.load(open(PROFILE_TRAFFIC))
    if d.get("source_sha") != kernel_source_sha():
        return None
    k = d.get("kernels", {}).get(kernel)
    return None if k is None else k.get("dram_bytes_per_launch")


# The NVML sampler runs in a separate process (the plain ctypes NVML calls of
# the driver's libnvidia-ml, read-only queries) and hands its samples over only
# after the timed region: a sampling thread in this process takes the
# interpreter lock every half millisecond, which delayed the host's launch of
# the first timed step by ~0.1 ms.  The SM clock's maximum does not change
# while the process runs and its query takes about a millisecond (measured on
# B300), so it is read once before sampling starts.
_NVML_CHILD = r"""
import ctypes, select, sys, time
lib = ctypes.CDLL("libnvidia-ml.so.1")
if lib.nvmlInit_v2() != 0:
    print("ERR nvmlInit", flush=True); sys.exit(0)
h = ctypes.c_void_p()
pci, idx = sys.argv[1], int(sys.argv[2])
if not (pci != "-" and lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(pci.encode()), ctypes.byref(h)) == 0):
    if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) != 0:
        print("ERR no NVML handle", flush=True); sys.exit(0)
mx = ctypes.c_uint()
if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:
    print("ERR no max clock", flush=True); sys.exit(0)
print("READY", flush=True)
sm, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
out = []
while not select.select([sys.stdin], [], [], 0.0005)[0]:
    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, ctypes.byref(rs)):
        break
    if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)):
        pw.value = 0
    out.append("%.7f %d %d %d %d" % (time.perf_counter(), sm.value, mx.value, pw.value, rs.value))
print("\n".join(out), flush=True)
"""


class ClockSampler:
    """SM clock, max clock, power and throttle reasons of one GPU, polled
    through NVML about every half millisecond by a separate process, so that
    even a timed region of a few milliseconds holds samples.  Falls back to
    nvidia-smi at 100 ms when NVML cannot be loaded."""
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    REASON_BITS = {"hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20, "hw_thermal_slowdown": 0x40,
                   "sw_power_cap": 0x4}

    def __init__(self, gpu_index, pci_bus_id=None):
        self.pci_bus_id = pci_bus_id
        self.error = None
        g = str(gpu_index).strip()
        self.gpu_index = int(g) if g.isdigit() else 0
        self.samples = []          # (time, sm_mhz, max_mhz, power_w, set of reasons)
        self.thread = None
        self.proc = None
        self.nvml = None
        self.source = None

    def start(self):
        try:
            self.nvml = subprocess.Popen(
                [sys.executable, "-c", _NVML_CHILD, self.pci_bus_id or "-", str(self.gpu_index)],
                stdin=subprocess.PIPE, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self.nvml.stdout.readline().strip()
            if first == "READY":
                self.source = "nvml (separate process), ~0.5 ms"
                return
            self.error = first or "NVML sampler exited"
            self.nvml.wait(timeout=5)
        except (OSError, ValueError, subprocess.TimeoutExpired) as e:
            self.error = f"{type(e).__name__}: {e}"
        self.nvml = None
        fields = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={fields}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            return
        self.source = "nvidia-smi, 100 ms"

        def read():
            for line in self.proc.stdout:
                p = [x.strip() for x in line.split(",")]
                if len(p) == 7:
                    try:
                        self.samples.append((time.perf_counter(), float(p[0]), float(p[1]), float(p[2]),
                                             {n for n, x in zip(self.NAMES, p[3:]) if x.lower() == "active"}))
                    except ValueError:
                        pass
        self.thread = threading.Thread(target=read, daemon=True)
        self.thread.start()

    def stop(self):
        if self.nvml is not None:
            try:
                out, _ = self.nvml.communicate(input="stop\n", timeout=10)
            except subprocess.TimeoutExpired:
                self.nvml.kill()
                out = ""
            for line in out.splitlines():
                p = line.split()
                if len(p) == 5:
                    rs = int(p[4])
                    self.samples.append((float(p[0]), float(p[1]), float(p[2]), int(p[3]) / 1000.0,
                                         {n for n, b in self.REASON_BITS.items() if rs & b}))
            self.nvml = None
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        """Samples taken inside [t0, t1] only; says so when there are none."""
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            r = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples_in_region": 0,
                 "source": self.source, "note": "no clock sample fell inside the timed region"}
            if self.error:
                r["nvml_error"] = self.error
            return r
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": sorted(set().union(*(s[4] for s in inside))), "samples_in_region": len(inside),
                "power_w_max": max(s[3] for s in inside), "source": self.source}


def cpu_baseline_run(w, x, frames):
    """Time the fp64 oracle (as it stands) on the first `frames` frames of the workload."""
    import oracle
    sub = {k: (v[:, :frames].contiguous() if k != "state_in" else v) for k, v in x.items()}
    t0 = time.perf_counter()
    oracle.frame_forward(sub["q"], sub["k"], sub["v"], sub["alpha"], sub["beta"], sub["state_in"],
                         B=w.B, H=w.H, F=frames, N=w.N, dk=w.dk, dv=w.dv, want_out=True)
    dt = time.perf_counter() - t0
    return w.B * frames * w.N, dt, oracle.max_threads()


def workload_desc(w):
    """The workload's name and shape, the same string on both arms."""
    return (f"{w.name}: 60 s 720p latent sequence, B={w.B} H={w.H} F={w.F} N={w.N} "
            f"dk={w.dk} dv={w.dv}, bf16 q/k/v/out, fp32 alpha/beta/state")


def run_reference(args, w):
    """--impl reference: the fp64 CPU oracle on a bounded sample of the workload per step."""
    from frame_wise_gated_forward_b300 import inputs, replicas
    rank, _, world = replicas.env_world()
    if rank != 0:
        return
    import oracle
    x = inputs.workload_inputs(w)
    # calibrate: one frame, then size the per-step sample to the budget
    _, t1, cores = cpu_baseline_run(w, x, 1)
    per_step = args.reference_budget_s / max(1, args.steps + args.warmup)
    frames = int(max(1, min(w.F, per_step / max(t1, 1e-6))))
    for _ in range(args.warmup):
        cpu_baseline_run(w, x, frames)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cpu_baseline_run(w, x, frames)
    dt = time.perf_counter() - t0
    tokens = w.B * frames * w.N
    value = tokens * args.steps / dt
    sample = f"first {frames} of {w.F} latent frames ({tokens} tokens x {w.H} heads, all outputs) per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_desc(w), "tokens_per_step_per_gpu": tokens,
                                        "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    import torch

    from frame_wise_gated_forward_b300 import inputs, replicas
    w = inputs.WORKLOADS[WORKLOAD]
    if args.impl == "reference":
        run_reference(args, w)
        return

    from frame_wise_gated_forward_b300 import api, build
    rank, local_rank, world = replicas.env_world()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    replicas.init("nccl")
    build.build()
    peaks = load_peaks()

    x = inputs.workload_inputs(w)
    xd = {k: v.to(device) for k, v in x.items()}
    zero_state = inputs.has_zero_state(w)
    s_in = None if zero_state else xd["state_in"]
    out = torch.empty((w.B, w.F, w.N, w.H, w.dv), dtype=torch.bfloat16, device=device)
    st = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        api.frame_forward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in, out=out, state_out=st)

    # the clock sampler starts before the warm-up, so that the GPU goes from the
    # warm-up steps straight into the timed ones (an idle pause in between lets
    # the clocks drop, and the first timed steps would pay for the ramp)
    cvd = [c for c in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if c.strip()]
    props = torch.cuda.get_device_properties(device)
    pci = None
    if hasattr(props, "pci_bus_id"):
        pci = f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"
    sampler = ClockSampler(cvd[local_rank].strip() if local_rank < len(cvd) else local_rank, pci)
    sampler.start()
    time.sleep(0.3)
    for _ in range(max(3, args.warmup)):
        step()
    api.sync_status()

    # ---------------------------------------------------------------- timed region
    torch.cuda.synchronize(device)
    replicas.barrier(device)
    torch.cuda.synchronize(device)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    tw0 = time.perf_counter()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    tw1 = time.perf_counter()
    replicas.barrier(device)
    torch.cuda.synchronize(device)
    sampler.stop()
    api.sync_status()
    sec = e0.elapsed_time(e1) / 1e3
    sec_max = replicas.max_over_ranks(sec, device)
    tokens = w.tokens
    value = replicas.throughput(tokens, args.steps, sec_max, world)
    clocks = sampler.summary(tw0, tw1)

    # ------------------------------------------------ per-kernel event timing
    nk = min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nk)]
    for row in evs:
        for e in row:
            e.record(stream)  # materialise the CUDA event handles
    torch.cuda.synchronize(device)
    for i in range(nk):
        api.frame_forward_timed(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in, out, st, evs[i])
    torch.cuda.synchronize(device)
    api.sync_status()
    fsched = api.forward_schedule(w.B, w.H, w.F, w.N, w.dk, w.dv)
    sched = api.scan_schedule(w.B, w.H, w.dv)
    names = {2: ["counters_reset", "none", "fwd_single_pass"],
             1: ["k1_contract", "flags_reset", "k23_scan_output"]}.get(fsched, ["k1_contract", "k2_scan", "k3_output"])
    phase_ms = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(nk))
                for j, n in enumerate(names)}
    costs = kernel_costs(w)
    names = [n for n in names if n in costs]
    phases = {}
    for n in names:
        t = phase_ms[n] / 1e3
        phases[n] = {"ms": phase_ms[n], "GB/s": costs[n]["bytes"] / t / 1e9,
                     "overhead_bytes": costs[n]["overhead_bytes"],
                     "hbm_frac": costs[n]["bytes"] / t / 1e9 / peaks["hbm_gbs"],
                     "TFLOP/s": costs[n]["flops"] / t / 1e12,
                     "tensor_frac": costs[n]["flops"] / t / 1e12 / peaks["bf16_tflops"]}
    dom = max(names, key=lambda n: phase_ms[n])
    achieved = costs[dom]["bytes"] / (phase_ms[dom] / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(dom), "kernel": dom,
                "peak_source": peaks["source"], "algorithmic_bytes": costs[dom]["bytes"],
                "overhead_bytes": costs[dom]["overhead_bytes"]}
    ms_per_step = sec_max / args.steps * 1e3
    floor_ms = path_floor_bytes(w) / (peaks["hbm_gbs"] * 1e9) * 1e3

    # ------------------------ the same pass in the multi-launch schedule (context)
    nr = min(args.steps, 100)
    r0 = torch.cuda.Event(enable_timing=True)
    r1 = torch.cuda.Event(enable_timing=True)
    api.set_single_pass(False)
    try:
        step()
        torch.cuda.synchronize(device)
        r0.record(stream)
        for _ in range(nr):
            step()
        r1.record(stream)
        torch.cuda.synchronize(device)
        api.sync_status()
    finally:
        api.set_single_pass(True)
    multi_ms = r0.elapsed_time(r1) / nr
    multi_info = {"ms_per_step": multi_ms, "tokens_per_s": tokens / (multi_ms / 1e3), "steps": nr,
                  "what": "phase 1, then scan and output in one cooperative launch (A_f, U_f and the "
                          "per-frame states through HBM)"}

    # ------------------------------------- reverse direction (bidirectional stage)
    api.frame_forward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in, out=out, state_out=st, reverse=True)
    torch.cuda.synchronize(device)
    r0.record(stream)
    for _ in range(nr):
        api.frame_forward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in, out=out, state_out=st,
                          reverse=True)
    r1.record(stream)
    torch.cuda.synchronize(device)
    api.sync_status()
    rev_ms = r0.elapsed_time(r1) / nr
    reverse_info = {"ms_per_step": rev_ms, "tokens_per_s": tokens / (rev_ms / 1e3), "steps": nr}

    # ------------------------------- folded prologue (raw q, k and gate logits)
    xr = {k: v.to(device) for k, v in inputs.draw_raw(w.B, w.H, w.F, w.N, w.dk, w.dv, seed=0).items()}
    api.frame_forward_gated(xr["q"], xr["k"], xr["v"], xr["a_logit"], xr["b_logit"], 0.05, None,
                            out=out, state_out=st)
    torch.cuda.synchronize(device)
    r0.record(stream)
    for _ in range(nr):
        api.frame_forward_gated(xr["q"], xr["k"], xr["v"], xr["a_logit"], xr["b_logit"], 0.05, None,
                                out=out, state_out=st)
    r1.record(stream)
    torch.cuda.synchronize(device)
    api.sync_status()
    gated_ms = r0.elapsed_time(r1) / nr
    gated_info = {"ms_per_step": gated_ms, "tokens_per_s": tokens / (gated_ms / 1e3), "steps": nr,
                  "what": "raw q, k L2-normalized and sigmoid/softplus gates applied inside the kernels"}
    del xr

    # ------------------------------------------ 8-bit inputs (e4m3 q, k, v)
    x8 = {k: (v.to(device) if torch.is_tensor(v) else v)
          for k, v in inputs.draw_fp8(w.B, w.H, w.F, w.N, w.dk, w.dv, seed=0).items()}

    def step8():
        api.frame_forward_fp8(x8["q8"], x8["k8"], x8["v8"], x8["q_scale"], x8["k_scale"], x8["v_scale"],
                              x8["alpha"], x8["beta"], None, out=out, state_out=st)
    step8()
    torch.cuda.synchronize(device)
    r0.record(stream)
    for _ in range(nr):
        step8()
    r1.record(stream)
    torch.cuda.synchronize(device)
    api.sync_status()
    fp8_ms = r0.elapsed_time(r1) / nr
    fp8_floor_ms = path_floor_bytes(w, in_bytes=1) / (peaks["hbm_gbs"] * 1e9) * 1e3
    fp8_info = {"ms_per_step": fp8_ms, "tokens_per_s": tokens / (fp8_ms / 1e3), "steps": nr,
                "path_floor_ms": fp8_floor_ms, "path_frac": fp8_floor_ms / fp8_ms,
                "what": "q, k, v as per-tensor-scaled OCP FP8 E4M3 (1 byte each), decoded in shared memory; "
                        "out bf16, state fp32"}
    del x8

    # ---------------------------------------------------------- NVFP4 inputs
    x4 = {k: (v.to(device) if torch.is_tensor(v) else v)
          for k, v in inputs.draw_nvfp4(w.B, w.H, w.F, w.N, w.dk, w.dv, seed=0).items()}

    def step4():
        api.frame_forward_nvfp4(x4["q4"], x4["k4"], x4["v4"], x4["q_sf"], x4["k_sf"], x4["v_sf"], x4["q_gs"],
                                x4["k_gs"], x4["v_gs"], x4["alpha"], x4["beta"], None, out=out, state_out=st)
    step4()
    torch.cuda.synchronize(device)
    r0.record(stream)
    for _ in range(nr):
        step4()
    r1.record(stream)
    torch.cuda.synchronize(device)
    api.sync_status()
    fp4_ms = r0.elapsed_time(r1) / nr
    T = w.B * w.F * w.N
    fp4_floor_ms = (T * w.H * (2 * w.dk + w.dv) * (0.5 + 1.0 / 16) + T * w.H * w.dv * 2 + T * w.H * 4
                    + w.B * w.F * w.H * 4 + w.B * w.H * w.dv * w.dk * 4) / (peaks["hbm_gbs"] * 1e9) * 1e3
    fp4_info = {"ms_per_step": fp4_ms, "tokens_per_s": tokens / (fp4_ms / 1e3), "steps": nr,
                "path_floor_ms": fp4_floor_ms, "path_frac": fp4_floor_ms / fp4_ms,
                "what": "q, k, v as NVFP4 (E2M1 codes, E4M3 scale per 16, fp32 scale per tensor), decoded in "
                        "shared memory; out bf16, state fp32"}
    del x4

    # ------------------------------------------------------- backward (training)
    g = torch.Generator().manual_seed(1)
    d_out = torch.randn(out.shape, generator=g).to(torch.bfloat16).to(device)
    api.frame_backward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in, d_out)
    torch.cuda.synchronize(device)
    nb = min(args.steps, 20)
    r0.record(stream)
    for _ in range(nb):
        api.frame_backward(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in, d_out)
    r1.record(stream)
    torch.cuda.synchronize(device)
    api.sync_status()
    bwd_ms = r0.elapsed_time(r1) / nb
    # compulsory bytes: q, k, v, d_out, beta read; dq, dk, dv, d_beta written (bf16 / fp32)
    bwd_bytes = tokens * w.H * ((2 * w.dk + 2 * w.dv) * 2 + (2 * w.dk + w.dv) * 2 + 8)
    # the same gradients from the activations a training forward keeps (no recompute)
    _, _, sa, ss = api.frame_forward_save(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in)
    torch.cuda.synchronize(device)
    r0.record(stream)
    for _ in range(nb):
        api.frame_forward_save(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in, out=out, state_out=st,
                               saved_A=sa, saved_S=ss)
    r1.record(stream)
    torch.cuda.synchronize(device)
    fwd_save_ms = r0.elapsed_time(r1) / nb
    api.frame_backward_saved(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in, sa, ss, d_out)
    torch.cuda.synchronize(device)
    r0.record(stream)
    for _ in range(nb):
        api.frame_backward_saved(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], s_in, sa, ss, d_out)
    r1.record(stream)
    torch.cuda.synchronize(device)
    api.sync_status()
    bwd_saved_ms = r0.elapsed_time(r1) / nb
    backward_info = {"ms_per_step": bwd_ms, "tokens_per_s": tokens / (bwd_ms / 1e3), "steps": nb,
                     "path_floor_ms": bwd_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3,
                     "what": "gdn_frame_backward: dq, dk, dv, dalpha, dbeta, dS0 for upstream dO (forward states "
                             "recomputed)",
                     "from_saved_activations": {
                         "backward_ms": bwd_saved_ms, "forward_save_ms": fwd_save_ms,
                         "saved_bytes": sa.numel() * 2 + ss.numel() * 2,
                         "what": "gdn_frame_forward_save keeps A_f and the per-frame bf16 states; "
                                 "gdn_frame_backward_saved skips their recompute (bit-identical gradients)"}}
    del d_out, sa, ss

    # ------------------------------------------- interactive step (one frame)
    # the streaming rollout: F sequential gdn_frame_step calls on a resident state
    step_state = torch.zeros((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=device)
    step_out = torch.empty((w.B, w.N, w.H, w.dv), dtype=torch.bfloat16, device=device)
    frames = [tuple(xd[k][:, f].contiguous() for k in ("q", "k", "v", "alpha", "beta")) for f in range(w.F)]
    for f in range(3):
        api.frame_step(*frames[f], step_state, out=step_out, state_out=step_state)
    torch.cuda.synchronize(device)
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for f in range(w.F):
        api.frame_step(*frames[f], step_state, out=step_out, state_out=step_state)
    s1.record(stream)
    torch.cuda.synchronize(device)
    api.sync_status()
    step_us = s0.elapsed_time(s1) * 1e3 / w.F
    step_info = {"us_per_frame_step": step_us, "tokens_per_s": w.B * w.N / (step_us / 1e6),
                 "launches_per_step": 1, "memsets_per_step": 0, "frames": w.F,
                 "kernel": "one-launch step (one 4-CTA cluster per head, default)",
                 "floor_us": (w.B * w.N * w.H * (2 * w.dk + 2 * w.dv) * 2 + 2 * w.B * w.H * w.dv * w.dk * 4)
                 / (peaks["hbm_gbs"] * 1e9) * 1e6}
    del frames

    # ---------------------------------------------------------------------- e2e
    hx = {k: v.pin_memory() for k, v in x.items()}
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h_st = torch.empty(st.shape, dtype=st.dtype, pin_memory=True)
    hs_in = None if zero_state else hx["state_in"]
    api.frame_forward_host(hx["q"], hx["k"], hx["v"], hx["alpha"], hx["beta"], hs_in, out=h_out, state_out=h_st)
    torch.cuda.synchronize(device)
    replicas.barrier(device)
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.e2e_steps):
        api.frame_forward_host(hx["q"], hx["k"], hx["v"], hx["alpha"], hx["beta"], hs_in,
                               out=h_out, state_out=h_st)
    g1.record(stream)
    torch.cuda.synchronize(device)
    e2e_sec = replicas.max_over_ranks(g0.elapsed_time(g1) / 1e3, device)
    e2e_value = replicas.throughput(tokens, args.e2e_steps, e2e_sec, world)
    h2d = sum(hx[k].numel() * hx[k].element_size() for k in ("q", "k", "v", "alpha", "beta"))
    if hs_in is not None:
        h2d += hs_in.numel() * hs_in.element_size()
    d2h = h_out.numel() * h_out.element_size() + h_st.numel() * h_st.element_size()

    # -------------------------------------------------------- CPU baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_tok, dt, cores = cpu_baseline_run(w, x, w.F)
        cpu = {"value": n_tok / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"full {w.name} workload ({n_tok} tokens x {w.H} heads, all outputs), one pass, fp64"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(w),
                       "tokens_per_step_per_gpu": tokens,
                       "l2": "inputs 1.31 GB per step > 126 MB L2; no flush",
                       "parallelism": f"replicas x{world} (no data-path collective)",
                       "schedule": ("single pass: contraction, scan (one CTA per head) and output in one "
                                    "cooperative launch, L2-resident rings" if fsched == 2 else
                                    f"phase 1, then fused scan+output ({sched} state rows per scan CTA)" if fsched == 1
                                    else f"three launches ({-sched} state rows per scan CTA)")},
            "roofline": roofline,
            "phases": phases,
            "path_roofline": {"floor_ms": floor_ms, "frac": floor_ms / ms_per_step,
                              "ceiling_tokens_per_s": tokens / (floor_ms / 1e3) * world},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": args.e2e_steps},
            "multi_launch_schedule": multi_info,
            "step": step_info,
            "reverse_direction": reverse_info,
            "gated_prologue": gated_info,
            "fp8_inputs": fp8_info,
            "nvfp4_inputs": fp4_info,
            "backward": backward_info,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "gpu_launches": {2: 1, 1: 2}.get(fsched, 3) * args.steps,
        }
        print(json.dumps(line), flush=True)
    replicas.shutdown()


if __name__ == "__main__":
    main()
