"""Host logic of bench.py that needs no GPU: the source hash that keys the
recorded ncu DRAM traffic to the forward kernels as built, and the lookup of
that record."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402

CSRC = os.path.join(ROOT, "frame_wise_gated_forward_b300", "csrc")


def _tree(name):
    return open(os.path.join(CSRC, name), "rb").read()


def test_step_launcher_is_cut_out_of_the_api_source():
    api = _tree("gdn_api.cu")
    cut = bench.forward_part("gdn_api.cu", api)
    assert b"gdn_status launch_step_fused(" in api
    assert b"gdn_status launch_step_fused(" not in cut
    # only that one function goes: the forward's launch code stays
    assert b"launch_phases" in cut and b"plan_split" in cut
    assert len(api) - len(cut) < 4000
    # other files pass through unchanged
    k23 = _tree("gdn_k23_fused.cuh")
    assert bench.forward_part("gdn_k23_fused.cuh", k23) == k23


def test_hash_ignores_the_step_launcher_but_not_the_forward_sources():
    base = bench.kernel_source_sha()

    def edited(target, old, new):
        def read(f):
            t = _tree(f)
            if f == target:
                assert old in t
                t = t.replace(old, new, 1)
            return t
        return read

    # a change inside the step launcher leaves the hash alone
    same = bench.kernel_source_sha(edited("gdn_api.cu", b"gdn_status launch_step_fused(const PassArgs& a",
                                          b"gdn_status launch_step_fused(const PassArgs&  a"))
    assert same == base
    # a change to a forward kernel, the shared PTX header or the forward's
    # launch code changes it
    for f in ("gdn_fwd_single.cuh", "gdn_scan_head.cuh", "gdn_k1_contract.cuh", "gdn_k1_pair.cuh", "gdn_k3_output.cuh",
              "gdn_ptx.cuh"):
        assert bench.kernel_source_sha(edited(f, b"#pragma once", b"#pragma  once")) != base
    assert bench.kernel_source_sha(edited("gdn_api.cu", b"launch_phases(", b"launch_phases (")) != base
    # the step and backward kernels' files are not part of it
    assert "gdn_step_fused.cuh" not in bench.FORWARD_SOURCES and "gdn_bwd.cuh" not in bench.FORWARD_SOURCES


def test_traffic_lookup_checks_the_hash(tmp_path, monkeypatch):
    rec = {"source_sha": bench.kernel_source_sha(),
           "kernels": {"k23_scan_output": {"dram_bytes_per_launch": 123}}}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(p))
    assert bench.ncu_traffic("k23_scan_output") == 123
    assert bench.ncu_traffic("k1_contract") is None
    rec["source_sha"] = "0" * 16
    p.write_text(json.dumps(rec))
    assert bench.ncu_traffic("k23_scan_output") is None
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(tmp_path / "absent.json"))
    assert bench.ncu_traffic("k23_scan_output") is None


def test_clock_sampler_reads_the_sampling_process(monkeypatch):
    """The NVML samples come from a separate process that hands them over at
    stop(); their reason bits map to the names the timing rules use and only
    samples inside the timed region are summarised."""
    lines = ["10.0000000 1900 2032 400000 0", "10.5000000 2032 2032 500000 4", "11.5000000 2032 2032 510000 32"]

    class FakeChild:
        def __init__(self, *a, **k):
            import io
            self.stdout = io.StringIO("READY\n")

        def communicate(self, input=None, timeout=None):
            assert input is not None
            return "\n".join(lines) + "\n", ""

        def wait(self, timeout=None):
            return 0

        def kill(self):
            pass

    monkeypatch.setattr(bench.subprocess, "Popen", FakeChild)
    s = bench.ClockSampler(0, None)
    s.start()
    assert s.source.startswith("nvml")
    s.stop()
    assert len(s.samples) == 3
    r = s.summary(10.2, 11.0)   # only the sample at 10.5 s
    assert r["samples_in_region"] == 1 and r["sm_mhz"] == 2032.0 and r["reasons"] == ["sw_power_cap"]
    r = s.summary(9.0, 12.0)
    assert r["samples_in_region"] == 3 and r["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    assert bench.ClockSampler(0).summary(0.0, 1.0)["samples_in_region"] == 0
