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
