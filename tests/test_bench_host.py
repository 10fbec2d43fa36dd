"""bench.py's host-side bookkeeping without a GPU: the committed ncu traffic summaries are reported only for the
kernel source, plan and weight layout they were captured on."""
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_decode_traffic_record_matches_its_plan_only():
    rec = bench.recorded_traffic("decode", fused=True, tiled=True)
    assert rec is not None and len(rec) == 4 and all(v > 0 for v in rec)
    # the capture covers the fused launch on tile-contiguous weights: other plans get no traffic figure
    assert bench.recorded_traffic("decode", fused=True, tiled=False) is None
    assert bench.recorded_traffic("decode", fused=False, tiled=True) is None
    assert bench.recorded_traffic("prefill", fused=False, tiled=False) is None


def test_config_traffic_records_match_their_plans_only():
    # one record per configuration the bench times on a kernel it has a record for: the tiled GEMM 1 of each
    for name in ("prefill", "mxfp8", "mxfp8_act", "batched", "batched_tokens"):
        rec = bench.recorded_traffic(name, fused=False, tiled=True)
        assert rec is not None and len(rec) == 1 and rec[0] > 0, name
        assert bench.recorded_traffic(name, fused=False, tiled=False) is None, name
        assert bench.recorded_traffic(name, fused=True, tiled=True) is None, name
    assert bench.recorded_traffic("tiny", fused=False, tiled=False) is None


def _copy_with_gemm_tc(tmp_path, monkeypatch, extra):
    # a copy of the repository layout whose gemm_tc.cu has `extra` appended
    src = os.path.join(ROOT, "mixture_experts_layer_permute_gb300", "csrc", "gemm_tc.cu")
    csrc = tmp_path / "mixture_experts_layer_permute_gb300" / "csrc"
    csrc.mkdir(parents=True)
    with open(src, "rb") as f:
        (csrc / "gemm_tc.cu").write_bytes(f.read() + extra)
    shutil.copytree(os.path.join(ROOT, "profiles"), tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))


def test_traffic_record_dropped_when_the_kernel_code_changes(tmp_path, monkeypatch):
    _copy_with_gemm_tc(tmp_path, monkeypatch, b"static int moe_extra_symbol;\n")
    assert bench.recorded_traffic("decode", fused=True, tiled=True) is None


def test_traffic_record_kept_across_comment_edits(tmp_path, monkeypatch):
    _copy_with_gemm_tc(tmp_path, monkeypatch, b"\n// a remark\n/* and a block\n   comment */\n\n")
    assert bench.recorded_traffic("decode", fused=True, tiled=True) is not None


def test_describe_names_the_workload():
    ws = bench.workload_list("decode")
    assert [w.T for w in ws] == [1, 8, 32, 64]
    assert "decode" in bench.describe("decode", ws)
    assert "prefill" in bench.describe("prefill", bench.workload_list("prefill"))
