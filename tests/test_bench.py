"""bench.py's host logic on CPU: the kernel-source hash that voids a recorded
ncu traffic figure, and the reference (oracle) arm's JSON line."""
import json
import os
import subprocess
import sys

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_code_only_ignores_comments_and_layout():
    a = "int a; // one\n/* two\n lines */ int  b;\n"
    b = "int a;\nint b; // other comment\n"
    assert bench._code_only(a) == bench._code_only(b) == "int a; int b;"
    assert bench._code_only("int a = 1;") != bench._code_only("int a = 2;")


def test_kernel_source_hashes_cover_both_kernel_families():
    h_attn = bench.kernel_source_hash("pa_attn")
    h_tc = bench.kernel_source_hash("pa_tc")
    assert len(h_attn) == len(h_tc) == 16 and h_attn != h_tc


def test_recorded_traffic_needs_a_matching_source_hash(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    rec = {"pa_attn_v2_phase1/demo": {"dram_bytes_per_launch": 123,
                                      "source_hash": bench.kernel_source_hash("pa_attn")},
           "pa_tc_v1/demo": {"dram_bytes_per_launch": 456, "source_hash": "0" * 16}}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES",
                        {k: [os.path.join(ROOT, f) for f in v] for k, v in bench.KERNEL_SOURCES.items()})
    assert bench.recorded_traffic("demo", "pa_attn_v2_phase1") == 123
    assert bench.recorded_traffic("demo", "pa_tc_v1") is None   # kernel changed since
    assert bench.recorded_traffic("other", "pa_attn_v2_phase1") is None


def test_reference_arm_prints_one_json_line():
    """`bench.py --impl reference` times the fp64 oracle on the host and prints the
    contract's line (rank 0, no GPU needed)."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
