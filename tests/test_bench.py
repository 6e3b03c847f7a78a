"""bench.py's host logic on CPU (the kernel-source hash that voids a recorded
ncu traffic figure, the reference (oracle) arm's JSON line) and, on a GPU, its
end-to-end loop's outputs."""
import json
import os
import subprocess
import sys

import pytest

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


@pytest.mark.gpu
def test_end_to_end_loop_returns_the_decode_output():
    """bench.py's pipelined host-buffer loop: the outputs read back to host memory equal, bitwise,
    a direct decode of the same step's inputs (the copies and the two buffer sets are ordered)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_decode_v2_gb300 as pa
    import workloads as wl
    dec = bench.Decoder(wl.TINY, torch.device("cuda", 0))
    host_in = dec.pack_host_inputs()
    n = 5
    dec.e2e_steps(0, n, host_in)
    torch.cuda.synchronize()
    inp, w = dec.inp, dec.w
    S, H, D = inp.query.shape
    tmp, es, ml = pa.alloc_workspace(S, H, D, max(1, dec.np), device="cuda")
    for k in (n - 2, n - 1):
        kc, vc = dec.caches[k % dec.copies]
        ref = torch.empty_like(inp.query)
        pa.pa_decode(inp.query, kc, vc, inp.block_tables, inp.seq_lens, w.scale, w.partition_size,
                     ref, tmp, es, ml, max_seq_len_hint=dec.max_seq_len)
        torch.cuda.synchronize()
        assert torch.equal(dec.e2e_host_out[k % 2], ref.cpu())
