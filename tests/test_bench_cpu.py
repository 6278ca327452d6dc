"""Host logic of bench.py (CPU only): the L2 note each workload's line
carries, the tie between the committed DRAM counters and the kernel source,
and the config object."""
import os
import shutil

import bench
from decode_kv_cache_step_gb300.workloads import WORKLOADS


def test_l2_note_says_whether_the_caches_fit():
    assert bench.l2_note(WORKLOADS["qwen3_8b_b128_s3200"]).startswith("inputs larger than L2")
    assert bench.l2_note(WORKLOADS["long_b32_s16384_ragged"]).startswith("inputs larger than L2")
    tiny = WORKLOADS["tiny_b2_s256"]
    assert bench.l2_note(tiny).startswith("inputs fit in L2")
    assert bench.l2_note(tiny, 32).startswith("inputs fit in L2")      # 8 MiB: still in L2
    assert "stepped in turn" in bench.l2_note(tiny, 600)                # 150 MiB
    assert "stepped in turn" in bench.l2_note(WORKLOADS["qwen3_8b_b1_s2400"], 32)


def test_workload_config_keys():
    wl = WORKLOADS["qwen3_8b_b1_s2400"]
    cfg = bench.workload_config(wl, 1, 1, plan={"nchunk": 8})
    for key in ("workload", "layers", "B", "Hq", "Hkv", "d", "S", "W", "l2", "parallelism"):
        assert key in cfg
    assert cfg["workload"] == wl.name and cfg["launch_plan"] == {"nchunk": 8}
    assert "launch_plan" not in bench.workload_config(wl, 2)


def _copy_sources(tmp_path):
    root = tmp_path / "repo"
    csrc = root / "decode_kv_cache_step_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(bench.ROOT, "decode_kv_cache_step_gb300", "csrc", name), csrc)
    return root, csrc


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    root, csrc = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash()
    assert h0 == bench.kernel_source_hash()
    f = csrc / bench.KERNEL_SOURCES[0]
    f.write_text(f.read_text() + "\n// a comment\n/* and a\n block */\n\n")
    assert bench.kernel_source_hash() == h0
    f.write_text(f.read_text() + "\nstatic int lf_probe_symbol = 1;\n")
    assert bench.kernel_source_hash() != h0


def test_committed_traffic_only_for_the_same_source(tmp_path, monkeypatch):
    prof = tmp_path / "prof.md"
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(prof))
    assert bench.committed_traffic() is None                      # no summary
    prof.write_text(f"# x\n\nsource_sha: {bench.kernel_source_hash()}\n"
                    "traffic_bytes_per_launch: 123456\n")
    assert bench.committed_traffic() == 123456.0
    prof.write_text("source_sha: 0000000000000000\ntraffic_bytes_per_launch: 123456\n")
    assert bench.committed_traffic() is None                      # another kernel version
