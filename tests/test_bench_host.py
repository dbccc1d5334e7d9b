"""Host-side pieces of the benchmark's report (CPU only): the committed DRAM
records are used only while the kernel source they were taken on is
unchanged, the per-kernel flop counts add up to the layer's, and the peaks
come from the measured file when it is there."""
import json
import os
import shutil

import bench

REPO = bench.ROOT


def _copy_tree(tmp_path, kernel):
    rec_src = os.path.join(REPO, "profiles", f"{kernel}_{bench.WORKLOAD}.json")
    with open(rec_src) as f:
        rec = json.load(f)
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "kv_cache_compaction_gb300" / "csrc"
    csrc.mkdir(parents=True)
    shutil.copy(rec_src, tmp_path / "profiles")
    shutil.copy(os.path.join(REPO, "kv_cache_compaction_gb300", "csrc", rec["source"]), csrc)
    return rec, csrc / rec["source"]


def test_traffic_record_follows_the_source(tmp_path, monkeypatch):
    for kernel in ("attn_stats", "key_scores"):
        sub = tmp_path / kernel
        sub.mkdir()
        rec, src = _copy_tree(sub, kernel)
        monkeypatch.setattr(bench, "ROOT", str(sub))
        assert bench.traffic_for(kernel) == rec["dram_bytes_per_launch"]
        assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        with open(src, "a") as f:
            f.write("\n// changed\n")
        assert bench.traffic_for(kernel) is None
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "nowhere"))
    assert bench.traffic_for("attn_stats") is None


def test_layer_flops_are_the_sum_of_the_kernels():
    w = bench.workload()
    fl = bench.flops(w)
    parts = fl["attn_stats"] + fl["key_scores"] + fl["gram_mass"] + fl["gram_out"]
    assert abs(fl["layer"] - parts) <= 1e-9 * fl["layer"]
    # pass 1 multiplies twice (S and P.V) what pass 2 does (S only)
    assert fl["attn_stats"] == 2 * fl["key_scores"]


def test_peaks_come_from_the_measured_file():
    p = bench.peaks()
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        assert p["source"] == "measured"
        assert p["hbm_gbs"] == m["hbm_gbs"] and p["bf16_tflops"] == m["bf16_tflops"]
    else:
        assert p["source"] == "fallback"
