"""Host-side helpers of bench.py that feed the reported roofline numbers."""
import hashlib
import os
import shutil

import pytest

import bench
from sparse_rank_kv_gb300.synth import CONFIGS


def test_row_major_step_bytes_match_the_reported_figure():
    """Batch 8, 128K, local window 64 + 3 warm-up + (32 + 1) / 2 appended
    tokens on average: 361,742,336 bytes, the figure the benchmark line and the
    design notes quote for the pages' step."""
    cfg = CONFIGS["llama_b8_s128k"]
    n_loc = cfg.w + 3 + 33 / 2.0
    assert bench.hbm_bytes_per_step(cfg, 2, n_loc) == pytest.approx(361_742_336)


def test_record_step_bytes_follow_the_hit_rate():
    """With K/V records every selected chunk's keys and values are read, and
    only the missed chunks cost A rows plus the writes of their rebuilt keys
    and fetched values: the bytes fall linearly with the hit rate, by
    k c (r + 2 d) elements per (batch, KV head) between no hits and all hits."""
    cfg = CONFIGS["llama_b8_s128k"]
    E, n_loc = 2, 80.0
    full = bench.hbm_bytes_per_step(cfg, E, n_loc, alpha=0.0, records=True)
    none = bench.hbm_bytes_per_step(cfg, E, n_loc, alpha=1.0, records=True)
    half = bench.hbm_bytes_per_step(cfg, E, n_loc, alpha=0.5, records=True)
    span = E * cfg.b * cfg.h_kv * cfg.k * cfg.c * (cfg.r + 2 * cfg.d)
    assert full - none == pytest.approx(span)
    assert half == pytest.approx((full + none) / 2)
    # all hits: the landmarks, B, outliers, local window and the selected
    # chunks' cached keys and values, nothing else
    sel = cfg.k * cfg.c
    want = E * cfg.b * cfg.h_kv * (cfg.n * cfg.d + cfg.r * cfg.d + 2 * cfg.o * cfg.c * cfg.d
                                   + 2 * n_loc * cfg.d + 2 * sel * cfg.d)
    assert none == pytest.approx(want)


def _profile_tree(tmp_path, sha):
    src = os.path.join(bench.ROOT, "sparse_rank_kv_gb300", "csrc", "score_tc.cu")
    os.makedirs(tmp_path / "profiles")
    os.makedirs(tmp_path / "sparse_rank_kv_gb300" / "csrc")
    shutil.copy(src, tmp_path / "sparse_rank_kv_gb300" / "csrc" / "score_tc.cu")
    (tmp_path / "profiles" / "p.md").write_text(
        "# summary\n\n- source_file: sparse_rank_kv_gb300/csrc/score_tc.cu\n"
        f"- source_sha256: {sha}\n- dram_bytes_per_launch: 1234567\n")
    return src


def test_profile_traffic_is_used_only_for_the_profiled_source(tmp_path, monkeypatch):
    src = _profile_tree(tmp_path, "0" * 16)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile("p.md", "score_tc.cu") is None   # source changed since
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    (tmp_path / "profiles" / "p.md").write_text(
        "- source_sha256: %s\n- dram_bytes_per_launch: 1234567\n" % sha)
    assert bench.traffic_from_profile("p.md", "score_tc.cu") == 1234567.0
    assert bench.traffic_from_profile("missing.md", "score_tc.cu") is None
