"""Host-side helpers of bench.py: the algorithmic bytes behind the roofline, the
profile-traffic lookup that goes stale with its source, and the percentile."""
import hashlib
import os

import pytest

import bench
import synth


def test_step_bytes_of_the_7b_workload():
    """Per-stage algorithmic bytes at the Vicuna-7B shape: the heads read W1, b1, W2 and h
    and write and read u back; attention reads the cache and the tree's q/k/v and writes
    fp32 outputs; verification reads lm_head and X and writes one fp32 per node."""
    wl = synth.WORKLOADS["vicuna7b"]
    T = 65
    b = bench.step_bytes(wl, T)
    H, V, K, B = 4096, 32000, 5, 1
    assert b["heads"] == 2 * (K * H * H + K * H + K * V * H + B * H) + 2 * 2 * B * K * H == 1478623232
    L, Hkv, Hq, D = 2048, 32, 32, 128
    assert b["attention"] == 2 * (2 * L * Hkv * D + B * T * (Hq + 2 * Hkv) * D) + 4 * B * T * Hq * D
    assert b["verify"] == 2 * (V * H + B * T * H) + 4 * B * T
    assert sum(b.values()) == 1777516804


def test_profile_traffic_is_dropped_when_the_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    src.write_text("// some kernel\n")
    digest = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    prof = tmp_path / "profiles" / "k.md"
    prof.write_text(f"traffic_bytes_per_launch: 12345\nsource_file: kernel.cu\nsource_sha256: {digest}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile("k") == 12345.0
    src.write_text("// the kernel, changed\n")
    assert bench.traffic_from_profile("k") is None
    assert bench.traffic_from_profile("missing") is None


def test_committed_heads_profile_matches_its_source():
    """The heads summary under profiles/ was captured on the current heads.cu, so the
    bench's roofline reports its DRAM traffic (about the algorithmic bytes)."""
    t = bench.traffic_from_profile("heads_vicuna7b")
    assert t is not None
    assert 1.0 <= t / 1478623232 < 1.01


@pytest.mark.parametrize("q,want", [(50, 3), (99, 5), (0, 1), (100, 5)])
def test_percentile_nearest_rank(q, want):
    assert bench.pct([5, 1, 4, 2, 3], q) == want
