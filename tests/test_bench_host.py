"""Host-side checks of the benchmark's bookkeeping (no GPU): the algorithmic byte and flop
counts the roofline divides by, the visible-pair count of the chunked-limited window, and
the rule that a committed profile's DRAM traffic is reported only for the kernel source it
was taken on."""
from __future__ import annotations

import os

import numpy as np
import pytest

import bench
from paged_kv_chunk_gb300 import synthetic as syn


def test_step_bytes_of_the_small_cohort():
    """Conformer-small (B 64, T 16, H 4, D 64, C 256, R 287, bf16), counted by hand: the
    chunk's K and V read and written (4 x 524288), the cached K/V read (2 x 64 x 256 x 512),
    q read and out written (2 x 524288), the rel table once (287 x 512)."""
    chunk = 64 * 16 * 4 * 64 * 2
    fused = 4 * chunk + 2 * 64 * 256 * 4 * 64 * 2 + 2 * chunk + 287 * 4 * 64 * 2
    assert fused == 20_069_888
    assert bench.workload_bytes(syn.SMALL) == fused
    assert bench.workload_bytes(syn.SMALL, fused=False) == fused + 2 * chunk


def test_step_bytes_of_a_heterogeneous_cohort_follow_each_cache_length():
    cfg = syn.HETERO
    Cs = syn.cache_lengths(cfg)
    assert len(set(Cs.tolist())) > 1
    row = cfg.H * cfg.D * 2
    chunk = cfg.B * cfg.T * row
    expect = 6 * chunk + 2 * int(Cs.sum()) * row + cfg.R * row
    assert bench.workload_bytes(cfg) == expect


@pytest.mark.parametrize("cs,left", [(1, 0), (3, 2), (8, 7), (5, 0), (50, 3)])
def test_chunked_pairs_against_brute_force(cs, left):
    lengths = [0, 1, 7, 16, 23, 64, 101]
    brute = 0
    for L in lengths:
        for i in range(L):
            for j in range(L):
                if i // cs - left <= j // cs <= i // cs:
                    brute += 1
    assert bench.chunked_pairs(lengths, cs, left) == brute


def test_packed_flops_count_three_products_per_pair():
    lengths = [3, 0, 5]
    H, D = 2, 64
    pairs = sum(L * L for L in lengths)
    assert bench.packed_flops(lengths, H, D) == pairs * H * 3 * 2 * D


def _fake_tree(tmp_path, text):
    d = tmp_path / "paged_kv_chunk_gb300" / "csrc"
    d.mkdir(parents=True)
    (d / "k.cu").write_text(text)
    (tmp_path / "profiles").mkdir()
    return tmp_path


def test_source_digest_ignores_comments_and_spacing(tmp_path, monkeypatch):
    root = _fake_tree(tmp_path, "int f(int x) { return x + 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    base = bench.source_digest(["k.cu"])
    (root / "paged_kv_chunk_gb300" / "csrc" / "k.cu").write_text(
        "// a comment\nint f(int x)\n{\n    /* block */ return x + 1;   // why\n}\n")
    assert bench.source_digest(["k.cu"]) == base
    (root / "paged_kv_chunk_gb300" / "csrc" / "k.cu").write_text("int f(int x) { return x + 2; }\n")
    assert bench.source_digest(["k.cu"]) != base


def test_profiled_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    root = _fake_tree(tmp_path, "int f(int x) { return x + 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    sha = bench.source_digest(["k.cu"])
    (root / "profiles" / "p.md").write_text(
        f"# p\n\nkernel_source_sha: {sha}\ndram_bytes_per_launch: 123456\n")
    assert bench.profiled_traffic("p", ["k.cu"]) == 123456.0
    (root / "paged_kv_chunk_gb300" / "csrc" / "k.cu").write_text("int f(int x) { return x - 1; }\n")
    assert bench.profiled_traffic("p", ["k.cu"]) is None
    assert bench.profiled_traffic("missing", ["k.cu"]) is None


def test_committed_profiles_name_their_source_and_traffic():
    """Every committed kernel summary that the benchmark reads carries both fields."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    for name in sorted(os.listdir(os.path.join(root, "profiles"))):
        if not name.startswith(("chunk_step_", "packed_varlen")):
            continue
        text = open(os.path.join(root, "profiles", name)).read()
        assert "kernel_source_sha:" in text and "dram_bytes_per_launch:" in text, name
        traffic = float(text.split("dram_bytes_per_launch:")[1].split()[0])
        assert np.isfinite(traffic) and traffic > 0, name


@pytest.mark.parametrize("config", ["tiny", "projection_small", "packed_varlen"])
def test_reference_arm_prints_one_contract_line(config):
    """`bench.py --impl reference` times the oracle and prints one JSON line with the
    contract's keys, for a streaming, a projection and a packed workload."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", config,
                          "--steps", "1", "--warmup", "0"], cwd=root, check=True,
                         capture_output=True, text=True, timeout=600).stdout
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["value"] > 0 and j["cpu_baseline"]["kind"] == "oracle"
