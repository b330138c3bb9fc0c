"""Host-side checks of the benchmark's bookkeeping (no GPU): the algorithmic byte and flop
counts the roofline divides by, the visible-pair count of the chunked-limited window, the
rule that a recorded ncu capture's DRAM traffic is reported only for the kernel source it
was taken on, and the multi-rank plumbing (the relaunch under torch.distributed.run, the
process group, barrier and max over ranks) as two gloo ranks on the CPU."""
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
    import json
    root = _fake_tree(tmp_path, "int f(int x) { return x + 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    sha = bench.source_digest(["k.cu"])
    (root / "profiles" / "traffic.json").write_text(json.dumps(
        {"p": {"kernel_source_sha": sha, "dram_bytes_per_launch": 123456, "capture": "ncu ..."}}))
    traffic, src = bench.profiled_traffic("p", ["k.cu"])
    assert traffic == 123456.0 and sha in src
    (root / "paged_kv_chunk_gb300" / "csrc" / "k.cu").write_text("int f(int x) { return x - 1; }\n")
    assert bench.profiled_traffic("p", ["k.cu"])[0] is None
    assert bench.profiled_traffic("missing", ["k.cu"])[0] is None


def test_recorded_traffic_names_source_capture_and_bytes():
    """Every capture recorded for the benchmark carries its source digest, its command and a
    positive byte count, and each has its text summary beside it."""
    import json
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    recs = json.load(open(os.path.join(root, bench.TRAFFIC_FILE)))
    assert recs
    for name, rec in recs.items():
        assert len(rec["kernel_source_sha"]) == 16, name
        assert rec["capture"].startswith("ncu ") and "--clock-control none" in rec["capture"], name
        assert np.isfinite(rec["dram_bytes_per_launch"]) and rec["dram_bytes_per_launch"] > 0, name
        assert os.path.exists(os.path.join(root, "profiles", name + ".md")), name


def test_torchrun_relaunch_command():
    argv = bench.torchrun_argv(4, ["--gpus", "4", "--steps", "3"], 29511)
    assert argv[1:3] == ["-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in argv and "127.0.0.1" in argv and "29511" in argv
    assert argv[-4:] == ["--gpus", "4", "--steps", "3"] and argv[-5].endswith("bench.py")


def _rank_plumbing(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    r, w, local = bench.dist_setup()
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 * (r + 1), w)
    bench.barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    q.put((r, w, local, slowest))


def test_bench_rank_plumbing_two_gloo_ranks():
    """The benchmark's own setup, barrier and max over ranks, as two gloo ranks on the CPU:
    every rank sees the slowest rank's time."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = bench.free_port()
    procs = [ctx.Process(target=_rank_plumbing, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 0, 20.0), (1, 2, 1, 20.0)]


def test_gpus_flag_launches_that_many_ranks():
    """`bench.py --gpus 2` outside a launcher runs itself as two ranks; the reference arm's
    rank 0 prints the one line, rank 1 exits without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"], cwd=root, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["n_gpus"] == 2


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
