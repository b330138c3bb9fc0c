"""The multi-rank host path on CPU: two gloo ranks (spawned processes, rendezvous on
127.0.0.1) shard the work with the package's partitioning, each computes its share on the
CPU oracle, and the union must equal the single-process result exactly.  The same module
supplies the barrier and the max-over-ranks timing that the benchmark uses under torchrun.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from paged_kv_chunk_gb300 import dist as pdist
from paged_kv_chunk_gb300 import synthetic as syn

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD), LOCAL_RANK=str(rank))
    import oracle
    r, world, _ = pdist.setup("gloo")
    assert (r, world) == (rank, WORLD)
    result = {}
    # packed: length-balanced bins of the utterances
    cfg = syn.PackedConfig("mr", num_seqs=9, min_len=3, max_len=40, H=2, D=16, dtype="f32", seed=5)
    x = syn.packed_inputs(cfg)
    bins = pdist.balance_segments(x["lengths"], world)
    mine = pdist.pack_subset(x, bins[r])
    result["segs"] = bins[r]
    result["packed"] = oracle.packed_relattn(mine["q"], mine["k"], mine["v"], mine["cu_seqlens"],
                                             mine["pos_bias_u"], mine["pos_bias_v"], mine["rel"])
    # streaming: a contiguous shard of the cohort's streams
    scfg = syn.StreamingConfig("mrs", B=5, H=2, D=16, T=3, C=6, block_size=4, dtype="f32", seed=6)
    sx = syn.streaming_inputs(scfg)
    sh = pdist.stream_shard(scfg.B, world, r)
    result["streams"] = list(sh)
    result["stream_out"] = oracle.chunk_relattn(
        sx["q"][sh.start:sh.stop], sx["cache_k"][sh.start:sh.stop], sx["cache_v"][sh.start:sh.stop],
        sx["k_new"][sh.start:sh.stop], sx["v_new"][sh.start:sh.stop], sx["pos_bias_u"],
        sx["pos_bias_v"], sx["rel"])
    # timing helpers
    pdist.barrier()
    result["max"] = pdist.max_over_ranks(10.0 + 3.0 * r)
    np.save(os.path.join(out_dir, f"rank{r}.npy"), result, allow_pickle=True)
    torch.distributed.destroy_process_group()


@pytest.fixture(scope="module")
def rank_results(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("ranks"))
    mp.start_processes(_rank_main, args=(_free_port(), out), nprocs=WORLD, join=True,
                       start_method="spawn")
    return [np.load(os.path.join(out, f"rank{r}.npy"), allow_pickle=True).item() for r in range(WORLD)]


def test_packed_shards_cover_every_utterance_once_and_match(rank_results):
    import oracle
    cfg = syn.PackedConfig("mr", num_seqs=9, min_len=3, max_len=40, H=2, D=16, dtype="f32", seed=5)
    x = syn.packed_inputs(cfg)
    full = oracle.packed_relattn(x["q"], x["k"], x["v"], x["cu_seqlens"], x["pos_bias_u"],
                                 x["pos_bias_v"], x["rel"])
    segs = sorted(s for r in rank_results for s in r["segs"])
    assert segs == list(range(cfg.num_seqs))
    cu = x["cu_seqlens"]
    for r in rank_results:
        rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in r["segs"]])
        np.testing.assert_array_equal(r["packed"], full[rows])


def test_stream_shards_cover_the_cohort_and_match(rank_results):
    import oracle
    scfg = syn.StreamingConfig("mrs", B=5, H=2, D=16, T=3, C=6, block_size=4, dtype="f32", seed=6)
    sx = syn.streaming_inputs(scfg)
    full = oracle.chunk_relattn(sx["q"], sx["cache_k"], sx["cache_v"], sx["k_new"], sx["v_new"],
                                sx["pos_bias_u"], sx["pos_bias_v"], sx["rel"])
    assert sorted(b for r in rank_results for b in r["streams"]) == list(range(scfg.B))
    for r in rank_results:
        np.testing.assert_array_equal(r["stream_out"], full[r["streams"]])


def test_max_over_ranks_is_the_slowest_rank(rank_results):
    assert [r["max"] for r in rank_results] == [10.0 + 3.0 * (WORLD - 1)] * WORLD


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_balanced_bins_bound(world):
    rng = np.random.default_rng(world)
    lengths = rng.integers(50, 1501, size=256)
    bins = pdist.balance_segments(lengths, world)
    assert sorted(s for b in bins for s in b) == list(range(len(lengths)))
    cost = lengths.astype(np.int64) ** 2
    loads = [int(cost[b].sum()) for b in bins]
    assert max(loads) <= cost.sum() / world + cost.max()


@pytest.mark.parametrize("B,world", [(64, 1), (64, 3), (5, 8), (256, 8)])
def test_stream_shard_partitions(B, world):
    shards = [pdist.stream_shard(B, world, r) for r in range(world)]
    assert [b for s in shards for b in s] == list(range(B))
    sizes = [len(s) for s in shards]
    assert max(sizes) - min(sizes) <= 1
