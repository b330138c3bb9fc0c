"""GPU parity: the CUDA path against the fp64 oracle, through the C ABI.

Every workload of the five configurations is checked: element by element where the
oracle finishes in seconds, else on sampled output rows the oracle computes one by
one.  Edge cases cover ragged pages and stages, every supported chunk-tile shape,
block sizes 8..256, empty caches, longer tables, invalid block ids and packed rows
with empty, single-frame and tile-straddling segments.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_chunk_gb300 import capi
from paged_kv_chunk_gb300 import synthetic as syn

from helpers import (check_close, dev, dev_pool, gpu_stream_inputs, host_pool, oracle_chunk,
                     sample_rows, stream_case, to_np, TOL_BF16_INTERNAL)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean_status():
    capi.oasr_device_status(clear=True)
    yield


def _run_step(cfg, x, fused):
    d = gpu_stream_inputs(x, cfg.dtype)
    if fused:
        out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], d["k_pool"], d["v_pool"],
                                         d["block_table"], d["cache_seqlens"], d["pos_bias_u"],
                                         d["pos_bias_v"], d["rel"])
    else:
        capi.oasr_paged_append(d["k_new"], d["v_new"], d["k_pool"], d["v_pool"], d["block_table"],
                               d["cache_seqlens"])
        out = capi.oasr_chunk_relattn_paged(d["q"], d["k_pool"], d["v_pool"], d["block_table"],
                                            d["cache_seqlens"], d["pos_bias_u"], d["pos_bias_v"],
                                            d["rel"])
    torch.cuda.synchronize()
    return out, d


FULL = [syn.TINY, syn.SMALL]
SAMPLED = [syn.LARGE] + list(syn.SWEEP)


# ------------------------------------------------------------------------- append


@pytest.mark.parametrize("cfg", [syn.TINY, syn.SMALL, syn.LARGE, syn.WINDOW_RING, syn.HETERO]
                         + list(syn.SWEEP), ids=lambda c: c.name)
def test_append_bit_exact(cfg):
    x = stream_case(cfg)
    d = gpu_stream_inputs(x, cfg.dtype)
    capi.oasr_paged_append(d["k_new"], d["v_new"], d["k_pool"], d["v_pool"], d["block_table"],
                           d["cache_seqlens"])
    kp, vp = x["k_pool"].copy(), x["v_pool"].copy()
    skipped = oracle.paged_append(syn.to_bits(x["k_new"], cfg.dtype),
                                  syn.to_bits(x["v_new"], cfg.dtype), kp, vp, x["block_table"],
                                  x["cache_seqlens"])
    assert skipped == 0
    np.testing.assert_array_equal(host_pool(d["k_pool"], cfg.dtype), kp)
    np.testing.assert_array_equal(host_pool(d["v_pool"], cfg.dtype), vp)
    assert capi.oasr_device_status() == 0


def test_append_skips_bad_blocks_and_flags():
    cfg = syn.StreamingConfig("bad", B=3, H=2, D=64, T=5, C=6, block_size=8, dtype="bf16", seed=7)
    x = stream_case(cfg)
    bt = x["block_table"].copy()
    bt[1, 1] = cfg.pool_blocks + 5          # stream 1's chunk page points outside the pool
    x["block_table"] = bt
    d = gpu_stream_inputs(x, cfg.dtype)
    capi.oasr_paged_append(d["k_new"], d["v_new"], d["k_pool"], d["v_pool"], d["block_table"],
                           d["cache_seqlens"])
    kp, vp = x["k_pool"].copy(), x["v_pool"].copy()
    skipped = oracle.paged_append(syn.to_bits(x["k_new"], "bf16"), syn.to_bits(x["v_new"], "bf16"),
                                  kp, vp, bt, x["cache_seqlens"])
    assert skipped > 0
    np.testing.assert_array_equal(host_pool(d["k_pool"], "bf16"), kp)
    assert capi.oasr_device_status() & capi.STATUS_BOUNDS_BIT


# ---------------------------------------------------------------- chunk attention


@pytest.mark.parametrize("cfg", FULL, ids=lambda c: c.name)
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_chunk_attention_full(cfg, fused):
    x = stream_case(cfg)
    out, _ = _run_step(cfg, x, fused)
    ref = oracle_chunk(x)
    check_close(to_np(out), ref, cfg.dtype, cfg.name)
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("cfg", SAMPLED, ids=lambda c: c.name)
def test_chunk_attention_sampled_full_size(cfg):
    """Full-size workload in the launch configuration the benchmark times (fused step);
    2048 sampled output rows compared with the oracle, plus the two-call path."""
    x = stream_case(cfg)
    out, _ = _run_step(cfg, x, fused=True)
    rng = np.random.default_rng(cfg.seed + 1)
    rows = sample_rows(rng, cfg.B, cfg.T, cfg.H, 2048)
    ref = oracle_chunk(x, rows=rows)
    got = to_np(out)
    b, i, h = rows[:, 0], rows[:, 1], rows[:, 2]
    check_close(got[b, i, h], ref[b, i, h], cfg.dtype, cfg.name)
    # append + attention as two calls: the same result up to summation order (the fused
    # step may read the chunk as a stage of its own)
    out2, _ = _run_step(cfg, x, fused=False)
    got2 = to_np(out2)
    check_close(got2[b, i, h], ref[b, i, h], cfg.dtype, cfg.name + " two calls")
    assert float(np.abs(got - got2).max()) <= TOL_BF16_INTERNAL, "fused step and append + attention differ"
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("cfg", [syn.SMALL, syn.LARGE, syn.HETERO] + list(syn.SWEEP),
                         ids=lambda c: c.name)
def test_fused_step_writes_the_same_pool(cfg):
    """The fused step's append (which may read the chunk into its own stage and write the
    pool from there) leaves the pools bit-identical to the stand-alone append, at every
    chunk size the dispatch routes to a different kernel form."""
    x = stream_case(cfg)
    _, d1 = _run_step(cfg, x, fused=True)
    _, d2 = _run_step(cfg, x, fused=False)
    assert torch.equal(d1["k_pool"].view(torch.int16), d2["k_pool"].view(torch.int16))
    assert torch.equal(d1["v_pool"].view(torch.int16), d2["v_pool"].view(torch.int16))


def test_paging_permutation_is_invisible():
    """Results are bit-identical whichever physical blocks the table names."""
    cfg = syn.SMALL
    x0 = stream_case(cfg)
    n_pages = cfg.mbps
    ident = np.arange(cfg.B * n_pages, dtype=np.int32).reshape(cfg.B, n_pages)
    x1 = stream_case(cfg, block_table=ident)
    rev = (cfg.pool_blocks - 1 - ident).astype(np.int32)
    x2 = stream_case(cfg, block_table=rev)
    outs = [_run_step(cfg, x, fused=True)[0] for x in (x0, x1, x2)]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


EDGE = [
    # (B, H, T, C, block_size, R extra, dtype)
    (2, 2, 1, 0, 16, 0, "bf16"),       # a single key
    (3, 2, 1, 7, 8, 0, "bf16"),        # T=1 decode-like step
    (2, 3, 4, 5, 8, 0, "bf16"),        # ragged page and stage
    (2, 2, 16, 0, 16, 0, "bf16"),      # no cache
    (2, 2, 16, 48, 16, 3, "bf16"),     # keys end exactly on a stage; longer table
    (3, 2, 16, 113, 32, 0, "bf16"),    # ragged 32-row page
    (2, 2, 13, 200, 64, 0, "bf16"),    # block = stage
    (2, 2, 16, 300, 128, 0, "bf16"),   # a stage inside a page
    (2, 2, 16, 270, 256, 5, "bf16"),   # largest block
    (2, 2, 17, 40, 16, 0, "bf16"),     # two m-tiles, ragged
    (2, 2, 32, 96, 16, 0, "bf16"),     # two m-tiles, full
    (2, 2, 33, 20, 16, 0, "bf16"),     # four m-tiles, ragged
    (2, 2, 64, 130, 16, 0, "bf16"),    # four m-tiles, full
    (3, 1, 16, 100, 16, 0, "bf16"),    # a single head
    (2, 6, 9, 70, 32, 0, "bf16"),      # six heads, T not a power of two
    (2, 4, 16, 530, 32, 0, "bf16"),    # past the largest position table, 32-row pages
    (2, 2, 16, 288, 8, 0, "bf16"),     # a whole-CTA position table from one batch of rel loads
    (2, 2, 16, 290, 8, 0, "bf16"),     # one page more: a second batch
    (2, 2, 16, 528, 8, 0, "bf16"),     # the largest table that fits (544 keys)
    (2, 2, 16, 530, 8, 0, "bf16"),     # one page past it: the per-stage band
    (2, 2, 11, 61, 16, 4, "bf16"),     # odd chunk start: unaligned table reads; longer table
    (80, 4, 5, 37, 8, 0, "bf16"),      # more than one wave of CTAs: the four-per-SM kernel
    (2, 2, 5, 77, 8, 2, "f32"),
    (2, 3, 40, 33, 16, 0, "f32"),
    (1, 1, 1, 0, 8, 0, "f32"),
    # chunks of 33-64 frames with an even head count: the tcgen05 kernel (a head pair per tile)
    (2, 2, 33, 0, 16, 0, "bf16"),      # the shortest such chunk, no history: one stage
    (3, 4, 40, 7, 8, 0, "bf16"),       # odd history, 8-row pages: five boxes per stage
    (2, 2, 64, 200, 64, 3, "bf16"),    # one page per stage; longer rel table
    (2, 2, 48, 200, 256, 0, "bf16"),   # pages of 256 rows: 64-row boxes inside a page
    (1, 2, 64, 1000, 128, 0, "bf16"),  # a long history in 128-row pages
    (2, 6, 50, 61, 32, 0, "bf16"),     # three head pairs, T not a power of two
    (3, 2, 63, 1, 16, 0, "bf16"),      # one cached frame: the last stage holds one key
    (2, 3, 48, 90, 16, 0, "bf16"),     # odd H: the mma.sync kernel for the same chunk
]


@pytest.mark.parametrize("B,H,T,C,bs,extra,dtype", EDGE)
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_chunk_attention_edge_cases(B, H, T, C, bs, extra, dtype, fused):
    cfg = syn.StreamingConfig("edge", B=B, H=H, D=64, T=T, C=C, block_size=bs, dtype=dtype,
                              seed=31 + T + C)
    x = stream_case(cfg, R=cfg.R + extra)
    out, _ = _run_step(cfg, x, fused)
    check_close(to_np(out), oracle_chunk(x), dtype, f"edge B{B} H{H} T{T} C{C} bs{bs}")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("T,scale", [(8, 0.9), (40, 0.9), (40, -0.3), (64, 0.0)], ids=str)
def test_chunk_scale_argument(T, scale):
    """The scale argument, including a negative one (its sign is folded into q+u and q+v on
    the tensor-core path) and zero (uniform weights)."""
    cfg = syn.StreamingConfig("scale", B=2, H=2, D=64, T=T, C=24, block_size=16, dtype="bf16",
                              seed=5)
    x = stream_case(cfg)
    d = gpu_stream_inputs(x, "bf16")
    capi.oasr_paged_append(d["k_new"], d["v_new"], d["k_pool"], d["v_pool"], d["block_table"],
                           d["cache_seqlens"])
    out = capi.oasr_chunk_relattn_paged(d["q"], d["k_pool"], d["v_pool"], d["block_table"],
                                        d["cache_seqlens"], d["pos_bias_u"], d["pos_bias_v"],
                                        d["rel"], scale=scale)
    check_close(to_np(out), oracle_chunk(x, scale=scale), "bf16", f"scale {scale}")


@pytest.mark.parametrize("T", [8, 48])
def test_invalid_block_id_is_flagged_and_contained(T):
    """A bad block id in one stream's table raises the bounds bit; the other streams'
    rows are still exact and nothing is read or written outside the pool (T = 48: the append
    and the tensor-core kernel)."""
    cfg = syn.StreamingConfig("badid", B=3, H=2, D=64, T=T, C=40, block_size=16, dtype="bf16",
                              seed=9)
    x = stream_case(cfg)
    bt = x["block_table"].copy()
    bt[1, 0] = -3
    bt[1, 1] = cfg.pool_blocks + 100
    d = gpu_stream_inputs(x, "bf16")
    d["block_table"] = torch.from_numpy(bt).cuda()
    out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], d["k_pool"], d["v_pool"],
                                     d["block_table"], d["cache_seqlens"], d["pos_bias_u"],
                                     d["pos_bias_v"], d["rel"])
    torch.cuda.synchronize()
    assert capi.oasr_device_status() & capi.STATUS_BOUNDS_BIT
    ref = oracle_chunk(x)
    got = to_np(out)
    for b in (0, 2):
        check_close(got[b], ref[b], "bf16", f"stream {b}")


@pytest.mark.parametrize("C,T,bad_page", [(40, 8, 2), (44, 8, 3), (44, 8, 2), (0, 16, 0),
                                         (40, 40, 3), (32, 48, 4), (0, 64, 1)],
                         ids=lambda v: str(v))
def test_fused_step_with_an_invalid_chunk_page(C, T, bad_page):
    """A chunk page that names no valid block: the fused step falls back to writing the
    chunk, fencing it and reading it from the pool; the rows of that page read as zeros
    (and are not written), everything else is exact."""
    cfg = syn.StreamingConfig("badchunk", B=3, H=2, D=64, T=T, C=C, block_size=16, dtype="bf16",
                              seed=12)
    x = stream_case(cfg)
    bt = x["block_table"].copy()
    bt[1, bad_page] = cfg.pool_blocks + 7
    d = gpu_stream_inputs(x, "bf16")
    d["block_table"] = torch.from_numpy(bt).cuda()
    out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], d["k_pool"], d["v_pool"],
                                     d["block_table"], d["cache_seqlens"], d["pos_bias_u"],
                                     d["pos_bias_v"], d["rel"])
    torch.cuda.synchronize()
    assert capi.oasr_device_status() & capi.STATUS_BOUNDS_BIT
    got = to_np(out)
    ref = oracle_chunk(x)
    for b in (0, 2):
        check_close(got[b], ref[b], "bf16", f"stream {b}")
    # stream 1: every key in the bad page (cached or chunk) is a zero key and value
    x1 = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in x.items()}
    for p in range(C + T):
        if p // cfg.block_size == bad_page:
            if p < C:
                x1["cache_k"][1, p] = 0
                x1["cache_v"][1, p] = 0
            else:
                x1["k_new"][1, p - C] = 0
                x1["v_new"][1, p - C] = 0
    check_close(got[1], oracle_chunk(x1)[1], "bf16", "stream 1 (bad chunk page)")


# ----------------------------------------------------------------------- packed


def _packed_case(lengths, dtype="bf16", seed=3, H=2, R_extra=0):
    cfg = syn.PackedConfig("p", num_seqs=len(lengths), min_len=1, max_len=max(max(lengths), 1),
                           H=H, D=64, dtype=dtype, seed=seed)
    x = syn.packed_inputs(cfg, lengths=lengths)
    if R_extra:
        rng = np.random.default_rng(seed + 99)
        x["rel"] = syn.normal(rng, (x["rel"].shape[0] + R_extra, H, 64), dtype)
    return cfg, x


def _run_packed(x, dtype):
    d = {k: dev(x[k], dtype) for k in ("q", "k", "v", "pos_bias_u", "pos_bias_v", "rel")}
    cu = torch.from_numpy(x["cu_seqlens"]).cuda()
    out = capi.oasr_packed_relattn_varlen(d["q"], d["k"], d["v"], cu, max(x["max_seqlen"], 1),
                                          d["pos_bias_u"], d["pos_bias_v"], d["rel"])
    torch.cuda.synchronize()
    return out


def _oracle_packed(x, rows=None):
    return oracle.packed_relattn(x["q"], x["k"], x["v"], x["cu_seqlens"], x["pos_bias_u"],
                                 x["pos_bias_v"], x["rel"], rows=rows)


@pytest.mark.parametrize("lengths", [
    [1], [64], [65], [7, 0, 130, 1, 64, 200, 3], [300, 299, 1, 0, 0, 150],
    [128], [129], [256, 255, 257, 127],
    [16, 17, 31, 33, 112, 113, 144, 145],   # the last stage's P.V stops at its 16-key step
], ids=str)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_packed_full(lengths, dtype):
    _, x = _packed_case(lengths, dtype=dtype)
    out = _run_packed(x, dtype)
    check_close(to_np(out), _oracle_packed(x), dtype, f"packed {lengths}")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("scale", [0.3, -0.2, 0.0], ids=str)
def test_packed_scale_argument(scale):
    """Any scale, including a negative one (folded into the sign of q+u and q+v) and zero."""
    _, x = _packed_case([200, 1, 77], seed=14)
    d = {k: dev(x[k], "bf16") for k in ("q", "k", "v", "pos_bias_u", "pos_bias_v", "rel")}
    cu = torch.from_numpy(x["cu_seqlens"]).cuda()
    out = capi.oasr_packed_relattn_varlen(d["q"], d["k"], d["v"], cu, x["max_seqlen"], d["pos_bias_u"],
                                          d["pos_bias_v"], d["rel"], scale=scale)
    torch.cuda.synchronize()
    ref = oracle.packed_relattn(x["q"], x["k"], x["v"], x["cu_seqlens"], x["pos_bias_u"],
                                x["pos_bias_v"], x["rel"], scale=scale)
    check_close(to_np(out), ref, "bf16", f"packed scale {scale}")


def test_packed_longer_table():
    _, x = _packed_case([90, 33], R_extra=10)
    out = _run_packed(x, "bf16")
    check_close(to_np(out), _oracle_packed(x), "bf16", "longer table")


def test_packed_full_size_sampled():
    """The 256-utterance packed row: 4096 sampled (token, head) rows plus every row of
    the shortest and the longest segment."""
    cfg = syn.PACKED
    x = syn.packed_inputs(cfg)
    out = _run_packed(x, cfg.dtype)
    rng = np.random.default_rng(77)
    total = int(x["cu_seqlens"][-1])
    t = rng.choice(total, size=4096, replace=False)
    h = rng.integers(0, cfg.H, size=4096)
    rows = [np.stack([t, h], 1)]
    for s in (int(np.argmin(x["lengths"])), int(np.argmax(x["lengths"]))):
        a, e = x["cu_seqlens"][s], x["cu_seqlens"][s + 1]
        tt = np.repeat(np.arange(a, e), cfg.H)
        hh = np.tile(np.arange(cfg.H), e - a)
        rows.append(np.stack([tt, hh], 1))
    rows = np.concatenate(rows).astype(np.int32)
    ref = _oracle_packed(x, rows=rows)
    got = to_np(out)
    check_close(got[rows[:, 0], rows[:, 1]], ref[rows[:, 0], rows[:, 1]], cfg.dtype, "packed full")
    assert capi.oasr_device_status() == 0


def test_packed_segment_order_and_concatenation():
    lengths = [70, 5, 129]
    _, x = _packed_case(lengths, seed=11)
    full = _run_packed(x, "bf16")
    cu = x["cu_seqlens"]
    for s in range(len(lengths)):
        a, e = cu[s], cu[s + 1]
        alone = dict(x, q=x["q"][a:e], k=x["k"][a:e], v=x["v"][a:e],
                     cu_seqlens=np.array([0, e - a], np.int32), max_seqlen=int(e - a))
        assert torch.equal(_run_packed(alone, "bf16"), full[a:e])


def test_streaming_rows_equal_packed_rows_gpu():
    """Chunk attention at cache C equals rows C..C+T-1 of the packed attention over one
    segment of C+T frames (same keys; same rel rows), on the GPU."""
    B, H, T, C = 1, 2, 16, 80
    cfg = syn.StreamingConfig("sp", B=B, H=H, D=64, T=T, C=C, block_size=16, dtype="bf16",
                              seed=21)
    L = C + T
    rng = np.random.default_rng(5)
    relp = syn.normal(rng, (2 * L - 1, H, 64), "bf16")
    x = stream_case(cfg)
    x["rel"] = relp[: cfg.R]
    out_s, _ = _run_step(cfg, x, fused=True)
    qq = np.concatenate([syn.normal(rng, (C, H, 64), "bf16"), x["q"][0]])
    px = dict(q=qq, k=np.concatenate([x["cache_k"][0], x["k_new"][0]]),
              v=np.concatenate([x["cache_v"][0], x["v_new"][0]]),
              cu_seqlens=np.array([0, L], np.int32), pos_bias_u=x["pos_bias_u"],
              pos_bias_v=x["pos_bias_v"], rel=relp, max_seqlen=L)
    out_p = _run_packed(px, "bf16")
    check_close(to_np(out_s[0]), to_np(out_p[C:]), "bf16", "streaming vs packed")


# ------------------------------------------- heterogeneous offsets, padding lane


def _hetero_inputs(Cs, T, H, bs, seed, R):
    """Streams with different cache lengths sharing one rel table of R rows."""
    rng = np.random.default_rng(seed)
    B = len(Cs)
    cmax = max(Cs)
    pages = -(-(cmax + T) // bs)
    nb = 2 * B * pages
    x = {
        "q": syn.normal(rng, (B, T, H, 64), "bf16"),
        "k_new": syn.normal(rng, (B, T, H, 64), "bf16"),
        "v_new": syn.normal(rng, (B, T, H, 64), "bf16"),
        "pos_bias_u": syn.normal(rng, (H, 64), "bf16"),
        "pos_bias_v": syn.normal(rng, (H, 64), "bf16"),
        "rel": syn.normal(rng, (R, H, 64), "bf16"),
        "block_table": syn.block_table(rng, B, pages, nb),
        "cache_seqlens": np.array(Cs, np.int32),
        "caches": [(syn.normal(rng, (1, c, H, 64), "bf16"), syn.normal(rng, (1, c, H, 64), "bf16"))
                   for c in Cs],
    }
    kp = syn.canary_pool(nb, bs, H, 64, "bf16")
    vp = syn.canary_pool(nb, bs, H, 64, "bf16")
    for b, (ck, cv) in enumerate(x["caches"]):
        if Cs[b]:
            oracle.paged_append(syn.to_bits(ck, "bf16"), syn.to_bits(cv, "bf16"), kp, vp,
                                x["block_table"][b:b + 1], np.zeros(1, np.int32))
    x["k_pool"], x["v_pool"] = kp, vp
    return x


@pytest.mark.parametrize("Cs,T", [([0, 17, 64, 130, 255, 3], 16), ([0, 300, 527, 130, 511, 45], 16),
                                  ([0, 17, 64, 130, 255, 3], 48), ([0, 300, 527, 130, 511, 45], 64)],
                         ids=["short", "long", "short_T48", "long_T64"])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_heterogeneous_cache_lengths_one_launch(fused, Cs, T):
    """Streams at different offsets in one launch (Scheduler page, section 4.3): each reads
    its own cache_seqlens and indexes the shared table at distance C_b + i - j (the long
    cohort's position tables take two batches of rel loads; T = 48 and 64 run on the
    tensor-core kernel, whose work items then have different stage counts)."""
    H, bs = 4, 16
    R = max(Cs) + 2 * T - 1 + 4
    x = _hetero_inputs(Cs, T, H, bs, seed=123, R=R)
    cfg = syn.StreamingConfig("het", B=len(Cs), H=H, D=64, T=T, C=max(Cs), block_size=bs,
                              dtype="bf16", seed=0)
    out, _ = _run_step(cfg, x, fused)
    got = to_np(out)
    for b, C in enumerate(Cs):
        ck, cv = x["caches"][b]
        ref = oracle.chunk_relattn(x["q"][b:b + 1], ck, cv, x["k_new"][b:b + 1],
                                   x["v_new"][b:b + 1], x["pos_bias_u"], x["pos_bias_v"], x["rel"])
        check_close(got[b:b + 1], ref, "bf16", f"stream {b} (C={C})")
    assert capi.oasr_device_status() == 0


def test_padding_lanes_share_a_scratch_block():
    """Padding rows whose block tables point only at one scratch block outside the
    streams' pages (ASR Engine page, section 9, padding lane) compute garbage only for
    themselves: the real streams' rows and pages are exact."""
    cfg = syn.StreamingConfig("pad", B=3, H=4, D=64, T=16, C=80, block_size=16, dtype="bf16",
                              seed=77)
    x = stream_case(cfg)
    n_pad = 2
    scratch = cfg.pool_blocks - 1
    assert scratch not in x["block_table"]
    bt = np.concatenate([x["block_table"], np.full((n_pad, cfg.mbps), scratch, np.int32)])
    xp = dict(x)
    for k in ("q", "k_new", "v_new"):
        xp[k] = np.concatenate([x[k], np.zeros((n_pad,) + x[k].shape[1:], np.float32)])
    xp["block_table"] = bt
    xp["cache_seqlens"] = np.concatenate([x["cache_seqlens"], np.zeros(n_pad, np.int32)])
    cfgp = syn.StreamingConfig("pad", B=cfg.B + n_pad, H=4, D=64, T=16, C=80, block_size=16,
                               dtype="bf16", seed=77, num_blocks=cfg.pool_blocks,
                               max_blocks_per_seq=cfg.mbps)
    out, d = _run_step(cfgp, xp, fused=True)
    check_close(to_np(out[: cfg.B]), oracle_chunk(x), "bf16", "real streams")
    kp = host_pool(d["k_pool"], "bf16")
    expect = x["k_pool"].copy()
    oracle.paged_append(syn.to_bits(x["k_new"], "bf16"), syn.to_bits(x["v_new"], "bf16"), expect,
                        x["v_pool"].copy(), x["block_table"], x["cache_seqlens"])
    used = np.zeros(cfg.pool_blocks, bool)
    used[x["block_table"].ravel()] = True
    np.testing.assert_array_equal(kp[used], expect[used])
    assert capi.oasr_device_status() == 0


# ------------------------------------------------- chunked-limited packed (Nemotron offline)

NEMOTRON_CHUNK, NEMOTRON_LEFT = 8, 7   # 64-frame query blocks see 64 + 7 * 8 = 120 keys


def _run_chunked(x, dtype, cs, left):
    d = {k: dev(x[k], dtype) for k in ("q", "k", "v", "pos_bias_u", "pos_bias_v", "rel")}
    cu = torch.from_numpy(x["cu_seqlens"]).cuda()
    out = capi.oasr_packed_relattn_chunked(d["q"], d["k"], d["v"], cu, max(x["max_seqlen"], 1),
                                           d["pos_bias_u"], d["pos_bias_v"], d["rel"], cs, left)
    torch.cuda.synchronize()
    return out


def _oracle_chunked(x, cs, left, rows=None):
    return oracle.packed_relattn_chunked(x["q"], x["k"], x["v"], x["cu_seqlens"], x["pos_bias_u"],
                                         x["pos_bias_v"], x["rel"], cs, left, rows=rows)


@pytest.mark.parametrize("cs,left", [(8, 7), (1, 0), (4, 2), (16, 1), (3, 50), (128, 0), (5, 30)],
                         ids=lambda v: str(v))
@pytest.mark.parametrize("lengths", [
    [1], [64], [129], [7, 0, 130, 1, 64, 200, 3], [300, 257, 1, 150],
], ids=str)
def test_chunked_full(lengths, cs, left):
    _, x = _packed_case(lengths, seed=5)
    out = _run_chunked(x, "bf16", cs, left)
    check_close(to_np(out), _oracle_chunked(x, cs, left), "bf16", f"chunked {lengths} {cs},{left}")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("cs,left", [(8, 7), (1, 0), (3, 4)], ids=lambda v: str(v))
def test_chunked_full_f32(cs, left):
    _, x = _packed_case([70, 1, 33, 140], dtype="f32", seed=6)
    out = _run_chunked(x, "f32", cs, left)
    check_close(to_np(out), _oracle_chunked(x, cs, left), "f32", f"chunked f32 {cs},{left}")
    assert capi.oasr_device_status() == 0


def test_chunked_one_chunk_is_the_bidirectional_call():
    """A chunk as long as every segment is the plain packed attention: the same window for any
    chunk at least that long (bit for bit), and the bidirectional result of the oracle."""
    lengths = [300, 1, 129, 64]
    _, x = _packed_case(lengths, seed=8)
    a = _run_chunked(x, "bf16", max(lengths), 0)
    assert torch.equal(a, _run_chunked(x, "bf16", 7 * max(lengths), 3))
    ref = _oracle_packed(x)
    check_close(to_np(a), ref, "bf16", "one chunk")
    check_close(to_np(_run_packed(x, "bf16")), ref, "bf16", "bidirectional")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("H,scale", [(2, -0.3), (4, 0.0), (6, 0.2), (16, None), (3, None), (1, -0.5)],
                         ids=str)
def test_chunked_heads_and_scale(H, scale):
    """Head counts and scales of the chunked call: even counts run two heads per tensor-core
    tile (a negative scale's sign folded into q+u and q+v), odd ones the one-head kernel."""
    _, x = _packed_case([150, 1, 64, 97, 0, 230], seed=31, H=H)
    d = {k: dev(x[k], "bf16") for k in ("q", "k", "v", "pos_bias_u", "pos_bias_v", "rel")}
    cu = torch.from_numpy(x["cu_seqlens"]).cuda()
    out = capi.oasr_packed_relattn_chunked(d["q"], d["k"], d["v"], cu, x["max_seqlen"],
                                           d["pos_bias_u"], d["pos_bias_v"], d["rel"], 8, 7,
                                           scale=scale)
    torch.cuda.synchronize()
    ref = oracle.packed_relattn_chunked(x["q"], x["k"], x["v"], x["cu_seqlens"], x["pos_bias_u"],
                                        x["pos_bias_v"], x["rel"], 8, 7, scale=scale)
    check_close(to_np(out), ref, "bf16", f"chunked H {H} scale {scale}")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("n", [511, 512], ids=str)
def test_chunked_segment_limit(n):
    """The most segments the chunked call's head-pair mode takes (511) and one more (the
    one-head kernel then takes the call), lengths 0..90."""
    rng = np.random.default_rng(93 + n)
    lengths = [int(v) for v in rng.integers(0, 91, size=n)]
    _, x = _packed_case(lengths, seed=94, H=4)
    out = _run_chunked(x, "bf16", 8, 7)
    check_close(to_np(out), _oracle_chunked(x, 8, 7), "bf16", f"{n} segments")
    assert capi.oasr_device_status() == 0


def test_chunked_full_size_sampled():
    """The 256-utterance packed row under the Nemotron window: 4096 sampled rows plus
    every row of the shortest and the longest segment."""
    cfg = syn.PACKED
    x = syn.packed_inputs(cfg)
    out = _run_chunked(x, cfg.dtype, NEMOTRON_CHUNK, NEMOTRON_LEFT)
    rng = np.random.default_rng(78)
    total = int(x["cu_seqlens"][-1])
    t = rng.choice(total, size=4096, replace=False)
    h = rng.integers(0, cfg.H, size=4096)
    rows = [np.stack([t, h], 1)]
    for s in (int(np.argmin(x["lengths"])), int(np.argmax(x["lengths"]))):
        a, e = x["cu_seqlens"][s], x["cu_seqlens"][s + 1]
        rows.append(np.stack([np.repeat(np.arange(a, e), cfg.H), np.tile(np.arange(cfg.H), e - a)], 1))
    rows = np.concatenate(rows).astype(np.int32)
    ref = _oracle_chunked(x, NEMOTRON_CHUNK, NEMOTRON_LEFT, rows=rows)
    got = to_np(out)
    check_close(got[rows[:, 0], rows[:, 1]], ref[rows[:, 0], rows[:, 1]], cfg.dtype, "chunked full")
    assert capi.oasr_device_status() == 0


# --------------------------------------------------------- fixed-window ring (eviction)


@pytest.mark.parametrize("bs,T,window,mbps", [(16, 16, 64, 12), (8, 16, 40, 20), (4, 12, 20, 40),
                                              (4, 6, 1, 40), (16, 12, 3, 12), (8, 5, 0, 20)],
                         ids=str)
def test_window_commit_matches_oracle(bs, T, window, mbps):
    """Bit-exact against the oracle's bookkeeping on random states, including windows shorter
    than a page (where only full pages may go and no cached length is negative)."""
    rng = np.random.default_rng(bs * 100 + T + 7 * window)
    B = 37
    bt = np.stack([rng.permutation(1000)[:mbps] for _ in range(B)]).astype(np.int32)
    cs = rng.integers(0, mbps * bs - T + 1, size=B).astype(np.int32)
    cs[:3] = [0, window, max(window - T, 0)]
    d_bt = torch.from_numpy(bt).cuda()
    d_cs = torch.from_numpy(cs).cuda()
    capi.oasr_window_commit(d_bt, d_cs, T, bs, window)
    torch.cuda.synchronize()
    ref_bt, ref_cs = oracle.window_commit(bt, cs, T, bs, window)
    np.testing.assert_array_equal(d_bt.cpu().numpy(), ref_bt)
    np.testing.assert_array_equal(d_cs.cpu().numpy(), ref_cs)
    assert (ref_cs >= 0).all()
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("bs,T,window", [(16, 16, 48), (8, 16, 40), (16, 8, 40), (16, 12, 3),
                                         (8, 5, 1)], ids=str)
def test_window_session_matches_the_sliding_history(bs, T, window):
    """A stream session under a trained window: every step is one fused append + attention
    launch followed by the commit with eviction; each step's output equals the oracle over
    the last cache_seqlens frames of the stream's own history, and the tables follow the
    oracle's bookkeeping exactly."""
    B, H, steps = 4, 2, 9
    rng = np.random.default_rng(bs + T + window)
    mbps = -(-(max(window, bs) + T) // bs) + 1
    nblk = B * mbps + 5
    bt = rng.permutation(nblk)[: B * mbps].reshape(B, mbps).astype(np.int32)
    cs = np.zeros(B, np.int32)
    R = max(window, bs) + 2 * T - 1
    u, vb, rel = (syn.normal(rng, shp, "bf16") for shp in ((H, 64), (H, 64), (R, H, 64)))
    d = {"u": dev(u, "bf16"), "vb": dev(vb, "bf16"), "rel": dev(rel, "bf16")}
    kp = dev_pool(syn.canary_pool(nblk, bs, H, 64, "bf16"), "bf16")
    vp = dev_pool(syn.canary_pool(nblk, bs, H, 64, "bf16"), "bf16")
    d_bt, d_cs = torch.from_numpy(bt).cuda(), torch.from_numpy(cs).cuda()
    hk = np.zeros((B, 0, H, 64), np.float32)
    hv = np.zeros((B, 0, H, 64), np.float32)
    for _ in range(steps):
        q, kn, vn = (syn.normal(rng, (B, T, H, 64), "bf16") for _ in range(3))
        out = capi.oasr_chunk_step_paged(dev(q, "bf16"), dev(kn, "bf16"), dev(vn, "bf16"), kp, vp,
                                         d_bt, d_cs, d["u"], d["vb"], d["rel"])
        C = int(cs[0])
        ref = oracle.chunk_relattn(q, hk[:, hk.shape[1] - C:], hv[:, hv.shape[1] - C:], kn, vn, u, vb, rel)
        check_close(to_np(out), ref, "bf16", f"window step C={C}")
        capi.oasr_window_commit(d_bt, d_cs, T, bs, window)
        bt, cs = oracle.window_commit(bt, cs, T, bs, window)
        np.testing.assert_array_equal(d_bt.cpu().numpy(), bt)
        np.testing.assert_array_equal(d_cs.cpu().numpy(), cs)
        hk = np.concatenate([hk, kn], 1)
        hv = np.concatenate([hv, vn], 1)
    assert 0 <= int(cs[0]) <= max(window, bs - 1)
    assert capi.oasr_device_status() == 0


# ------------------------------------------------ projections feeding the path


@pytest.mark.parametrize("M,R,H", [(1024, 287, 4), (4096, 543, 8), (77, 5, 2), (130, 300, 4)],
                         ids=str)
def test_projection_matches_oracle(M, R, H):
    """q/k/v with bias and the positional projection, one launch, against fp64 products of
    the same bf16 inputs (tiles straddled by M and R included)."""
    rng = np.random.default_rng(M + R)
    d = 64 * H
    x, pos = syn.normal(rng, (M, d), "bf16"), syn.normal(rng, (R, d), "bf16")
    w_qkv = syn.normal(rng, (3 * d, d), "bf16", sigma=1.0 / np.sqrt(d))
    w_pos = syn.normal(rng, (d, d), "bf16", sigma=1.0 / np.sqrt(d))
    b = syn.normal(rng, (3 * d,), "bf16")
    got = capi.oasr_project_qkv_pos(dev(x, "bf16"), dev(w_qkv, "bf16"), dev(b, "bf16"),
                                    dev(pos, "bf16"), dev(w_pos, "bf16"), H)
    torch.cuda.synchronize()
    ref = oracle.project_qkv_pos(x, w_qkv, b, pos, w_pos, H)
    for name, g, r in zip(("q", "k", "v", "rel"), got, ref):
        check_close(to_np(g), r, "bf16", name)
    assert capi.oasr_device_status() == 0


def test_projection_feeds_the_step():
    """The projected q, k_new, v_new and rel go straight into the fused step: the result
    equals the attention oracle on the oracle's own projections of the same inputs."""
    cfg = syn.StreamingConfig("proj", B=4, H=4, D=64, T=16, C=48, block_size=16, dtype="bf16", seed=21)
    x = stream_case(cfg)
    rng = np.random.default_rng(22)
    d = 64 * cfg.H
    xs = syn.normal(rng, (cfg.B * cfg.T, d), "bf16")
    pos = syn.normal(rng, (cfg.R, d), "bf16")
    w_qkv = syn.normal(rng, (3 * d, d), "bf16", sigma=1.0 / np.sqrt(d))
    w_pos = syn.normal(rng, (d, d), "bf16", sigma=1.0 / np.sqrt(d))
    b = syn.normal(rng, (3 * d,), "bf16")
    q, kn, vn, rel = capi.oasr_project_qkv_pos(dev(xs, "bf16"), dev(w_qkv, "bf16"), dev(b, "bf16"),
                                               dev(pos, "bf16"), dev(w_pos, "bf16"), cfg.H)
    shp = (cfg.B, cfg.T, cfg.H, 64)
    d_in = gpu_stream_inputs(x, "bf16")
    out = capi.oasr_chunk_step_paged(q.view(shp), kn.view(shp), vn.view(shp), d_in["k_pool"],
                                     d_in["v_pool"], d_in["block_table"], d_in["cache_seqlens"],
                                     d_in["pos_bias_u"], d_in["pos_bias_v"], rel)
    torch.cuda.synchronize()
    # the oracle sees the kernel's bf16 projections (their rounding is the projection's own
    # error, tested above), so this checks the hand-off of layouts between the two launches
    ref = oracle.chunk_relattn(to_np(q).reshape(shp), x["cache_k"], x["cache_v"], to_np(kn).reshape(shp),
                               to_np(vn).reshape(shp), x["pos_bias_u"], x["pos_bias_v"], to_np(rel))
    check_close(to_np(out), ref, "bf16", "projection -> step")


# ------------------------------------------------------------------------- maximum sizes


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
@pytest.mark.parametrize("T", [16, 64])
def test_widest_block_table(fused, T):
    """The widest block table the bf16 path takes (512 pages), filled to its last key: the
    chunk's last row lands in the table's last slot (T = 64: the tensor-core kernel)."""
    bs, mbps = 8, 512
    cfg = syn.StreamingConfig("widest", B=2, H=2, D=64, T=T, C=mbps * bs - T, block_size=bs,
                              dtype="bf16", seed=71, max_blocks_per_seq=mbps)
    assert cfg.mbps == mbps
    x = stream_case(cfg)
    out, d = _run_step(cfg, x, fused)
    check_close(to_np(out), oracle_chunk(x), "bf16", f"widest table, fused={fused}")
    kp = x["k_pool"].copy()
    vp = x["v_pool"].copy()
    oracle.paged_append(syn.to_bits(x["k_new"], "bf16"), syn.to_bits(x["v_new"], "bf16"), kp, vp,
                        x["block_table"], x["cache_seqlens"])
    assert np.array_equal(host_pool(d["k_pool"], "bf16"), kp)
    assert np.array_equal(host_pool(d["v_pool"], "bf16"), vp)
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("cfg", [syn.SMALL, syn.LARGE], ids=lambda c: c.name)
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_engine_sized_block_table(cfg, fused):
    """The engine's table geometry (ASR Engine page, section 6: max_blocks_per_seq sized for
    unlimited history, 512 pages): the cohort's pages first and every later entry -1.  The
    kernel sizes its work from the keys it can bound (the rel table's R - T + 1), so the result
    and the pools are bit-identical to the exact-size table's, and no entry past the pages is
    read (the status word stays clear)."""
    x = stream_case(cfg)
    out_exact, d_exact = _run_step(cfg, x, fused)
    wide = np.full((cfg.B, 512), -1, np.int32)
    wide[:, :cfg.mbps] = x["block_table"]
    xw = dict(x)
    xw["block_table"] = wide
    out_wide, d_wide = _run_step(cfg, xw, fused)
    assert torch.equal(out_exact.view(torch.int16), out_wide.view(torch.int16))
    assert torch.equal(d_exact["k_pool"].view(torch.int16), d_wide["k_pool"].view(torch.int16))
    assert torch.equal(d_exact["v_pool"].view(torch.int16), d_wide["v_pool"].view(torch.int16))
    rng = np.random.default_rng(cfg.seed + 5)
    rows = sample_rows(rng, cfg.B, cfg.T, cfg.H, 512)
    ref = oracle_chunk(x, rows=rows)
    b, i, h = rows[:, 0], rows[:, 1], rows[:, 2]
    check_close(to_np(out_wide)[b, i, h], ref[b, i, h], "bf16", "engine-sized table")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [4, 16, 40])
def test_short_rel_table_is_flagged(dtype, T):
    """A rel table shorter than C + 2T - 1 rows breaks the call's precondition: the call stays
    in bounds and raises the bounds bit of the status word."""
    cfg = syn.StreamingConfig("short_rel", B=2, H=2, D=64, T=T, C=100, block_size=16, dtype=dtype,
                              seed=55)
    x = stream_case(cfg, R=cfg.R - 5)
    _run_step(cfg, x, fused=True)
    assert capi.oasr_device_status() & capi.STATUS_BOUNDS_BIT
    _run_step(cfg, stream_case(cfg), fused=True)
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("window", [None, (8, 7)], ids=["bidirectional", "chunked"])
def test_packed_most_segments(window):
    """The largest segment count the packed calls take (1024), lengths 0..40."""
    rng = np.random.default_rng(91)
    lengths = [int(v) for v in rng.integers(0, 41, size=1024)]
    _, x = _packed_case(lengths, seed=92)
    if window is None:
        out = _run_packed(x, "bf16")
        ref = _oracle_packed(x)
    else:
        out = _run_chunked(x, "bf16", *window)
        ref = _oracle_chunked(x, *window)
    check_close(to_np(out), ref, "bf16", f"1024 segments, window {window}")
    assert capi.oasr_device_status() == 0
