"""Seeded random sweep of the streaming and packed entry points against the oracle.

The hand-picked cases in test_gpu_parity.py sit on the boundaries the kernels dispatch on;
this sweep draws shapes between and across them: chunk lengths 1..64, block sizes 8..256,
per-stream cache lengths (a heterogeneous cohort in every case), block tables with spare
entries, rel tables longer than needed, fused and two-call steps, bf16 and fp32; packed rows
with empty, single-frame and long segments, bidirectional and chunked-limited.  Every case
is compared element by element with the oracle, the pools the step leaves are compared bit
for bit with the oracle's append, and the device status word must stay clean.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_chunk_gb300 import capi
from paged_kv_chunk_gb300 import synthetic as syn

from helpers import check_close, dev, dev_pool, host_pool, to_np

pytestmark = pytest.mark.gpu

T_CHOICES = [1, 2, 3, 5, 8, 11, 16, 17, 24, 31, 32, 33, 48, 63, 64]
BS_CHOICES = [8, 16, 32, 64, 128, 256]
H_CHOICES = [1, 2, 3, 4, 8]
CMAX_CHOICES = [0, 40, 200, 560, 1100]


def _stream_params(seed):
    rng = np.random.default_rng(20_000 + seed)
    T = int(rng.choice(T_CHOICES))
    bs = int(rng.choice(BS_CHOICES))
    H = int(rng.choice(H_CHOICES))
    B = int(rng.integers(1, 6))
    cmax = int(rng.choice(CMAX_CHOICES))
    Cs = [int(c) for c in rng.integers(0, cmax + 1, size=B)]
    dtype = "f32" if rng.random() < 0.2 else "bf16"
    fused = bool(rng.random() < 0.5)
    spare_pages = int(rng.integers(0, 4))
    r_extra = int(rng.integers(0, 6))
    return rng, dict(T=T, bs=bs, H=H, B=B, Cs=Cs, dtype=dtype, fused=fused,
                     spare_pages=spare_pages, r_extra=r_extra)


def _stream_inputs(rng, T, bs, H, B, Cs, dtype, spare_pages, r_extra):
    mbps = -(-(max(Cs) + T) // bs) + spare_pages
    nb = 2 * B * mbps
    R = max(Cs) + 2 * T - 1 + r_extra
    x = {
        "q": syn.normal(rng, (B, T, H, 64), dtype),
        "k_new": syn.normal(rng, (B, T, H, 64), dtype),
        "v_new": syn.normal(rng, (B, T, H, 64), dtype),
        "pos_bias_u": syn.normal(rng, (H, 64), dtype),
        "pos_bias_v": syn.normal(rng, (H, 64), dtype),
        "rel": syn.normal(rng, (R, H, 64), dtype),
        "block_table": syn.block_table(rng, B, mbps, nb),
        "cache_seqlens": np.array(Cs, np.int32),
        "caches": [(syn.normal(rng, (1, c, H, 64), dtype), syn.normal(rng, (1, c, H, 64), dtype))
                   for c in Cs],
    }
    kp = syn.canary_pool(nb, bs, H, 64, dtype)
    vp = syn.canary_pool(nb, bs, H, 64, dtype)
    for b, (ck, cv) in enumerate(x["caches"]):
        if Cs[b]:
            assert oracle.paged_append(syn.to_bits(ck, dtype), syn.to_bits(cv, dtype), kp, vp,
                                       x["block_table"][b:b + 1], np.zeros(1, np.int32)) == 0
    x["k_pool"], x["v_pool"] = kp, vp
    return x


def _bits(pool):
    """Raw bits of a pool (the NaN canaries compare equal only as bits)."""
    return pool.view(np.uint32) if pool.dtype == np.float32 else pool


@pytest.fixture(autouse=True)
def _clean_status():
    capi.oasr_device_status(clear=True)
    yield


@pytest.mark.parametrize("seed", range(36))
def test_random_streaming_step(seed):
    rng, p = _stream_params(seed)
    x = _stream_inputs(rng, p["T"], p["bs"], p["H"], p["B"], p["Cs"], p["dtype"],
                       p["spare_pages"], p["r_extra"])
    dtype = p["dtype"]
    d = {k: dev(x[k], dtype) for k in ("q", "k_new", "v_new", "pos_bias_u", "pos_bias_v", "rel")}
    kp, vp = dev_pool(x["k_pool"], dtype), dev_pool(x["v_pool"], dtype)
    bt = torch.from_numpy(x["block_table"]).cuda()
    cs = torch.from_numpy(x["cache_seqlens"]).cuda()
    if p["fused"]:
        out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], kp, vp, bt, cs,
                                         d["pos_bias_u"], d["pos_bias_v"], d["rel"])
    else:
        capi.oasr_paged_append(d["k_new"], d["v_new"], kp, vp, bt, cs)
        out = capi.oasr_chunk_relattn_paged(d["q"], kp, vp, bt, cs, d["pos_bias_u"],
                                            d["pos_bias_v"], d["rel"])
    torch.cuda.synchronize()
    got = to_np(out)
    what = f"seed {seed} {p}"
    for b, (ck, cv) in enumerate(x["caches"]):
        ref = oracle.chunk_relattn(x["q"][b:b + 1], ck, cv, x["k_new"][b:b + 1],
                                   x["v_new"][b:b + 1], x["pos_bias_u"], x["pos_bias_v"], x["rel"])
        check_close(got[b:b + 1], ref, dtype, f"{what}, stream {b}")
    # the pools afterwards: the history untouched, the chunk appended, every other slot a canary
    kp_ref, vp_ref = x["k_pool"].copy(), x["v_pool"].copy()
    assert oracle.paged_append(syn.to_bits(x["k_new"], dtype), syn.to_bits(x["v_new"], dtype),
                               kp_ref, vp_ref, x["block_table"], x["cache_seqlens"]) == 0
    assert np.array_equal(_bits(host_pool(kp, dtype)), _bits(kp_ref)), what
    assert np.array_equal(_bits(host_pool(vp, dtype)), _bits(vp_ref)), what
    assert capi.oasr_device_status() == 0, what


def _packed_params(seed):
    rng = np.random.default_rng(30_000 + seed)
    n = int(rng.integers(1, 13))
    kinds = rng.choice(["zero", "one", "short", "long"], size=n, p=[0.1, 0.1, 0.5, 0.3])
    lengths = [0 if k == "zero" else 1 if k == "one" else
               int(rng.integers(2, 140)) if k == "short" else int(rng.integers(140, 700))
               for k in kinds]
    if max(lengths) == 0:
        lengths[0] = int(rng.integers(1, 50))
    H = int(rng.choice(H_CHOICES))
    dtype = "f32" if rng.random() < 0.2 else "bf16"
    window = None
    if rng.random() < 0.5:
        window = (int(rng.integers(1, 21)), int(rng.integers(0, 7)))
    r_extra = int(rng.integers(0, 6))
    return rng, dict(lengths=lengths, H=H, dtype=dtype, window=window, r_extra=r_extra)


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
@pytest.mark.parametrize("shape", ["whole_and_split", "all_split"])
def test_tensor_core_items_split_over_pairs(shape, fused):
    """Chunks of 33-64 frames whose (stream, head pair) items do not divide evenly over the SMs:
    the leftover items run split by key stages over CTA pairs, each CTA finishing one head of
    the item.  Cohort sizes taken from the device's SM count reach both forms (whole items plus
    split ones, every item split); cache lengths of 0 among the split items give items of one
    stage (kept whole), and a second identical call returns the same bits."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    H, T, bs = 4, 40, 16                     # two head pairs per stream
    n_items = sms + sms // 4 if shape == "whole_and_split" else max(sms // 2 - 4, 4)
    B = n_items // 2
    rng = np.random.default_rng(61 if shape == "whole_and_split" else 62)
    Cs = [int(c) for c in rng.integers(0, 300, size=B)]
    Cs[-1] = Cs[-3] = 0                      # one-stage items among the last (split) ones
    Cs[-2] = 299
    x = _stream_inputs(rng, T, bs, H, B, Cs, "bf16", 1, 0)
    d = {k: dev(x[k], "bf16") for k in ("q", "k_new", "v_new", "pos_bias_u", "pos_bias_v", "rel")}
    kp, vp = dev_pool(x["k_pool"], "bf16"), dev_pool(x["v_pool"], "bf16")
    bt = torch.from_numpy(x["block_table"]).cuda()
    cs = torch.from_numpy(x["cache_seqlens"]).cuda()
    outs = []
    for rep in range(2):
        if fused:
            if rep:   # the pool back to its state before the step
                kp.copy_(dev_pool(x["k_pool"], "bf16"))
                vp.copy_(dev_pool(x["v_pool"], "bf16"))
            outs.append(capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], kp, vp, bt, cs,
                                                   d["pos_bias_u"], d["pos_bias_v"], d["rel"]))
        else:
            if not rep:
                capi.oasr_paged_append(d["k_new"], d["v_new"], kp, vp, bt, cs)
            outs.append(capi.oasr_chunk_relattn_paged(d["q"], kp, vp, bt, cs, d["pos_bias_u"],
                                                      d["pos_bias_v"], d["rel"]))
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    got = to_np(outs[0])
    for b, (ck, cv) in enumerate(x["caches"]):
        ref = oracle.chunk_relattn(x["q"][b:b + 1], ck, cv, x["k_new"][b:b + 1],
                                   x["v_new"][b:b + 1], x["pos_bias_u"], x["pos_bias_v"], x["rel"])
        check_close(got[b:b + 1], ref, "bf16", f"{shape} B={B}, stream {b} (C={Cs[b]})")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("seed", range(24))
def test_random_packed_row(seed):
    rng, p = _packed_params(seed)
    lengths, H, dtype = p["lengths"], p["H"], p["dtype"]
    cfg = syn.PackedConfig("fuzz", num_seqs=len(lengths), min_len=1, max_len=max(lengths), H=H,
                           D=64, dtype=dtype, seed=40_000 + seed)
    x = syn.packed_inputs(cfg, lengths=lengths)
    if p["r_extra"]:
        x["rel"] = syn.normal(rng, (x["rel"].shape[0] + p["r_extra"], H, 64), dtype)
    d = {k: dev(x[k], dtype) for k in ("q", "k", "v", "pos_bias_u", "pos_bias_v", "rel")}
    cu = torch.from_numpy(x["cu_seqlens"]).cuda()
    if p["window"] is None:
        out = capi.oasr_packed_relattn_varlen(d["q"], d["k"], d["v"], cu, x["max_seqlen"],
                                              d["pos_bias_u"], d["pos_bias_v"], d["rel"])
        ref = oracle.packed_relattn(x["q"], x["k"], x["v"], x["cu_seqlens"], x["pos_bias_u"],
                                    x["pos_bias_v"], x["rel"])
    else:
        cs_, left = p["window"]
        out = capi.oasr_packed_relattn_chunked(d["q"], d["k"], d["v"], cu, x["max_seqlen"],
                                               d["pos_bias_u"], d["pos_bias_v"], d["rel"], cs_,
                                               left)
        ref = oracle.packed_relattn_chunked(x["q"], x["k"], x["v"], x["cu_seqlens"],
                                            x["pos_bias_u"], x["pos_bias_v"], x["rel"], cs_, left)
    torch.cuda.synchronize()
    check_close(to_np(out), ref, dtype, f"seed {seed} {p}")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("B,H,T,bs,cmax,seed", [
    (80, 4, 1, 8, 40, 1),       # 320 CTAs, single-frame chunks
    (96, 4, 8, 8, 120, 2),      # 384 CTAs, 8-row pages
    (64, 8, 16, 32, 250, 3),    # 512 CTAs, 32-row pages
])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_multiwave_short_histories(B, H, T, bs, cmax, seed, fused):
    """Grids of more than two CTAs per SM with short, unequal histories: the two-stage
    position-table form that three or four CTAs share an SM with."""
    rng = np.random.default_rng(50_000 + seed)
    Cs = [int(c) for c in rng.integers(0, cmax + 1, size=B)]
    x = _stream_inputs(rng, T, bs, H, B, Cs, "bf16", 1, 2)
    d = {k: dev(x[k], "bf16") for k in ("q", "k_new", "v_new", "pos_bias_u", "pos_bias_v", "rel")}
    kp, vp = dev_pool(x["k_pool"], "bf16"), dev_pool(x["v_pool"], "bf16")
    bt = torch.from_numpy(x["block_table"]).cuda()
    cs = torch.from_numpy(x["cache_seqlens"]).cuda()
    if fused:
        out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], kp, vp, bt, cs,
                                         d["pos_bias_u"], d["pos_bias_v"], d["rel"])
    else:
        capi.oasr_paged_append(d["k_new"], d["v_new"], kp, vp, bt, cs)
        out = capi.oasr_chunk_relattn_paged(d["q"], kp, vp, bt, cs, d["pos_bias_u"],
                                            d["pos_bias_v"], d["rel"])
    torch.cuda.synchronize()
    got = to_np(out)
    for b, (ck, cv) in enumerate(x["caches"]):
        ref = oracle.chunk_relattn(x["q"][b:b + 1], ck, cv, x["k_new"][b:b + 1],
                                   x["v_new"][b:b + 1], x["pos_bias_u"], x["pos_bias_v"], x["rel"])
        check_close(got[b:b + 1], ref, "bf16", f"B{B} H{H} T{T} stream {b} (C={Cs[b]})")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("B,H,T,bs,cmin,cmax,seed", [
    (40, 8, 16, 16, 300, 530, 4),    # 320 CTAs: the persistent form, one to two items per CTA
    (128, 8, 16, 32, 400, 512, 5),   # 1024 items over 304 CTAs: three to four items each
    (64, 8, 1, 8, 250, 520, 6),      # single-frame chunks, 8-row pages
    (96, 4, 11, 64, 330, 500, 7),    # ragged chunk, 64-row pages
])
@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_multiwave_long_histories(B, H, T, bs, cmin, cmax, seed, fused):
    """Grids of several waves with long, unequal histories: the persistent form, whose producer
    runs one (stream, head) item ahead of its consumers.  Every output row against the oracle,
    both pools bit for bit against the oracle's append."""
    rng = np.random.default_rng(60_000 + seed)
    Cs = [int(c) for c in rng.integers(cmin, cmax + 1, size=B)]
    x = _stream_inputs(rng, T, bs, H, B, Cs, "bf16", 0, 3)
    d = {k: dev(x[k], "bf16") for k in ("q", "k_new", "v_new", "pos_bias_u", "pos_bias_v", "rel")}
    kp, vp = dev_pool(x["k_pool"], "bf16"), dev_pool(x["v_pool"], "bf16")
    bt = torch.from_numpy(x["block_table"]).cuda()
    cs = torch.from_numpy(x["cache_seqlens"]).cuda()
    if fused:
        out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], kp, vp, bt, cs,
                                         d["pos_bias_u"], d["pos_bias_v"], d["rel"])
    else:
        capi.oasr_paged_append(d["k_new"], d["v_new"], kp, vp, bt, cs)
        out = capi.oasr_chunk_relattn_paged(d["q"], kp, vp, bt, cs, d["pos_bias_u"],
                                            d["pos_bias_v"], d["rel"])
    torch.cuda.synchronize()
    got = to_np(out)
    for b, (ck, cv) in enumerate(x["caches"]):
        ref = oracle.chunk_relattn(x["q"][b:b + 1], ck, cv, x["k_new"][b:b + 1],
                                   x["v_new"][b:b + 1], x["pos_bias_u"], x["pos_bias_v"], x["rel"])
        check_close(got[b:b + 1], ref, "bf16", f"B{B} H{H} T{T} bs{bs} stream {b} (C={Cs[b]})")
    kp_ref, vp_ref = x["k_pool"].copy(), x["v_pool"].copy()
    assert oracle.paged_append(syn.to_bits(x["k_new"], "bf16"), syn.to_bits(x["v_new"], "bf16"),
                               kp_ref, vp_ref, x["block_table"], x["cache_seqlens"]) == 0
    assert np.array_equal(host_pool(kp, "bf16"), kp_ref)
    assert np.array_equal(host_pool(vp, "bf16"), vp_ref)
    assert capi.oasr_device_status() == 0


def test_multiwave_invalid_chunk_page():
    """In a persistent grid, streams whose chunk page names no valid block take the
    write-fence-read path (their chunk keys on that page read as zeros and are flagged) while
    the streams around them keep the direct path; every other row is exact."""
    rng = np.random.default_rng(61_000)
    B, H, T, bs = 40, 8, 16, 16
    Cs = [int(c) for c in rng.integers(300, 531, size=B)]
    x = _stream_inputs(rng, T, bs, H, B, Cs, "bf16", 0, 0)
    bad = [3, 17, 38]
    bt = x["block_table"].copy()
    for b in bad:
        bt[b, (Cs[b] + T - 1) // bs] = -7      # the page holding the chunk's last row
    d = {k: dev(x[k], "bf16") for k in ("q", "k_new", "v_new", "pos_bias_u", "pos_bias_v", "rel")}
    kp, vp = dev_pool(x["k_pool"], "bf16"), dev_pool(x["v_pool"], "bf16")
    out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], kp, vp,
                                     torch.from_numpy(bt).cuda(),
                                     torch.from_numpy(x["cache_seqlens"]).cuda(),
                                     d["pos_bias_u"], d["pos_bias_v"], d["rel"])
    torch.cuda.synchronize()
    got = to_np(out)
    assert capi.oasr_device_status() & capi.STATUS_BOUNDS_BIT
    for b, (ck, cv) in enumerate(x["caches"]):
        kn, vn = x["k_new"][b:b + 1].copy(), x["v_new"][b:b + 1].copy()
        if b in bad:
            # keys on the invalid page read as zero rows
            page = (Cs[b] + T - 1) // bs
            for t in range(T):
                if (Cs[b] + t) // bs == page:
                    kn[0, t] = 0.0
                    vn[0, t] = 0.0
        ref = oracle.chunk_relattn(x["q"][b:b + 1], ck, cv, kn, vn, x["pos_bias_u"],
                                   x["pos_bias_v"], x["rel"])
        check_close(got[b:b + 1], ref, "bf16", f"stream {b} (C={Cs[b]}, bad={b in bad})")
