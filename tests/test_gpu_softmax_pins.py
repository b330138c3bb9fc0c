"""GPU pins of the softmax and of the rel-row index, through the C ABI.

Scheduler page, section 4.3: the score is the content score plus matrix_bd / sqrt(d_k);
Model Layer page, Nemotron ASR section: the rel_shift order of the table rows.

Peaked softmax.  The random parity inputs (N(0,1)/8) give nearly uniform softmax rows, so
they never make a running maximum jump.  Here every input is a multiple of 1/4 (exact in
bf16, and every score is exact in fp32), the scale is 1/4, and the key rows are multiplied by
1, 2 and 4 over the first, second and last third of each stream's or segment's keys
("late": the row maxima arrive in later stages, rising by far more than 2^8 from the first
stage, so every kernel's rescale of its running output and sum is taken, and in the
streaming kernels the partial states that the consumer warps combine have very different
maxima), or by 4, 2, 1 ("early": later keys underflow next to the first stage's maximum).
Outputs are O(1), so they are gated on the stated 2e-2 bar plus an rms-relative bound.

One-hot rel probe.  q = e_0, u = v = 0, k = 0, and the table is zero except one row m0 of
head h, 40 sqrt(D) e_0: the pair (query i, key j) that reads row m0 scores 40 and every other
pair 0, so the output of query i is the value row of that key, or the mean of the value rows
when no key of the query reads row m0.  Value row j holds the bits of j + 1 in its first 11
dims, so the key is read back from the output.  Sweeping m0 over every row of the table
(one head per m0, eight at a time) recovers the whole (query, key) -> row map the kernel
uses; it must equal the oracle's and, on the hand-worked geometry, the fixture's.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_chunk_gb300 import capi
from paged_kv_chunk_gb300 import synthetic as syn

from helpers import TOL_BF16, TOL_F32, dev, dev_pool, to_np

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
PEAK_SCALE = 0.25
PEAK_RMS_REL = 1e-2     # rms(gpu - oracle) / rms(oracle) on O(1) outputs
BITS = 11               # value dims that carry the key number (keys < 2047)


@pytest.fixture(autouse=True)
def _clean_status():
    capi.oasr_device_status(clear=True)
    yield


def _gate(got, ref, dtype, what):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    max_abs = float(err.max())
    rms_rel = float(np.sqrt(np.mean(err ** 2)) / max(np.sqrt(np.mean(ref ** 2)), 1e-30))
    if dtype == "f32":
        assert max_abs <= TOL_F32, f"{what}: max abs err {max_abs:.3e}"
    else:
        assert max_abs <= TOL_BF16, f"{what}: max abs err {max_abs:.3e}"
        assert rms_rel <= PEAK_RMS_REL, f"{what}: rms-relative err {rms_rel:.3e}"
    return max_abs, rms_rel


def _key_gain(n_keys, order):
    """Per-key multiplier 1, 2, 4 over thirds of the keys (reversed for 'early')."""
    g = np.float32(2.0) ** np.minimum(3 * np.arange(n_keys) // max(n_keys, 1), 2).astype(np.float32)
    return g if order == "late" else g[::-1].copy()


def _log2_scores(qu, kk, qv, rr):
    """Scores of one (stream, head) in log2 units, for checking the inputs' design only."""
    return PEAK_SCALE * math.log2(math.e) * (qu @ kk.T + qv @ rr.T)


# ----------------------------------------------------------------- peaked, streaming


def _peaked_stream(rng, B, T, C, H, bs, dtype, order):
    K = C + T
    gain = _key_gain(K, order)[None, :, None, None]
    keys = syn.quarters(rng, (B, K, H, 64)) * gain
    vals = syn.quarters(rng, (B, K, H, 64))
    R = C + 2 * T - 1
    x = {
        "q": syn.quarters(rng, (B, T, H, 64)),
        "pos_bias_u": syn.quarters(rng, (H, 64)),
        "pos_bias_v": syn.quarters(rng, (H, 64)),
        "rel": syn.quarters(rng, (R, H, 64)),
        "cache_k": keys[:, :C], "k_new": keys[:, C:],
        "cache_v": vals[:, :C], "v_new": vals[:, C:],
    }
    mbps = -(-K // bs)
    nb = 2 * B * mbps
    x["block_table"] = syn.block_table(rng, B, mbps, nb)
    x["cache_seqlens"] = np.full(B, C, np.int32)
    kp = syn.canary_pool(nb, bs, H, 64, dtype)
    vp = syn.canary_pool(nb, bs, H, 64, dtype)
    if C:
        assert oracle.paged_append(syn.to_bits(x["cache_k"], dtype), syn.to_bits(x["cache_v"], dtype),
                                   kp, vp, x["block_table"], np.zeros(B, np.int32)) == 0
    x["k_pool"], x["v_pool"] = kp, vp
    return x


def _stream_rise(x, T, C):
    """Fraction of the output rows whose maximum over all keys exceeds their maximum over the
    first 64 keys by more than 8 (log2 units)."""
    K = C + T
    z = len(x["rel"]) - T
    rows = np.array([[z - (C + i - j) for j in range(K)] for i in range(T)])
    B, H = x["q"].shape[0], x["q"].shape[2]
    risen = []
    for b in range(B):
        for h in range(H):
            kk = np.concatenate([x["cache_k"][b, :, h], x["k_new"][b, :, h]]).astype(np.float64)
            q = x["q"][b, :, h].astype(np.float64)
            for i in range(T):
                s = _log2_scores(q[i] + x["pos_bias_u"][h], kk, q[i] + x["pos_bias_v"][h],
                                 x["rel"][rows[i], h].astype(np.float64))
                risen.append(s.max() - s[:64].max() > 8.0)
    return float(np.mean(risen))


@pytest.mark.parametrize("T,C", [(1, 0), (1, 300), (1, 530), (16, 0), (16, 300), (16, 530),
                                 (64, 0), (64, 300), (64, 530), (4, 120), (32, 200)], ids=str)
@pytest.mark.parametrize("order", ["late", "early"])
@pytest.mark.parametrize("mode", ["fused", "two_calls", "f32"])
def test_peaked_streaming(T, C, order, mode):
    dtype = "f32" if mode == "f32" else "bf16"
    rng = np.random.default_rng(7000 + 3 * T + C)
    B, H, bs = 2, 2, 16
    x = _peaked_stream(rng, B, T, C, H, bs, dtype, order)
    if order == "late" and C + T >= 192:
        assert _stream_rise(x, T, C) >= 0.75, "inputs do not make the row maxima rise"
    d = {k: dev(x[k], dtype) for k in ("q", "k_new", "v_new", "pos_bias_u", "pos_bias_v", "rel")}
    kp, vp = dev_pool(x["k_pool"], dtype), dev_pool(x["v_pool"], dtype)
    bt = torch.from_numpy(x["block_table"]).cuda()
    cs = torch.from_numpy(x["cache_seqlens"]).cuda()
    if mode == "two_calls":
        capi.oasr_paged_append(d["k_new"], d["v_new"], kp, vp, bt, cs)
        out = capi.oasr_chunk_relattn_paged(d["q"], kp, vp, bt, cs, d["pos_bias_u"],
                                            d["pos_bias_v"], d["rel"], scale=PEAK_SCALE)
    else:
        out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], kp, vp, bt, cs,
                                         d["pos_bias_u"], d["pos_bias_v"], d["rel"],
                                         scale=PEAK_SCALE)
    torch.cuda.synchronize()
    ref = oracle.chunk_relattn(x["q"], x["cache_k"], x["cache_v"], x["k_new"], x["v_new"],
                               x["pos_bias_u"], x["pos_bias_v"], x["rel"], scale=PEAK_SCALE)
    assert np.abs(ref).max() > 0.25, "outputs are not O(1)"
    _gate(to_np(out), ref, dtype, f"T={T} C={C} {order} {mode}")
    assert capi.oasr_device_status() == 0


@pytest.mark.parametrize("fused", [False, True], ids=["two_calls", "fused"])
def test_peaked_streaming_multiwave(fused):
    """A grid of more than two CTAs per SM with a short history: the two-stage position-table
    form that three or four CTAs share an SM with."""
    rng = np.random.default_rng(7050)
    B, H, T, C, bs = 40, 8, 8, 184, 8
    x = _peaked_stream(rng, B, T, C, H, bs, "bf16", "late")
    d = {k: dev(x[k], "bf16") for k in ("q", "k_new", "v_new", "pos_bias_u", "pos_bias_v", "rel")}
    kp, vp = dev_pool(x["k_pool"], "bf16"), dev_pool(x["v_pool"], "bf16")
    bt = torch.from_numpy(x["block_table"]).cuda()
    cs = torch.from_numpy(x["cache_seqlens"]).cuda()
    if fused:
        out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], kp, vp, bt, cs,
                                         d["pos_bias_u"], d["pos_bias_v"], d["rel"],
                                         scale=PEAK_SCALE)
    else:
        capi.oasr_paged_append(d["k_new"], d["v_new"], kp, vp, bt, cs)
        out = capi.oasr_chunk_relattn_paged(d["q"], kp, vp, bt, cs, d["pos_bias_u"],
                                            d["pos_bias_v"], d["rel"], scale=PEAK_SCALE)
    torch.cuda.synchronize()
    ref = oracle.chunk_relattn(x["q"], x["cache_k"], x["cache_v"], x["k_new"], x["v_new"],
                               x["pos_bias_u"], x["pos_bias_v"], x["rel"], scale=PEAK_SCALE)
    _gate(to_np(out), ref, "bf16", f"multiwave fused={fused}")
    assert capi.oasr_device_status() == 0


# ------------------------------------------------------------------- peaked, packed


def _peaked_packed(rng, lengths, H, dtype, order):
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    total = int(cu[-1])
    gain = np.concatenate([_key_gain(L, order) for L in lengths])[:, None, None]
    R = 2 * max(lengths) - 1
    return {
        "q": syn.quarters(rng, (total, H, 64)),
        "k": syn.quarters(rng, (total, H, 64)) * gain,
        "v": syn.quarters(rng, (total, H, 64)),
        "cu_seqlens": cu,
        "pos_bias_u": syn.quarters(rng, (H, 64)),
        "pos_bias_v": syn.quarters(rng, (H, 64)),
        "rel": syn.quarters(rng, (R, H, 64)),
        "max_seqlen": max(lengths),
    }


PACKED_LENGTHS = [1, 130, 700, 257]


@pytest.mark.parametrize("window", [None, (8, 7), (64, 4)], ids=["bidirectional", "cs8_left7",
                                                                 "cs64_left4"])
@pytest.mark.parametrize("order", ["late", "early"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_peaked_packed(window, order, dtype):
    rng = np.random.default_rng(7100 + (0 if window is None else window[0]))
    H = 2
    x = _peaked_packed(rng, PACKED_LENGTHS, H, dtype, order)
    if order == "late" and window is None:
        # the 700-frame segment: rows whose maximum rises by more than 2^8 after its first
        # 128-key stage
        s0 = int(x["cu_seqlens"][2])
        q = x["q"][s0:s0 + 700, 0].astype(np.float64)
        k = x["k"][s0:s0 + 700, 0].astype(np.float64)
        s = PEAK_SCALE * math.log2(math.e) * ((q + x["pos_bias_u"][0]) @ k.T)
        assert (s.max(1) - s[:, :128].max(1) > 8.0).mean() > 0.9
    d = {k: dev(x[k], dtype) for k in ("q", "k", "v", "pos_bias_u", "pos_bias_v", "rel")}
    cu = torch.from_numpy(x["cu_seqlens"]).cuda()
    args = (x["q"], x["k"], x["v"], x["cu_seqlens"], x["pos_bias_u"], x["pos_bias_v"], x["rel"])
    if window is None:
        out = capi.oasr_packed_relattn_varlen(d["q"], d["k"], d["v"], cu, x["max_seqlen"],
                                              d["pos_bias_u"], d["pos_bias_v"], d["rel"],
                                              scale=PEAK_SCALE)
        ref = oracle.packed_relattn(*args, scale=PEAK_SCALE)
    else:
        out = capi.oasr_packed_relattn_chunked(d["q"], d["k"], d["v"], cu, x["max_seqlen"],
                                               d["pos_bias_u"], d["pos_bias_v"], d["rel"],
                                               window[0], window[1], scale=PEAK_SCALE)
        ref = oracle.packed_relattn_chunked(*args, window[0], window[1], scale=PEAK_SCALE)
    torch.cuda.synchronize()
    assert np.abs(ref).max() > 0.25
    _gate(to_np(out), ref, dtype, f"{window} {order} {dtype}")
    assert capi.oasr_device_status() == 0


# --------------------------------------------------------------- one-hot rel probe


def _value_bits(n_keys):
    """Value rows that carry their key number: dim d of row j is bit d of j + 1."""
    j = np.arange(n_keys)[:, None] + 1
    v = np.zeros((n_keys, 64), np.float32)
    v[:, :BITS] = (j >> np.arange(BITS)[None, :]) & 1
    return v


def _decode(out_rows):
    """[n, 64] outputs -> key number per row, or -1 where the row is not one value row."""
    o = out_rows[:, :BITS]
    hit = np.all(np.abs(o - np.round(o)) < 1e-3, axis=1) & np.all(np.abs(out_rows[:, BITS:]) < 1e-3,
                                                                   axis=1)
    key = (np.round(o).astype(np.int64) << np.arange(BITS)[None, :]).sum(1) - 1
    return np.where(hit, key, -1)


def _one_hot_rel(R, H, m0s):
    rel = np.zeros((R, H, 64), np.float32)
    for h, m in enumerate(m0s):
        if m is not None:
            rel[m, h, 0] = 40.0 * math.sqrt(64)
    return rel


def _probe_streaming(T, C, bs, fused, H=8):
    """Row map [T, C+T] of one stream (rel row of each (query, key) pair; -1 if none) as read
    back from the kernel and from the oracle."""
    K, R = C + T, C + 2 * T - 1
    vals = _value_bits(K)[None, :, None, :].repeat(H, 2)        # [1, K, H, 64]
    q = np.zeros((1, T, H, 64), np.float32)
    q[..., 0] = 1.0
    zeros_hd = np.zeros((H, 64), np.float32)
    mbps = -(-K // bs)
    nb = 3 * mbps
    rng = np.random.default_rng(T * 1000 + C)
    bt = syn.block_table(rng, 1, mbps, nb)
    cs = np.full(1, C, np.int32)
    kp = syn.canary_pool(nb, bs, H, 64, "bf16")
    vp = syn.canary_pool(nb, bs, H, 64, "bf16")
    if C:
        oracle.paged_append(syn.to_bits(np.zeros((1, C, H, 64), np.float32), "bf16"),
                            syn.to_bits(vals[:, :C], "bf16"), kp, vp, bt, np.zeros(1, np.int32))
    d_kp, d_vp = dev_pool(kp, "bf16"), dev_pool(vp, "bf16")
    d_bt, d_cs = torch.from_numpy(bt).cuda(), torch.from_numpy(cs).cuda()
    d_q, d_z = dev(q, "bf16"), dev(zeros_hd, "bf16")
    d_kn = dev(np.zeros((1, T, H, 64), np.float32), "bf16")
    d_vn = dev(vals[:, C:], "bf16")
    got_map = -np.ones((T, K), np.int64)
    ref_map = -np.ones((T, K), np.int64)
    for g0 in range(0, R, H):
        m0s = [m if m < R else None for m in range(g0, g0 + H)]
        rel = _one_hot_rel(R, H, m0s)
        d_rel = dev(rel, "bf16")
        if fused:
            out = capi.oasr_chunk_step_paged(d_q, d_kn, d_vn, d_kp, d_vp, d_bt, d_cs, d_z, d_z, d_rel)
        else:
            if g0 == 0:
                capi.oasr_paged_append(d_kn, d_vn, d_kp, d_vp, d_bt, d_cs)
            out = capi.oasr_chunk_relattn_paged(d_q, d_kp, d_vp, d_bt, d_cs, d_z, d_z, d_rel)
        torch.cuda.synchronize()
        got = to_np(out)[0]                                       # [T, H, 64]
        ref = oracle.chunk_relattn(q, np.zeros((1, C, H, 64), np.float32), vals[:, :C],
                                   np.zeros((1, T, H, 64), np.float32), vals[:, C:], zeros_hd,
                                   zeros_hd, rel)[0]
        for h, m in enumerate(m0s):
            if m is None:
                continue
            gk, rk = _decode(got[:, h]), _decode(ref[:, h])
            np.testing.assert_array_equal(gk, rk, err_msg=f"rel row {m}: keys read")
            hit = rk >= 0
            np.testing.assert_allclose(got[hit, h], ref[hit, h], rtol=0, atol=1e-6)
            # rows with no key on row m0 return the mean of their values
            np.testing.assert_allclose(got[~hit, h], ref[~hit, h], rtol=0, atol=4e-3)
            for i in np.nonzero(hit)[0]:
                assert got_map[i, gk[i]] == -1, "a pair read two rows"
                got_map[i, gk[i]] = m
                ref_map[i, rk[i]] = m
    assert capi.oasr_device_status() == 0
    return got_map, ref_map


def test_one_hot_rel_rows_match_fixture():
    g = json.load(open(os.path.join(GOLDEN, "relidx_tiny.json")))
    for fused in (False, True):
        got_map, ref_map = _probe_streaming(g["T"], g["C"], 8, fused, H=4)
        np.testing.assert_array_equal(got_map, np.array(g["row_of"]))
        np.testing.assert_array_equal(ref_map, got_map)


@pytest.mark.parametrize("T,C,bs", [(1, 0, 16), (1, 300, 16), (1, 530, 16), (16, 0, 16),
                                    (16, 300, 16), (16, 530, 16), (32, 0, 16), (32, 500, 16),
                                    (24, 301, 8), (64, 0, 16), (64, 300, 32), (64, 530, 16)],
                         ids=str)
def test_one_hot_rel_rows_streaming(T, C, bs):
    """Every (query, key) pair reads exactly one table row, the one the oracle reads."""
    got_map, ref_map = _probe_streaming(T, C, bs, fused=(T + C) % 2 == 0)
    assert (got_map >= 0).all(), "a pair read no row"
    np.testing.assert_array_equal(got_map, ref_map)


def _probe_packed(lengths, window, H=8):
    """Row maps [L, L] of every segment of two or more frames, as read back from the kernel
    and from the oracle; every output is also compared element-wise with the oracle."""
    cu = np.zeros(len(lengths) + 1, np.int32)
    cu[1:] = np.cumsum(lengths)
    total, Lmax = int(cu[-1]), max(lengths)
    R = 2 * Lmax - 1
    v = np.concatenate([_value_bits(L) for L in lengths])[:, None, :].repeat(H, 1)
    q = np.zeros((total, H, 64), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((total, H, 64), np.float32)
    z = np.zeros((H, 64), np.float32)
    d_q, d_k, d_v, d_z = dev(q, "bf16"), dev(k, "bf16"), dev(v, "bf16"), dev(z, "bf16")
    d_cu = torch.from_numpy(cu).cuda()
    maps_got = [-np.ones((L, L), np.int64) for L in lengths]
    maps_ref = [-np.ones((L, L), np.int64) for L in lengths]
    for g0 in range(0, R, H):
        m0s = [m if m < R else None for m in range(g0, g0 + H)]
        rel = _one_hot_rel(R, H, m0s)
        d_rel = dev(rel, "bf16")
        if window is None:
            out = capi.oasr_packed_relattn_varlen(d_q, d_k, d_v, d_cu, Lmax, d_z, d_z, d_rel)
            ref = oracle.packed_relattn(q, k, v, cu, z, z, rel)
        else:
            out = capi.oasr_packed_relattn_chunked(d_q, d_k, d_v, d_cu, Lmax, d_z, d_z, d_rel,
                                                   window[0], window[1])
            ref = oracle.packed_relattn_chunked(q, k, v, cu, z, z, rel, window[0], window[1])
        torch.cuda.synchronize()
        got = to_np(out)
        for h, m in enumerate(m0s):
            if m is None:
                continue
            gk, rk = _decode(got[:, h]), _decode(ref[:, h])
            np.testing.assert_array_equal(gk, rk, err_msg=f"rel row {m}: keys read")
            hit = rk >= 0
            np.testing.assert_allclose(got[hit, h], ref[hit, h], rtol=0, atol=1e-6)
            np.testing.assert_allclose(got[~hit, h], ref[~hit, h], rtol=0, atol=4e-3)
            for s, L in enumerate(lengths):
                if L < 2:
                    continue   # one key: its value row is the output whichever row is hit
                for i in range(L):
                    key = gk[cu[s] + i]
                    if key >= 0:
                        assert maps_got[s][i, key] == -1, "a pair read two rows"
                        maps_got[s][i, key] = m
                        maps_ref[s][i, rk[cu[s] + i]] = m
    assert capi.oasr_device_status() == 0
    return maps_got, maps_ref


def test_one_hot_rel_rows_packed_fixture():
    g = json.load(open(os.path.join(GOLDEN, "relidx_tiny.json")))["packed"]
    got, ref = _probe_packed([g["L"]], None, H=4)
    np.testing.assert_array_equal(got[0], np.array(g["row_of"]))
    np.testing.assert_array_equal(ref[0], got[0])


@pytest.mark.parametrize("window", [None, (8, 7)], ids=["bidirectional", "cs8_left7"])
def test_one_hot_rel_rows_packed(window):
    lengths = [1, 130, 700]
    got, ref = _probe_packed(lengths, window)
    for s, L in enumerate(lengths):
        if L < 2:
            continue   # compared element-wise only (a single key's value is every output)
        np.testing.assert_array_equal(got[s], ref[s], err_msg=f"segment {s}")
        if window is None:
            assert (got[s] >= 0).all(), f"segment {s}: a pair read no row"
        else:
            cs_, left = window
            i, j = np.meshgrid(np.arange(L), np.arange(L), indexing="ij")
            visible = (j // cs_ >= i // cs_ - left) & (j // cs_ <= i // cs_)
            assert ((got[s] >= 0) == visible).all(), f"segment {s}: pairs outside the window"
