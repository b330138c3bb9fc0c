"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test ties one part of the oracle to a library routine, a closed form, an
invariant or a hand-worked fixture, so that a dropped term, a wrong sign or index,
or a transposed operand fails at least one of them:

* u = v = rel = 0 reduces the method to plain scaled-dot-product attention, which
  torch's own CPU routine computes (content term, softmax, P.V, scale).
* The rel-pos bias decomposes as an additive float mask to that routine (the
  content and position terms add before the softmax; u and v enter as q + u, q + v).
* One-hot tables read back which table row each (query, key) pair uses; it must
  match the hand-worked fixture (rel_shift orientation, offset z) and the fact
  that the largest distance C + T - 1 is reached only by the last query against
  the first key.
* Closed forms: a single key returns its value row exactly; two keys give a
  logistic mix with the scale applied to both terms.
* Invariants: softmax rows sum to one and are non-negative; a table of equal rows
  changes nothing; the streaming rows equal the last T rows of the packed
  attention over one segment; packing is invariant to segment order and
  concatenation.
* The paged append matches a hand-worked fixture, skips invalid blocks, and
  round-trips under any block permutation.
* The chunked-limited (Nemotron offline) mask: SDPA with the chunk window and the
  rel-pos bias as an explicit float mask; single-frame chunks return their value
  rows; one chunk per segment is the bidirectional packed attention; the rows of
  chunk c equal one streaming step with the previous `left` chunks as its cache.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_chunk_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, shape, sigma=0.125):
    return (rng.standard_normal(shape) * sigma).astype(np.float32)


def _stream_case(rng, B=2, T=3, C=5, H=2, D=8, R=None):
    R = C + 2 * T - 1 if R is None else R
    return dict(q=_rand(rng, (B, T, H, D)), cache_k=_rand(rng, (B, C, H, D)),
                cache_v=_rand(rng, (B, C, H, D)), k_new=_rand(rng, (B, T, H, D)),
                v_new=_rand(rng, (B, T, H, D)), pos_bias_u=_rand(rng, (H, D)),
                pos_bias_v=_rand(rng, (H, D)), rel=_rand(rng, (R, H, D)))


def _sdpa(q, k, v, scale, mask=None):
    """torch's CPU scaled-dot-product attention in float64; q [Lq,D], k,v [Lk,D]."""
    t = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))[None, None]
    m = None if mask is None else t(mask)
    o = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=m,
                                                         scale=scale)
    return o[0, 0].numpy()


# --------------------------------------------------------------------------- SDPA


def test_zero_bias_is_sdpa_streaming():
    rng = np.random.default_rng(1)
    c = _stream_case(rng, B=3, T=4, C=7, H=2, D=16)
    for key in ("pos_bias_u", "pos_bias_v", "rel"):
        c[key] = np.zeros_like(c[key])
    out = oracle.chunk_relattn(**c)
    scale = 1 / math.sqrt(16)
    for b in range(3):
        for h in range(2):
            K = np.concatenate([c["cache_k"][b, :, h], c["k_new"][b, :, h]])
            V = np.concatenate([c["cache_v"][b, :, h], c["v_new"][b, :, h]])
            ref = _sdpa(c["q"][b, :, h], K, V, scale)
            np.testing.assert_allclose(out[b, :, h], ref, rtol=0, atol=1e-12)


def test_zero_bias_is_sdpa_packed():
    rng = np.random.default_rng(2)
    lens = [5, 1, 9, 3]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total, H, D = int(cu[-1]), 3, 8
    q, k, v = (_rand(rng, (total, H, D)) for _ in range(3))
    z = np.zeros((H, D), np.float32)
    out = oracle.packed_relattn(q, k, v, cu, z, z, np.zeros((17, H, D), np.float32))
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        for h in range(H):
            ref = _sdpa(q[a:e, h], k[a:e, h], v[a:e, h], 1 / math.sqrt(D))
            np.testing.assert_allclose(out[a:e, h], ref, rtol=0, atol=1e-12)


def test_bias_is_additive_mask_to_sdpa():
    """(q+u).k and (q+v).r add before the softmax and share the scale.

    The table row for each pair is looked up from an explicit list of the
    distances each row holds (row 0 = the largest distance, descending by one).
    """
    rng = np.random.default_rng(3)
    B, T, C, H, D = 2, 5, 6, 2, 8
    R = C + 2 * T - 1 + 3           # a longer table than needed: only z = R - T matters
    c = _stream_case(rng, B=B, T=T, C=C, H=H, D=D, R=R)
    out = oracle.chunk_relattn(**c, scale=0.3)
    largest = R - T                 # distance held by row 0
    row_of_distance = {largest - m: m for m in range(R)}
    for b in range(B):
        for h in range(H):
            K = np.concatenate([c["cache_k"][b, :, h], c["k_new"][b, :, h]]).astype(np.float64)
            V = np.concatenate([c["cache_v"][b, :, h], c["v_new"][b, :, h]])
            qh = c["q"][b, :, h].astype(np.float64)
            qv = qh + c["pos_bias_v"][h]
            bias = np.empty((T, C + T))
            for i in range(T):
                for j in range(C + T):
                    bias[i, j] = qv[i] @ c["rel"][row_of_distance[C + i - j], h]
            ref = _sdpa(qh + c["pos_bias_u"][h], K, V, 0.3, mask=0.3 * bias)
            np.testing.assert_allclose(out[b, :, h], ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------- rel index (O1)


def _probe_rows_streaming(C, T, R, D=4):
    """Which rel row each (query, key) pair reads, recovered from outputs only."""
    H, K = 1, C + T
    assert D >= K
    scale = 1 / math.sqrt(D)
    q = np.zeros((1, T, H, D), np.float32)
    q[..., 0] = 1.0
    zeros_k = np.zeros((1, C, H, D), np.float32)
    eye = np.eye(K, D, dtype=np.float32)          # value row j = e_j, so out_i = p_i
    cache_v = eye[:C].reshape(1, C, H, D)
    v_new = eye[C:].reshape(1, T, H, D)
    z_hd = np.zeros((H, D), np.float32)
    row_of = -np.ones((T, K), dtype=np.int64)
    for m in range(R):
        rel = np.zeros((R, H, D), np.float32)
        rel[m, 0, 0] = 40.0 / scale               # scaled score 40 where row m is read
        p = oracle.chunk_relattn(q, zeros_k, cache_v, np.zeros((1, T, H, D), np.float32),
                                 v_new, z_hd, z_hd, rel)[0, :, 0, :K]
        for i in range(T):
            j = int(np.argmax(p[i]))
            if p[i, j] > 0.99:
                assert row_of[i, j] == -1, "a pair read two rows"
                row_of[i, j] = m
            else:
                np.testing.assert_allclose(p[i], 1.0 / K, atol=1e-12)
    return row_of


def test_rel_rows_match_hand_worked_fixture():
    g = json.load(open(os.path.join(GOLDEN, "relidx_tiny.json")))
    row_of = _probe_rows_streaming(g["C"], g["T"], g["R"])
    np.testing.assert_array_equal(row_of, np.array(g["row_of"]))


def test_rel_rows_extremes_and_shift():
    """Row 0 is the largest distance C+T-1 (last query, first key only); the
    last row of the minimal table is -(T-1) (first query, last key only); a
    longer table shifts every row by the extra length."""
    C, T = 3, 3
    R = C + 2 * T - 1
    row_of = _probe_rows_streaming(C, T, R, D=8)
    assert (row_of >= 0).all()
    assert row_of[T - 1, 0] == 0 and (row_of == 0).sum() == 1
    assert row_of[0, C + T - 1] == R - 1 and (row_of == R - 1).sum() == 1
    longer = _probe_rows_streaming(C, T, R + 2, D=8)
    np.testing.assert_array_equal(longer, row_of + 2)


def test_packed_rel_rows_match_fixture():
    g = json.load(open(os.path.join(GOLDEN, "relidx_tiny.json")))["packed"]
    L, R, D = g["L"], g["R"], 4
    scale = 1 / math.sqrt(D)
    cu = np.array([0, L], np.int32)
    q = np.zeros((L, 1, D), np.float32)
    q[..., 0] = 1.0
    k = np.zeros((L, 1, D), np.float32)
    v = np.eye(L, D, dtype=np.float32).reshape(L, 1, D)
    z = np.zeros((1, D), np.float32)
    row_of = -np.ones((L, L), np.int64)
    for m in range(R):
        rel = np.zeros((R, 1, D), np.float32)
        rel[m, 0, 0] = 40.0 / scale
        p = oracle.packed_relattn(q, k, v, cu, z, z, rel)[:, 0, :L]
        for i in range(L):
            j = int(np.argmax(p[i]))
            if p[i, j] > 0.99:
                row_of[i, j] = m
    np.testing.assert_array_equal(row_of, np.array(g["row_of"]))


# ----------------------------------------------------------------- closed forms


def test_single_key_returns_its_value():
    rng = np.random.default_rng(4)
    c = _stream_case(rng, B=2, T=1, C=0, H=3, D=8)
    out = oracle.chunk_relattn(**c)
    np.testing.assert_array_equal(out, c["v_new"].astype(np.float64))


def test_two_keys_position_term_closed_form():
    """T=1, C=1, zero content: weights are a logistic of scale*(v.r_row)."""
    D, H = 8, 1
    rng = np.random.default_rng(5)
    vb = _rand(rng, (H, D))
    rel = _rand(rng, (2, H, D))      # R = C + 2T - 1 = 2: row 0 = distance 1, row 1 = distance 0
    vals = _rand(rng, (2, D))
    scale = 0.7
    z = lambda *s: np.zeros(s, np.float32)
    out = oracle.chunk_relattn(z(1, 1, H, D), z(1, 1, H, D), vals[0].reshape(1, 1, H, D),
                               z(1, 1, H, D), vals[1].reshape(1, 1, H, D), z(H, D), vb, rel,
                               scale=scale)[0, 0, 0]
    a = scale * float(vb[0].astype(np.float64) @ rel[0, 0])   # key 0: distance 1 -> row 0
    b = scale * float(vb[0].astype(np.float64) @ rel[1, 0])   # key 1: distance 0 -> row 1
    w0 = 1.0 / (1.0 + math.exp(b - a))
    vals = vals.astype(np.float64)
    np.testing.assert_allclose(out, w0 * vals[0] + (1 - w0) * vals[1], rtol=0, atol=1e-14)


def test_two_keys_content_term_closed_form():
    D, H = 8, 1
    rng = np.random.default_rng(6)
    q, u = _rand(rng, (1, 1, H, D)), _rand(rng, (H, D))
    k0, k1 = _rand(rng, (1, 1, H, D)), _rand(rng, (1, 1, H, D))
    v0, v1 = _rand(rng, (1, 1, H, D)), _rand(rng, (1, 1, H, D))
    scale = 1.3
    zero = np.zeros((H, D), np.float32)
    out = oracle.chunk_relattn(q, k0, v0, k1, v1, u, zero, np.zeros((2, H, D), np.float32),
                               scale=scale)[0, 0, 0]
    qu = q[0, 0, 0].astype(np.float64) + u[0]
    a, b = scale * (qu @ k0[0, 0, 0]), scale * (qu @ k1[0, 0, 0])
    w0 = 1.0 / (1.0 + math.exp(b - a))
    v0, v1 = v0.astype(np.float64), v1.astype(np.float64)
    np.testing.assert_allclose(out, w0 * v0[0, 0, 0] + (1 - w0) * v1[0, 0, 0], atol=1e-14)


# ------------------------------------------------------------------- invariants


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(7)
    B, T, C, H, D = 2, 4, 12, 2, 16
    c = _stream_case(rng, B=B, T=T, C=C, H=H, D=D)
    c = {k: v * 8 for k, v in c.items()}       # larger scores: far from uniform
    eye = np.eye(C + T, D, dtype=np.float32)
    c["cache_v"] = np.broadcast_to(eye[:C][None, :, None, :], (B, C, H, D)).copy()
    c["v_new"] = np.broadcast_to(eye[C:][None, :, None, :], (B, T, H, D)).copy()
    p = oracle.chunk_relattn(**c)
    assert (p >= 0).all()
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-13)
    assert p.max() > 0.3                        # not trivially uniform


def test_equal_rel_rows_change_nothing():
    rng = np.random.default_rng(8)
    c = _stream_case(rng, B=2, T=4, C=6, H=2, D=8)
    base = oracle.chunk_relattn(**{**c, "rel": np.zeros_like(c["rel"])})
    row = _rand(rng, (1, 2, 8)) * 8
    const = oracle.chunk_relattn(**{**c, "rel": np.repeat(row, c["rel"].shape[0], 0)})
    np.testing.assert_allclose(const, base, atol=1e-13)


def test_streaming_rows_equal_packed_rows():
    """Chunk attention at cache C equals rows C..C+T-1 of the packed attention
    over one segment of C+T frames (same keys; the streaming table is the first
    C+2T-1 rows of the packed one)."""
    rng = np.random.default_rng(9)
    B, T, C, H, D = 1, 4, 9, 2, 8
    L = C + T
    Rp = 2 * L - 1
    relp = _rand(rng, (Rp, H, D))
    c = _stream_case(rng, B=B, T=T, C=C, H=H, D=D)
    c["rel"] = relp[: C + 2 * T - 1]
    out_s = oracle.chunk_relattn(**c)
    kk = np.concatenate([c["cache_k"][0], c["k_new"][0]])
    vv = np.concatenate([c["cache_v"][0], c["v_new"][0]])
    qq = np.concatenate([_rand(rng, (C, H, D)), c["q"][0]])
    out_p = oracle.packed_relattn(qq, kk, vv, np.array([0, L], np.int32), c["pos_bias_u"],
                                  c["pos_bias_v"], relp)
    np.testing.assert_allclose(out_s[0], out_p[C:], atol=1e-13)


def test_packing_is_concatenation_and_order_free():
    rng = np.random.default_rng(10)
    H, D = 2, 8
    lens = [7, 3, 11]
    R = 2 * 11 - 1
    u, vb, rel = _rand(rng, (H, D)), _rand(rng, (H, D)), _rand(rng, (R, H, D))
    segs = [tuple(_rand(rng, (n, H, D)) for _ in range(3)) for n in lens]

    def run(order):
        ls = [lens[s] for s in order]
        cu = np.concatenate([[0], np.cumsum(ls)]).astype(np.int32)
        cat = [np.concatenate([segs[s][t] for s in order]) for t in range(3)]
        return oracle.packed_relattn(*cat, cu, u, vb, rel), cu

    full, cu = run([0, 1, 2])
    for s in range(3):
        alone, _ = run([s])
        np.testing.assert_array_equal(full[cu[s]:cu[s + 1]], alone)
    perm, cup = run([2, 0, 1])
    np.testing.assert_array_equal(perm[cup[1]:cup[2]], full[cu[0]:cu[1]])
    np.testing.assert_array_equal(perm[cup[0]:cup[1]], full[cu[2]:cu[3]])


def test_row_subset_matches_full():
    rng = np.random.default_rng(11)
    c = _stream_case(rng, B=2, T=3, C=4, H=2, D=8)
    full = oracle.chunk_relattn(**c)
    rows = np.array([[1, 2, 0], [0, 0, 1]])
    part = oracle.chunk_relattn(**c, rows=rows)
    for b, i, h in rows:
        np.testing.assert_array_equal(part[b, i, h], full[b, i, h])
    assert np.isnan(part[0, 1, 0]).all()


def test_short_table_is_rejected():
    rng = np.random.default_rng(12)
    c = _stream_case(rng, B=1, T=3, C=4, H=1, D=4, R=4 + 2 * 3 - 2)
    with pytest.raises(ValueError):
        oracle.chunk_relattn(**c)


# ---------------------------------------------------------------------- append


def test_append_matches_hand_worked_fixture():
    g = json.load(open(os.path.join(GOLDEN, "append_tiny.json")))
    B, T, H, D = len(g["block_table"]), g["T"], 2, 3
    k_new = np.arange(B * T * H * D, dtype=np.float32).reshape(B, T, H, D) + 1
    v_new = -k_new
    shape = (g["num_blocks"], g["block_size"], H, D)
    kp, vp = np.full(shape, np.nan, np.float32), np.full(shape, np.nan, np.float32)
    skipped = oracle.paged_append(k_new, v_new, kp, vp, np.array(g["block_table"]),
                                  np.array(g["cache_seqlens"]))
    assert skipped == 0
    expect = np.full(shape, np.nan, np.float32)
    for e in g["expected_destinations"]:
        expect[e["block"], e["slot"]] = k_new[e["b"], e["t"]]
    np.testing.assert_array_equal(kp, expect)
    np.testing.assert_array_equal(vp, -expect)


def test_append_skips_invalid_blocks_and_positions():
    B, T, H, D, bs, nb = 2, 4, 1, 2, 2, 4
    k_new = np.ones((B, T, H, D), np.float32)
    bt = np.array([[0, 7], [1, 2]], np.int32)      # block 7 does not exist
    cs = np.array([0, 2], np.int32)                # stream 1 runs past its 2 table entries
    kp = np.zeros((nb, bs, H, D), np.float32)
    vp = np.zeros_like(kp)
    skipped = oracle.paged_append(k_new, k_new, kp, vp, bt, cs)
    assert skipped == 2 * H + 2 * H
    assert kp[0].sum() == 2 * D and kp[2].sum() == 2 * D and kp[1].sum() == 0
    assert kp[3].sum() == 0


def test_append_round_trips_under_any_block_permutation():
    """Appending the history chunk by chunk and reading the pool back in logical
    order gives the same sequence whatever physical blocks the table names;
    untouched blocks keep their canary."""
    rng = np.random.default_rng(13)
    B, H, D, bs, nb = 3, 2, 4, 4, 24
    steps, T = 5, 3
    seq = [_rand(rng, (B, T, H, D)) for _ in range(steps)]
    mbps = -(-steps * T // bs)
    logical = []
    for trial in range(3):
        bt = syn.block_table(rng, B, mbps, nb)
        kp = syn.canary_pool(nb, bs, H, D, "f32")
        vp = syn.canary_pool(nb, bs, H, D, "f32")
        for s in range(steps):
            cs = np.full((B,), s * T, np.int32)
            assert oracle.paged_append(seq[s], seq[s], kp, vp, bt, cs) == 0
        rows = np.stack([kp[bt[b]].reshape(-1, H, D)[: steps * T] for b in range(B)])
        logical.append(rows)
        used = np.zeros(nb, bool)
        used[bt.ravel()] = True
        assert np.isnan(kp[~used]).all()
    np.testing.assert_array_equal(logical[0], np.concatenate(seq, axis=1))
    np.testing.assert_array_equal(logical[1], logical[0])
    np.testing.assert_array_equal(logical[2], logical[0])


def test_append_bf16_bits_are_copied_exactly():
    rng = np.random.default_rng(14)
    cfg = syn.TINY
    x = syn.normal(rng, (2, 3, 4, 64), "bf16")
    bits = syn.to_bits(x, "bf16")
    np.testing.assert_array_equal(syn.from_bits(bits, "bf16"), x)
    kp = syn.canary_pool(16, 16, 4, 64, "bf16")
    vp = kp.copy()
    bt = syn.block_table(rng, 2, 8, 16)
    oracle.paged_append(bits, bits, kp, vp, bt, np.array([5, 0], np.int32))
    np.testing.assert_array_equal(kp[bt[0, 0], 5:8], bits[0])
    np.testing.assert_array_equal(kp[bt[1, 0], 0:3], bits[1])
    assert cfg.B == 2


# --------------------------------------------------- chunked-limited (Nemotron offline)


def _chunk_allowed(i, j, cs, left):
    """The chunked_limited window written out: own chunk and `left` earlier chunks."""
    ci, cj = i // cs, j // cs
    return ci - left <= cj <= ci


def _packed_case(rng, lens, H=2, D=8, extra_rows=0):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    R = 2 * max(lens) - 1 + 2 * extra_rows
    return cu, dict(q=_rand(rng, (total, H, D)), k=_rand(rng, (total, H, D)),
                    v=_rand(rng, (total, H, D)), pos_bias_u=_rand(rng, (H, D)),
                    pos_bias_v=_rand(rng, (H, D)), rel=_rand(rng, (R, H, D)))


@pytest.mark.parametrize("cs,left", [(4, 1), (3, 0), (2, 5), (5, 2)])
def test_chunked_is_sdpa_with_window_and_bias_mask(cs, left):
    rng = np.random.default_rng(21 + cs + left)
    lens = [11, 1, 7, 16]
    cu, c = _packed_case(rng, lens, extra_rows=2)
    H, D = c["q"].shape[1:]
    R = c["rel"].shape[0]
    scale = 0.35
    out = oracle.packed_relattn_chunked(c["q"], c["k"], c["v"], cu, c["pos_bias_u"],
                                        c["pos_bias_v"], c["rel"], cs, left, scale=scale)
    largest = (R - 1) // 2          # distance held by row 0 of the packed table
    row_of_distance = {largest - m: m for m in range(R)}
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        L = e - a
        for h in range(H):
            qh = c["q"][a:e, h].astype(np.float64)
            qv = qh + c["pos_bias_v"][h]
            mask = np.full((L, L), -np.inf)
            for i in range(L):
                for j in range(L):
                    if _chunk_allowed(i, j, cs, left):
                        mask[i, j] = scale * (qv[i] @ c["rel"][row_of_distance[i - j], h])
            ref = _sdpa(qh + c["pos_bias_u"][h], c["k"][a:e, h], c["v"][a:e, h], scale, mask=mask)
            np.testing.assert_allclose(out[a:e, h], ref, rtol=0, atol=1e-12)


def test_chunked_single_frame_chunks_return_values():
    rng = np.random.default_rng(31)
    cu, c = _packed_case(rng, [6, 9])
    out = oracle.packed_relattn_chunked(c["q"], c["k"], c["v"], cu, c["pos_bias_u"],
                                        c["pos_bias_v"], c["rel"], 1, 0)
    np.testing.assert_array_equal(out, c["v"].astype(np.float64))


def test_chunked_one_chunk_per_segment_is_bidirectional():
    rng = np.random.default_rng(32)
    lens = [13, 4, 20]
    cu, c = _packed_case(rng, lens)
    a = oracle.packed_relattn_chunked(c["q"], c["k"], c["v"], cu, c["pos_bias_u"],
                                      c["pos_bias_v"], c["rel"], max(lens), 0)
    b = oracle.packed_relattn(c["q"], c["k"], c["v"], cu, c["pos_bias_u"], c["pos_bias_v"],
                              c["rel"])
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


@pytest.mark.parametrize("cs,left", [(4, 2), (3, 1), (8, 7)])
def test_chunked_rows_equal_a_streaming_step(cs, left):
    """Each query block is one streaming step whose cache is the previous `left`
    chunks and whose chunk is the block's own frames (the relative table of the step
    is the slice of the packed table holding distances C+T-1 down to -(T-1))."""
    rng = np.random.default_rng(40 + cs)
    L = 5 * cs + 2                  # a partial last chunk
    cu, c = _packed_case(rng, [L])
    H, D = c["q"].shape[1:]
    Rp = c["rel"].shape[0]
    zp = (Rp - 1) // 2
    out = oracle.packed_relattn_chunked(c["q"], c["k"], c["v"], cu, c["pos_bias_u"],
                                        c["pos_bias_v"], c["rel"], cs, left)
    for ch in range((L + cs - 1) // cs):
        i0, i1 = ch * cs, min(L, (ch + 1) * cs)
        j0 = max(0, (ch - left) * cs)
        T, C = i1 - i0, i0 - j0
        Rs = C + 2 * T - 1
        # streaming row m holds distance (Rs - T) - m = C + T - 1 - m; packed row of that
        # distance is zp - (C + T - 1 - m)
        rel_s = c["rel"][zp - (C + T - 1): zp - (C + T - 1) + Rs]
        step = oracle.chunk_relattn(c["q"][None, i0:i1], c["k"][None, j0:i0], c["v"][None, j0:i0],
                                    c["k"][None, i0:i1], c["v"][None, i0:i1], c["pos_bias_u"],
                                    c["pos_bias_v"], rel_s)
        np.testing.assert_allclose(out[i0:i1], step[0], rtol=0, atol=1e-13)


# --------------------------------------------------------- fixed-window ring (eviction)


def test_window_pages_matches_the_pages_sizing():
    # "ceil(window / chunk_size) + 1 pages"; the pages' 32-stream pool of 160 pages is 5 per
    # stream, which a 4-chunk window gives
    assert oracle.window_pages(64, 16) == 5
    assert oracle.window_pages(56, 8) == 8
    assert oracle.window_pages(50, 16) == 5
    assert oracle.window_pages(0, 16) == 1


def test_window_commit_hand_worked():
    # block_size 4, window 8 frames, chunk T = 4
    bt = np.array([[10, 11, 12, 13],     # C = 8: n = 12 > 8 -> drop 1 page, C = 8
                   [20, 21, 22, 23],     # C = 4: n = 8 <= 8 -> C = 8, no rotation
                   [30, 31, 32, 33],     # C = 0: n = 4 -> C = 4
                   [40, 41, 42, 43]], np.int32)
    cs = np.array([8, 4, 0, 6], np.int32)  # C = 6: n = 10 > 8 -> d = 1 (P = 3), C = 6
    bt2, cs2 = oracle.window_commit(bt, cs, T=4, block_size=4, window_frames=8)
    np.testing.assert_array_equal(cs2, [8, 8, 4, 6])
    np.testing.assert_array_equal(bt2, [[11, 12, 10, 13],
                                        [20, 21, 22, 23],
                                        [30, 31, 32, 33],
                                        [41, 42, 40, 43]])


def test_window_commit_window_shorter_than_a_page():
    """Eviction moves whole pages: with a window shorter than a page the partly written
    newest page stays, so the cached length never goes negative (worked by hand)."""
    # n = 6 + 4 = 10 frames in pages [0, 1, 2] (page 2 holds frames 8, 9); window 1 would ask
    # for ceil(9 / 4) = 3 pages, but only the 2 full ones go: row [2, 0, 1, 3], C = 2
    bt2, cs2 = oracle.window_commit(np.array([[0, 1, 2, 3]], np.int32), np.array([6], np.int32),
                                    T=4, block_size=4, window_frames=1)
    np.testing.assert_array_equal(cs2, [2])
    np.testing.assert_array_equal(bt2, [[2, 0, 1, 3]])
    # a first chunk of 12 frames on 16-frame pages, window 3: no page is full, nothing moves
    bt2, cs2 = oracle.window_commit(np.array([[7, 8]], np.int32), np.array([0], np.int32),
                                    T=12, block_size=16, window_frames=3)
    np.testing.assert_array_equal(cs2, [12])
    np.testing.assert_array_equal(bt2, [[7, 8]])
    # n = 8 on 4-frame pages with window 0: both pages are full and both go
    bt2, cs2 = oracle.window_commit(np.array([[5, 6, 9]], np.int32), np.array([4], np.int32),
                                    T=4, block_size=4, window_frames=0)
    np.testing.assert_array_equal(cs2, [0])
    np.testing.assert_array_equal(bt2, [[5, 6, 9]])


@pytest.mark.parametrize("bs,T,window", [(16, 16, 64), (8, 16, 40), (16, 8, 48), (4, 12, 20),
                                         (4, 6, 1), (16, 12, 3), (8, 5, 0), (8, 3, 7)])
def test_window_commit_keeps_the_latest_frames_in_order(bs, T, window):
    """Track frame numbers through the paging for many steps: after every commit the cached
    frames are exactly the most recent ones, oldest first, and no block is lost.  The cached
    length is at most the window, or the frames of a partly written newest page when the
    window is shorter than a page, and never negative."""
    B, steps = 3, 12
    pages = -(-(max(window, bs) + T) // bs) + 1
    bt = np.arange(B * pages, dtype=np.int32).reshape(B, pages)
    cs = np.zeros(B, np.int32)
    slots = {}           # (block, slot) -> frame number
    frame = np.zeros(B, np.int64)
    for _ in range(steps):
        n = cs + T
        for b in range(B):
            for t in range(T):
                p = cs[b] + t
                slots[(int(bt[b, p // bs]), p % bs)] = frame[b] + t
            frame[b] += T
        bt2, cs2 = oracle.window_commit(bt, cs, T, bs, window)
        for b in range(B):
            assert sorted(bt2[b]) == sorted(bt[b])
            assert 0 <= cs2[b] <= max(window, n[b] % bs)
            assert cs2[b] >= min(frame[b], window) - bs + 1
            seen = [slots[(int(bt2[b, p // bs]), p % bs)] for p in range(cs2[b])]
            assert seen == list(range(frame[b] - cs2[b], frame[b]))
        bt, cs = bt2, cs2


# -------------------------------------------------- projections feeding the path


def test_projection_hand_worked():
    # d_model 2, H 1: q/k/v rows of w_qkv and the biases by hand
    x = np.array([[1.0, 2.0], [0.5, -1.0]])
    w_qkv = np.array([[1, 0], [0, 1],      # q = x
                      [1, 1], [1, -1],     # k = (x0 + x1, x0 - x1)
                      [2, 0], [0, 0]])     # v = (2 x0, 0)
    b = np.array([0, 0, 1, 0, 0, 3])
    pos = np.array([[3.0, 4.0]])
    w_pos = np.array([[0, 1], [1, 0]])     # swaps the two dims
    q, k, v, rel = oracle.project_qkv_pos(x, w_qkv, b, pos, w_pos, H=1)
    np.testing.assert_array_equal(q[:, 0], [[1, 2], [0.5, -1]])
    np.testing.assert_array_equal(k[:, 0], [[4, -1], [0.5, 1.5]])
    np.testing.assert_array_equal(v[:, 0], [[2, 3], [1, 3]])
    np.testing.assert_array_equal(rel[:, 0], [[4, 3]])


def test_projection_identity_weights_and_head_split():
    rng = np.random.default_rng(50)
    M, H, D, R = 5, 3, 4, 7
    dm = H * D
    x, pos = rng.standard_normal((M, dm)), rng.standard_normal((R, dm))
    b = rng.standard_normal(3 * dm)
    eye = np.eye(dm)
    q, k, v, rel = oracle.project_qkv_pos(x, np.concatenate([eye, 2 * eye, -eye]), b, pos, eye, H)
    np.testing.assert_allclose(q.reshape(M, dm), x + b[:dm], atol=1e-15)
    np.testing.assert_allclose(k.reshape(M, dm), 2 * x + b[dm:2 * dm], atol=1e-15)
    np.testing.assert_allclose(v.reshape(M, dm), -x + b[2 * dm:], atol=1e-15)
    np.testing.assert_allclose(rel.reshape(R, dm), pos, atol=1e-15)
    # head h holds dims [h*D, (h+1)*D)
    np.testing.assert_array_equal(q[:, 1], (x + b[:dm])[:, D:2 * D])


def test_projection_is_affine():
    rng = np.random.default_rng(51)
    M, H, D, R = 4, 2, 8, 3
    dm = H * D
    w_qkv, w_pos = rng.standard_normal((3 * dm, dm)), rng.standard_normal((dm, dm))
    b = rng.standard_normal(3 * dm)
    x1, x2 = rng.standard_normal((M, dm)), rng.standard_normal((M, dm))
    p1, p2 = rng.standard_normal((R, dm)), rng.standard_normal((R, dm))
    z = np.zeros(3 * dm)
    a = oracle.project_qkv_pos(x1 + x2, w_qkv, b, p1 + p2, w_pos, H)
    s1 = oracle.project_qkv_pos(x1, w_qkv, b, p1, w_pos, H)
    s2 = oracle.project_qkv_pos(x2, w_qkv, z, p2, w_pos, H)
    for t, u, w in zip(a, s1, s2):
        np.testing.assert_allclose(t, u + w, atol=1e-12)
