"""Plain fp64 CPU oracle for the paged-KV chunk attention with a shared
Transformer-XL relative-position term.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``paged_kv_chunk_gb300``) and imports nothing from it.

The arithmetic lives in ``oasr_oracle.c`` (plain loops in double); this module
only builds it with the host C compiler and marshals numpy arrays into it.

Sources (OASR documentation pages):
  * Scheduler page, section 4.3 "Heterogeneous-offset batching": the score is the
    content score plus the rel-pos bias matrix_bd / sqrt(d_k), masked per stream
    by its cache_seqlens.
  * Model Layer page, table "Three optional encoder declarations", row
    fixed_attention_window: one Transformer-XL table whose distances are
    cache + i - j, shared by a cohort with uniform cache_seqlens.
  * Model Layer page, Nemotron ASR section: Transformer-XL relative position
    with rel_shift (row 0 of the table holds the largest distance).
  * ASR Engine page, section 4.3 "Batched paged forward": block_table (B,
    blocks_per_seq) and cache_seqlens (B,) shared by all layers; the caller
    commits the cache length after the step.
  * ASR Engine page, section 4.1: packed micro-batches are one gapless
    varlen-attention row.
  * ASR Engine page, KV-pool sizing paragraphs: an encoder with a trained attention
    window pages by chunk and retains ceil(window / chunk) + 1 pages per stream; with
    history eviction the cached length is held at the window (window_commit below,
    plain Python index bookkeeping).

Parity pins (what ties this oracle to something other than itself) live in
``tests/test_oracle_pins.py``; every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oasr_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboasr_oracle.so")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oasr_oracle.c`` into ``oracle/_build/liboasr_oracle.so``.

    Uses gcc with OpenMP when the compiler accepts it, else a serial build.
    Returns the path of the shared library.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c99", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        L = ctypes.c_long
        Dbl = ctypes.c_double
        lib.oracle_paged_append.restype = L
        lib.oracle_paged_append.argtypes = [P, P, P, P, I, I, P, I, P, I, I, I, I, I]
        lib.oracle_chunk_relattn.restype = L
        lib.oracle_chunk_relattn.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I,
                                             Dbl, P, L, P]
        lib.oracle_packed_relattn.restype = L
        lib.oracle_packed_relattn.argtypes = [P, P, P, P, I, I, P, P, P, I, I, I, Dbl,
                                              P, L, P]
        lib.oracle_packed_relattn_chunked.restype = L
        lib.oracle_packed_relattn_chunked.argtypes = [P, P, P, P, I, I, P, P, P, I, I, I, Dbl,
                                                      I, I, P, L, P]
        lib.oracle_num_threads.restype = I
        lib.oracle_num_threads.argtypes = []
        lib.oracle_set_num_threads.restype = None
        lib.oracle_set_num_threads.argtypes = [I]
        _lib = lib
        return lib


def _f32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """Threads the compiled oracle uses (OpenMP max threads, or 1)."""
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads for the oracle's later calls (for timing; the results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))


def paged_append(k_new, v_new, k_pool, v_pool, block_table, cache_seqlens) -> int:
    """Write the chunk rows into the pools in place (byte copy); see the C file.

    k_new, v_new: [B, T, H, D]; k_pool, v_pool: [num_blocks, bs, H, D] of the
    same dtype (any fixed-size dtype: float32, or uint16 holding bf16 bits);
    block_table: int32 [B, max_blocks_per_seq]; cache_seqlens: int32 [B].
    Returns the number of (b, t, h) rows that were not written because their
    block lies outside the table or the pool.
    """
    lib = _load()
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new, dtype=k_new.dtype)
    for pool in (k_pool, v_pool):
        if not (pool.flags.c_contiguous and pool.dtype == k_new.dtype):
            raise ValueError("pools must be C-contiguous and of the chunk's dtype")
    B, T, H, D = k_new.shape
    nb, bs, H2, D2 = k_pool.shape
    if (H2, D2) != (H, D) or v_pool.shape != k_pool.shape:
        raise ValueError("pool shape does not match the chunk")
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cs = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    if bt.ndim != 2 or bt.shape[0] != B or cs.shape != (B,):
        raise ValueError("block_table must be [B, max_blocks_per_seq], cache_seqlens [B]")
    return int(lib.oracle_paged_append(_ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                       nb, bs, _ptr(bt), bt.shape[1], _ptr(cs),
                                       B, T, H, D, k_new.dtype.itemsize))


def chunk_relattn(q, cache_k, cache_v, k_new, v_new, pos_bias_u, pos_bias_v, rel,
                  scale=None, rows=None) -> np.ndarray:
    """Streaming chunk attention over an un-paged cache, in float64.

    q, k_new, v_new: [B, T, H, D]; cache_k, cache_v: [B, C, H, D] (C may be 0);
    pos_bias_u, pos_bias_v: [H, D]; rel: [R, H, D] with R >= C + 2T - 1 and
    z = R - T.  scale defaults to 1/sqrt(D).  rows: optional int array [n, 3]
    of (b, i, h) to compute; other rows of the result are NaN.
    Returns out [B, T, H, D] float64.
    """
    lib = _load()
    q = _f32(q)
    B, T, H, D = q.shape
    k_new, v_new = _f32(k_new), _f32(v_new)
    cache_k, cache_v = _f32(cache_k), _f32(cache_v)
    C = cache_k.shape[1]
    if cache_k.shape != (B, C, H, D) or cache_v.shape != (B, C, H, D):
        raise ValueError("cache must be [B, C, H, D]")
    if k_new.shape != q.shape or v_new.shape != q.shape:
        raise ValueError("k_new, v_new must be [B, T, H, D]")
    u, vb, rel = _f32(pos_bias_u), _f32(pos_bias_v), _f32(rel)
    if u.shape != (H, D) or vb.shape != (H, D) or rel.ndim != 3 or rel.shape[1:] != (H, D):
        raise ValueError("pos biases must be [H, D] and rel [R, H, D]")
    R = rel.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.full((B, T, H, D), np.nan, dtype=np.float64)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
        rp, nr = _ptr(rows), rows.shape[0]
    else:
        rp, nr = None, 0
    bad = lib.oracle_chunk_relattn(_ptr(q), _ptr(cache_k), _ptr(cache_v), _ptr(k_new),
                                   _ptr(v_new), _ptr(u), _ptr(vb), _ptr(rel), R, B, T, C,
                                   H, D, float(scale), rp, nr, _ptr(out))
    if bad:
        raise ValueError(f"rel table too short: {bad} rows need rows outside [0, {R})")
    return out


def packed_relattn(q, k, v, cu_seqlens, pos_bias_u, pos_bias_v, rel, scale=None,
                   rows=None) -> np.ndarray:
    """Packed varlen bidirectional attention over one gapless row, in float64.

    q, k, v: [total, H, D]; cu_seqlens: int [num_seqs + 1] starting at 0;
    rel: [R, H, D] with z = (R - 1) // 2 and R >= 2 * max_seqlen - 1.
    rows: optional int array [n, 2] of (token, h); other rows are NaN.
    Returns out [total, H, D] float64.
    """
    lib = _load()
    q, k, v = _f32(q), _f32(k), _f32(v)
    total, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share their shape")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    if cu.ndim != 1 or cu.shape[0] < 1 or cu[0] != 0 or cu[-1] != total or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, end at total and not decrease")
    u, vb, rel = _f32(pos_bias_u), _f32(pos_bias_v), _f32(rel)
    if u.shape != (H, D) or vb.shape != (H, D) or rel.ndim != 3 or rel.shape[1:] != (H, D):
        raise ValueError("pos biases must be [H, D] and rel [R, H, D]")
    R = rel.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.full((total, H, D), np.nan, dtype=np.float64)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        rp, nr = _ptr(rows), rows.shape[0]
    else:
        rp, nr = None, 0
    bad = lib.oracle_packed_relattn(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), cu.shape[0] - 1,
                                    total, _ptr(u), _ptr(vb), _ptr(rel), R, H, D,
                                    float(scale), rp, nr, _ptr(out))
    if bad:
        raise ValueError(f"{bad} rows need rel rows outside [0, {R}) or lie in no segment")
    return out


def packed_relattn_chunked(q, k, v, cu_seqlens, pos_bias_u, pos_bias_v, rel, chunk_size,
                           left_chunks, scale=None, rows=None) -> np.ndarray:
    """Chunked-limited packed attention (the Nemotron offline mask), in float64.

    As packed_relattn, but query i of a segment sees key j only when
    i // chunk_size - left_chunks <= j // chunk_size <= i // chunk_size (positions local to
    the segment).  Other rows than `rows` are NaN.
    """
    lib = _load()
    if chunk_size < 1 or left_chunks < 0:
        raise ValueError("chunk_size must be >= 1 and left_chunks >= 0")
    q, k, v = _f32(q), _f32(k), _f32(v)
    total, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share their shape")
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    if cu.ndim != 1 or cu.shape[0] < 1 or cu[0] != 0 or cu[-1] != total or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, end at total and not decrease")
    u, vb, rel = _f32(pos_bias_u), _f32(pos_bias_v), _f32(rel)
    if u.shape != (H, D) or vb.shape != (H, D) or rel.ndim != 3 or rel.shape[1:] != (H, D):
        raise ValueError("pos biases must be [H, D] and rel [R, H, D]")
    R = rel.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.full((total, H, D), np.nan, dtype=np.float64)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        rp, nr = _ptr(rows), rows.shape[0]
    else:
        rp, nr = None, 0
    bad = lib.oracle_packed_relattn_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), cu.shape[0] - 1,
                                            total, _ptr(u), _ptr(vb), _ptr(rel), R, H, D,
                                            float(scale), int(chunk_size), int(left_chunks), rp, nr,
                                            _ptr(out))
    if bad:
        raise ValueError(f"{bad} rows need rel rows outside [0, {R}) or lie in no segment")
    return out


def window_pages(window_frames: int, chunk_frames: int) -> int:
    """Pages a stream retains with a trained window when it pages by chunk:
    ceil(window / chunk) + 1 (the history plus the chunk being appended)."""
    if window_frames < 0 or chunk_frames < 1:
        raise ValueError("window_frames >= 0 and chunk_frames >= 1 required")
    return -(-window_frames // chunk_frames) + 1


def window_commit(block_table, cache_seqlens, T: int, block_size: int, window_frames: int):
    """Commit a step's chunk with history eviction, per stream (the caller-side commit of the
    ASR Engine page, section 4.3, plus the eviction that holds a trained window).

    After the chunk the stream holds n = cache_seqlens[b] + T frames in its first
    P = ceil(n / block_size) pages.  If n exceeds window_frames, the oldest
    d = ceil((n - window_frames) / block_size) pages are dropped, but never more than the
    floor(n / block_size) full ones: eviction moves whole pages, so a partly written newest
    page stays even when the window is shorter than a page (the cached length then exceeds
    the window by less than a page, and never goes negative).  The first P entries of the
    row are rotated left by d, so the dropped blocks become the next pages to be written, and
    the cached length becomes n - d * block_size.  Otherwise the cached length becomes n.
    Entries past the first P are left alone.  Returns new (block_table, cache_seqlens).
    """
    bt = np.array(block_table, dtype=np.int32, copy=True)
    cs = np.array(cache_seqlens, dtype=np.int32, copy=True)
    for b in range(bt.shape[0]):
        n = int(cs[b]) + T
        P = -(-n // block_size)
        d = 0
        if n > window_frames:
            d = min(-(-(n - window_frames) // block_size), n // block_size)
        row = list(bt[b, :P])
        bt[b, :P] = row[d:] + row[:d]
        cs[b] = n - d * block_size
    return bt, cs


def project_qkv_pos(x, w_qkv, b_qkv, pos_emb, w_pos, H: int):
    """The projections that feed the path, in float64 (Model Layer page, fixed_attention_window
    row: one positional projection per step serves the cohort; the Conformer rel-pos attention's
    linear_q / linear_k / linear_v with bias and linear_pos without, WeNet's layout).

    x: [M, d_model] (M = B*T frames); w_qkv: [3*d_model, d_model] (q rows, then k, then v);
    b_qkv: [3*d_model]; pos_emb: [R, d_model]; w_pos: [d_model, d_model].
    Returns q, k, v: [M, H, d_model/H] and rel: [R, H, d_model/H].
    """
    x = np.asarray(x, dtype=np.float64)
    pos_emb = np.asarray(pos_emb, dtype=np.float64)
    w_qkv = np.asarray(w_qkv, dtype=np.float64)
    w_pos = np.asarray(w_pos, dtype=np.float64)
    b_qkv = np.asarray(b_qkv, dtype=np.float64)
    M, dm = x.shape
    if w_qkv.shape != (3 * dm, dm) or b_qkv.shape != (3 * dm,) or w_pos.shape != (dm, dm) \
            or pos_emb.ndim != 2 or pos_emb.shape[1] != dm or dm % H:
        raise ValueError("shapes: x [M,d], w_qkv [3d,d], b_qkv [3d], pos_emb [R,d], w_pos [d,d]")
    y = x @ w_qkv.T + b_qkv
    D = dm // H
    q, k, v = (y[:, i * dm:(i + 1) * dm].reshape(M, H, D) for i in range(3))
    rel = (pos_emb @ w_pos.T).reshape(pos_emb.shape[0], H, D)
    return q, k, v, rel
