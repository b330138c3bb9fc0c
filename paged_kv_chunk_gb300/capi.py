"""Python binding of the C ABI in ``include/oasr_attn.h`` (``liboasr_attn.so``).

Argument marshalling only: each function checks that the torch tensors it is given
live on the current CUDA device with the layout the C ABI documents, derives the
sizes from their shapes and passes raw device pointers plus the current CUDA stream.
Every step of the computation runs in the library's CUDA kernels; there is no other
path, and a missing library raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import functools
import os
import re
import threading

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "liboasr_attn.so")
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "oasr_attn.h")

OASR_OK, OASR_ERR_INVALID_ARG, OASR_ERR_UNSUPPORTED, OASR_ERR_CUDA = 0, 1, 2, 3
OASR_ERR_BOUNDS, OASR_ERR_TIMEOUT = 4, 5
OASR_F32, OASR_BF16 = 0, 1
STATUS_BOUNDS_BIT, STATUS_TIMEOUT_BIT = 1, 2

_lock = threading.Lock()
_lib = None


class OasrError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


def load() -> ctypes.CDLL:
    """Load liboasr_attn.so (built by ``paged_kv_chunk_gb300.build``); raise if absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -m paged_kv_chunk_gb300.build`"
                               " (or __graft_entry__.build()) first")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        L.oasr_paged_append.argtypes = [P, P, P, P, I, I, P, I, P, I, I, I, I, I, S]
        L.oasr_chunk_relattn_paged.argtypes = [P, P, P, I, I, P, I, P, P, P, P, I, P, I, I, I, I,
                                               F, I, S]
        L.oasr_chunk_step_paged.argtypes = [P, P, P, P, P, I, I, P, I, P, P, P, P, I, P, I, I, I,
                                            I, F, I, S]
        L.oasr_packed_relattn_varlen.argtypes = [P, P, P, P, I, I, I, P, P, P, I, P, I, I, F, I, S]
        L.oasr_packed_relattn_chunked.argtypes = [P, P, P, P, I, I, I, P, P, P, I, P, I, I, F, I, I,
                                                  I, S]
        L.oasr_window_commit.argtypes = [P, P, I, I, I, I, I, S]
        L.oasr_project_qkv_pos.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, S]
        for fn in ("oasr_paged_append", "oasr_chunk_relattn_paged", "oasr_chunk_step_paged",
                   "oasr_packed_relattn_varlen", "oasr_packed_relattn_chunked",
                   "oasr_window_commit", "oasr_project_qkv_pos"):
            getattr(L, fn).restype = I
        L.oasr_status_string.argtypes = [I]
        L.oasr_status_string.restype = ctypes.c_char_p
        L.oasr_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), I]
        L.oasr_device_status.restype = I
        L.oasr_version.argtypes = []
        L.oasr_version.restype = I
        L.oasr_selftest_wait.argtypes = [ctypes.c_uint, S]
        L.oasr_selftest_wait.restype = I
        _lib = L
        return L


def header_symbols() -> list[str]:
    """Names of the functions ``include/oasr_attn.h`` declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oasr_[a-z0-9_]+)\s*\(", text)))


def _check(fn: str, status: int):
    if status != OASR_OK:
        msg = load().oasr_status_string(status).decode()
        raise OasrError(fn, status, msg)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return OASR_BF16
    if t.dtype == torch.float32:
        return OASR_F32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or float32")


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        # the kernels run on the current device: another device's pointer would be a fault
        raise ValueError(f"{name} is on {t.device}, the current device is "
                         f"cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def oasr_paged_append(k_new, v_new, k_pool, v_pool, block_table, cache_seqlens, stream=None):
    """Write the chunk (k_new, v_new [B,T,H,D]) into the pools [nb,bs,H,D] in place."""
    L = load()
    dt = _dtype_code(k_new)
    B, T, H, D = k_new.shape
    nb, bs = k_pool.shape[:2]
    if tuple(v_new.shape) != (B, T, H, D) or tuple(k_pool.shape[2:]) != (H, D) \
            or v_pool.shape != k_pool.shape:
        raise ValueError("shape mismatch between chunk and pools")
    if tuple(block_table.shape[:1]) != (B,) or tuple(cache_seqlens.shape) != (B,):
        raise ValueError("block_table must be [B, mbps] and cache_seqlens [B]")
    _check("oasr_paged_append", L.oasr_paged_append(
        _dev(k_new, "k_new", k_new.dtype, 4), _dev(v_new, "v_new", k_new.dtype, 4),
        _dev(k_pool, "k_pool", k_new.dtype, 4), _dev(v_pool, "v_pool", k_new.dtype, 4), nb, bs,
        _dev(block_table, "block_table", torch.int32, 2), block_table.shape[1],
        _dev(cache_seqlens, "cache_seqlens", torch.int32, 1), B, T, H, D, dt, _stream(stream)))


def _chunk_common(q, k_pool, v_pool, block_table, cache_seqlens, pos_bias_u, pos_bias_v, rel,
                  out):
    B, T, H, D = q.shape
    if k_pool.dim() != 4 or tuple(k_pool.shape[2:]) != (H, D):
        raise ValueError("k_pool must be [num_blocks, block_size, H, D]")
    if v_pool.shape != k_pool.shape:
        raise ValueError("v_pool must have k_pool's shape")
    if tuple(pos_bias_u.shape) != (H, D) or tuple(pos_bias_v.shape) != (H, D):
        raise ValueError("pos biases must be [H, D]")
    if rel.dim() != 3 or tuple(rel.shape[1:]) != (H, D):
        raise ValueError("rel must be [R, H, D]")
    if tuple(out.shape) != (B, T, H, D) or out.dtype != q.dtype:
        raise ValueError("out must be [B, T, H, D] of q's dtype")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(cache_seqlens.shape) != (B,):
        raise ValueError("block_table must be [B, mbps] and cache_seqlens [B]")
    return B, T, H, D


def oasr_chunk_relattn_paged(q, k_pool, v_pool, block_table, cache_seqlens, pos_bias_u,
                             pos_bias_v, rel, out=None, scale=None, stream=None):
    """Streaming chunk attention over the paged pool; returns out [B,T,H,D]."""
    L = load()
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    B, T, H, D = _chunk_common(q, k_pool, v_pool, block_table, cache_seqlens, pos_bias_u,
                               pos_bias_v, rel, out)
    scale = D ** -0.5 if scale is None else float(scale)
    _check("oasr_chunk_relattn_paged", L.oasr_chunk_relattn_paged(
        _dev(q, "q", q.dtype), _dev(k_pool, "k_pool", q.dtype), _dev(v_pool, "v_pool", q.dtype),
        k_pool.shape[0], k_pool.shape[1], _dev(block_table, "block_table", torch.int32),
        block_table.shape[1], _dev(cache_seqlens, "cache_seqlens", torch.int32),
        _dev(pos_bias_u, "pos_bias_u", q.dtype), _dev(pos_bias_v, "pos_bias_v", q.dtype),
        _dev(rel, "rel", q.dtype), rel.shape[0], _dev(out, "out", q.dtype), B, T, H, D, scale, dt,
        _stream(stream)))
    return out


def oasr_chunk_step_paged(q, k_new, v_new, k_pool, v_pool, block_table, cache_seqlens,
                          pos_bias_u, pos_bias_v, rel, out=None, scale=None, stream=None):
    """Fused append + streaming chunk attention; returns out [B,T,H,D]."""
    L = load()
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    B, T, H, D = _chunk_common(q, k_pool, v_pool, block_table, cache_seqlens, pos_bias_u,
                               pos_bias_v, rel, out)
    if tuple(k_new.shape) != (B, T, H, D) or tuple(v_new.shape) != (B, T, H, D):
        raise ValueError("k_new, v_new must be [B, T, H, D]")
    scale = D ** -0.5 if scale is None else float(scale)
    _check("oasr_chunk_step_paged", L.oasr_chunk_step_paged(
        _dev(q, "q", q.dtype), _dev(k_new, "k_new", q.dtype), _dev(v_new, "v_new", q.dtype),
        _dev(k_pool, "k_pool", q.dtype), _dev(v_pool, "v_pool", q.dtype), k_pool.shape[0],
        k_pool.shape[1], _dev(block_table, "block_table", torch.int32), block_table.shape[1],
        _dev(cache_seqlens, "cache_seqlens", torch.int32), _dev(pos_bias_u, "pos_bias_u", q.dtype),
        _dev(pos_bias_v, "pos_bias_v", q.dtype), _dev(rel, "rel", q.dtype), rel.shape[0],
        _dev(out, "out", q.dtype), B, T, H, D, scale, dt, _stream(stream)))
    return out


def oasr_packed_relattn_varlen(q, k, v, cu_seqlens, max_seqlen, pos_bias_u, pos_bias_v, rel,
                               out=None, scale=None, stream=None):
    """Packed varlen bidirectional rel-pos attention; returns out [total,H,D]."""
    L = load()
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    total, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or out.shape != q.shape:
        raise ValueError("q, k, v, out must share their shape [total, H, D]")
    if tuple(pos_bias_u.shape) != (H, D) or tuple(pos_bias_v.shape) != (H, D):
        raise ValueError("pos biases must be [H, D]")
    if rel.dim() != 3 or tuple(rel.shape[1:]) != (H, D):
        raise ValueError("rel must be [R, H, D]")
    scale = D ** -0.5 if scale is None else float(scale)
    _check("oasr_packed_relattn_varlen", L.oasr_packed_relattn_varlen(
        _dev(q, "q", q.dtype), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype),
        _dev(cu_seqlens, "cu_seqlens", torch.int32, 1), cu_seqlens.shape[0] - 1, int(max_seqlen),
        total, _dev(pos_bias_u, "pos_bias_u", q.dtype), _dev(pos_bias_v, "pos_bias_v", q.dtype),
        _dev(rel, "rel", q.dtype), rel.shape[0], _dev(out, "out", q.dtype), H, D, scale, dt,
        _stream(stream)))
    return out


def oasr_packed_relattn_chunked(q, k, v, cu_seqlens, max_seqlen, pos_bias_u, pos_bias_v, rel,
                                chunk_size, left_chunks, out=None, scale=None, stream=None):
    """Chunked-limited packed attention (own chunk + left_chunks earlier chunks per query);
    returns out [total,H,D]."""
    L = load()
    dt = _dtype_code(q)
    if out is None:
        out = torch.empty_like(q)
    total, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or out.shape != q.shape:
        raise ValueError("q, k, v, out must share their shape [total, H, D]")
    if tuple(pos_bias_u.shape) != (H, D) or tuple(pos_bias_v.shape) != (H, D):
        raise ValueError("pos biases must be [H, D]")
    if rel.dim() != 3 or tuple(rel.shape[1:]) != (H, D):
        raise ValueError("rel must be [R, H, D]")
    scale = D ** -0.5 if scale is None else float(scale)
    _check("oasr_packed_relattn_chunked", L.oasr_packed_relattn_chunked(
        _dev(q, "q", q.dtype), _dev(k, "k", q.dtype), _dev(v, "v", q.dtype),
        _dev(cu_seqlens, "cu_seqlens", torch.int32, 1), cu_seqlens.shape[0] - 1, int(max_seqlen),
        total, _dev(pos_bias_u, "pos_bias_u", q.dtype), _dev(pos_bias_v, "pos_bias_v", q.dtype),
        _dev(rel, "rel", q.dtype), rel.shape[0], _dev(out, "out", q.dtype), H, D, scale,
        int(chunk_size), int(left_chunks), dt, _stream(stream)))
    return out


def oasr_window_commit(block_table, cache_seqlens, T, block_size, window_frames, stream=None):
    """Commit a step's chunk with fixed-window history eviction, in place on the device:
    rotates each full stream's block-table row and advances cache_seqlens."""
    L = load()
    if block_table.dim() != 2 or cache_seqlens.dim() != 1 or cache_seqlens.shape[0] != block_table.shape[0]:
        raise ValueError("block_table must be [B, max_blocks_per_seq] and cache_seqlens [B]")
    B, mbps = block_table.shape
    _check("oasr_window_commit", L.oasr_window_commit(
        _dev(block_table, "block_table", torch.int32, 2), _dev(cache_seqlens, "cache_seqlens", torch.int32, 1),
        B, mbps, int(block_size), int(T), int(window_frames), _stream(stream)))


def oasr_project_qkv_pos(x, w_qkv, b_qkv, pos_emb, w_pos, H, q=None, k=None, v=None, rel=None,
                         stream=None):
    """q, k, v = x . w_qkv^T + b_qkv (split in three, [M, H, 64] each) and
    rel = pos_emb . w_pos^T ([R, H, 64]), bf16, one launch; returns (q, k, v, rel)."""
    L = load()
    M, d = x.shape
    R = pos_emb.shape[0]
    if tuple(w_qkv.shape) != (3 * d, d) or tuple(b_qkv.shape) != (3 * d,) or \
            tuple(w_pos.shape) != (d, d) or pos_emb.dim() != 2 or pos_emb.shape[1] != d or d % H:
        raise ValueError("shapes: x [M,d], w_qkv [3d,d], b_qkv [3d], pos_emb [R,d], w_pos [d,d]")
    D = d // H
    q = torch.empty((M, H, D), dtype=x.dtype, device=x.device) if q is None else q
    k = torch.empty((M, H, D), dtype=x.dtype, device=x.device) if k is None else k
    v = torch.empty((M, H, D), dtype=x.dtype, device=x.device) if v is None else v
    rel = torch.empty((R, H, D), dtype=x.dtype, device=x.device) if rel is None else rel
    if any(tuple(t.shape) != (M, H, D) for t in (q, k, v)) or tuple(rel.shape) != (R, H, D):
        raise ValueError("q, k, v must be [M, H, d/H] and rel [R, H, d/H]")
    _check("oasr_project_qkv_pos", L.oasr_project_qkv_pos(
        _dev(x, "x", x.dtype, 2), _dev(w_qkv, "w_qkv", x.dtype, 2), _dev(b_qkv, "b_qkv", x.dtype, 1),
        _dev(pos_emb, "pos_emb", x.dtype, 2), _dev(w_pos, "w_pos", x.dtype, 2),
        _dev(q, "q", x.dtype), _dev(k, "k", x.dtype), _dev(v, "v", x.dtype), _dev(rel, "rel", x.dtype),
        M, R, d, H, _dtype_code(x), _stream(stream)))
    return q, k, v, rel


def oasr_device_status(clear: bool = True) -> int:
    """Raw device status bits (1 = an index was out of range, 2 = a wait timed out)."""
    L = load()
    flags = ctypes.c_uint(0)
    _check("oasr_device_status", L.oasr_device_status(ctypes.byref(flags), int(clear)))
    return int(flags.value)


def oasr_version() -> int:
    return int(load().oasr_version())


def oasr_selftest_wait(limit_us: int = 20000, stream=None) -> None:
    """Diagnostic: the library's bounded wait on a barrier that nothing signals.  It runs
    out after ``limit_us`` microseconds and raises the timeout bit (2) of the device status
    word, as any of the library's kernels does when a copy it waits for never lands."""
    _check("oasr_selftest_wait", load().oasr_selftest_wait(int(limit_us), _stream(stream)))


# NVTX ranges around every call into the library, for Nsight timelines: set OASR_NVTX=1
# before the import.
NVTX = os.environ.get("OASR_NVTX", "") == "1"


def _traced(fn):
    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        torch.cuda.nvtx.range_push(fn.__name__)
        try:
            return fn(*args, **kwargs)
        finally:
            torch.cuda.nvtx.range_pop()
    return wrapper


if NVTX:
    for _name in ("oasr_paged_append", "oasr_chunk_relattn_paged", "oasr_chunk_step_paged",
                  "oasr_packed_relattn_varlen", "oasr_packed_relattn_chunked", "oasr_window_commit",
                  "oasr_project_qkv_pos", "oasr_selftest_wait"):
        globals()[_name] = _traced(globals()[_name])
