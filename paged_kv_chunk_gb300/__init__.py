"""Paged-KV chunk attention with a shared Transformer-XL relative-position term, for
GB300 (sm_103a).

The compute lives in ``liboasr_attn.so`` (C ABI: ``include/oasr_attn.h``), built from
``csrc/`` by ``paged_kv_chunk_gb300.build``.  ``paged_kv_chunk_gb300.capi`` binds it for
torch CUDA tensors; ``paged_kv_chunk_gb300.synthetic`` draws the seeded workloads.
Importing this package loads nothing; the library is loaded on first use and a missing
build raises.

One streaming encoder step of a cohort, per attention layer (all tensors on the current
CUDA device; the layer's pools, the shared block table and cache lengths persist)::

    from paged_kv_chunk_gb300 import capi
    q, k_new, v_new, rel = capi.oasr_project_qkv_pos(x, w_qkv, b_qkv, pos_emb, w_pos, H)
    out = capi.oasr_chunk_step_paged(q.view(B, T, H, 64), k_new.view(B, T, H, 64),
                                     v_new.view(B, T, H, 64), k_pool, v_pool,
                                     block_table, cache_seqlens, pos_bias_u, pos_bias_v, rel)
    # after the step's last layer: advance the cache lengths (cache_seqlens += T), or with
    # a trained window commit with eviction:
    capi.oasr_window_commit(block_table, cache_seqlens, T, block_size, window_frames)

The offline pass over packed utterances is ``oasr_packed_relattn_varlen`` (or
``oasr_packed_relattn_chunked`` under the Nemotron chunked-limited window).
"""
from .capi import (OasrError, oasr_chunk_relattn_paged, oasr_chunk_step_paged,  # noqa: F401
                   oasr_device_status, oasr_packed_relattn_chunked, oasr_packed_relattn_varlen,
                   oasr_paged_append, oasr_project_qkv_pos, oasr_selftest_wait, oasr_version,
                   oasr_window_commit)

__all__ = ["OasrError", "oasr_paged_append", "oasr_chunk_relattn_paged", "oasr_chunk_step_paged",
           "oasr_packed_relattn_varlen", "oasr_packed_relattn_chunked", "oasr_window_commit",
           "oasr_project_qkv_pos", "oasr_device_status", "oasr_selftest_wait", "oasr_version"]
