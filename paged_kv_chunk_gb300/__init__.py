"""Paged-KV chunk attention with a shared Transformer-XL relative-position term, for
GB300 (sm_103a).

The compute lives in ``liboasr_attn.so`` (C ABI: ``include/oasr_attn.h``), built from
``csrc/`` by ``paged_kv_chunk_gb300.build``.  ``paged_kv_chunk_gb300.capi`` binds it for
torch CUDA tensors; ``paged_kv_chunk_gb300.synthetic`` draws the seeded workloads.
Importing this package loads nothing; the library is loaded on first use and a missing
build raises.
"""
from .capi import (OasrError, oasr_chunk_relattn_paged, oasr_chunk_step_paged,  # noqa: F401
                   oasr_device_status, oasr_packed_relattn_chunked, oasr_packed_relattn_varlen,
                   oasr_paged_append, oasr_project_qkv_pos, oasr_selftest_wait, oasr_version,
                   oasr_window_commit)

__all__ = ["OasrError", "oasr_paged_append", "oasr_chunk_relattn_paged", "oasr_chunk_step_paged",
           "oasr_packed_relattn_varlen", "oasr_packed_relattn_chunked", "oasr_window_commit",
           "oasr_project_qkv_pos", "oasr_device_status", "oasr_selftest_wait", "oasr_version"]
