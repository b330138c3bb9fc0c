"""Shared test helpers: build inputs, run the oracle, compare against it.

Tolerances (written here once, used by every parity test):
  * fp32 path: max |gpu - oracle| <= 1e-5.
  * bf16 path: max |gpu - oracle| <= 2e-2 (the stated bar) and, because outputs of
    N(0,1)/8 inputs are only ~1e-2 in scale, a tighter internal gate of
    max abs <= 4e-3 and rms(gpu - oracle) / rms(oracle) <= 1e-2, which an indexing
    mistake (a wrong rel row, a dropped page) would fail.
  * paged append: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_chunk_gb300 import synthetic as syn

TOL_F32 = 1e-5
TOL_BF16 = 2e-2
TOL_BF16_INTERNAL = 4e-3
TOL_BF16_RMS_REL = 1e-2


def dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    """float32 numpy (dtype-exact) -> CUDA tensor of the storage dtype."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == "bf16":
        t = t.to(torch.bfloat16)
    return t.cuda()


def dev_pool(pool: np.ndarray, dtype: str) -> torch.Tensor:
    """Raw pool (uint16 bf16 bits, or float32) -> CUDA tensor."""
    if dtype == "bf16":
        return torch.from_numpy(pool.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(pool).cuda()


def host_pool(t: torch.Tensor, dtype: str) -> np.ndarray:
    """CUDA pool -> raw numpy (uint16 bits or float32)."""
    t = t.cpu()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def stream_case(cfg: syn.StreamingConfig, seed=None, R=None, block_table=None):
    """Inputs of one step plus pools holding the history (written by the oracle's
    append of the whole cache at cache_seqlens = 0); untouched slots keep canaries."""
    x = syn.streaming_inputs(cfg, seed, R=R)
    if block_table is not None:
        x["block_table"] = np.ascontiguousarray(block_table, dtype=np.int32)
    kp = syn.canary_pool(x["num_blocks"], cfg.block_size, cfg.H, cfg.D, cfg.dtype)
    vp = syn.canary_pool(x["num_blocks"], cfg.block_size, cfg.H, cfg.D, cfg.dtype)
    if cfg.C > 0:
        zeros = np.zeros((cfg.B,), np.int32)
        ck = syn.to_bits(x["cache_k"], cfg.dtype)
        cv = syn.to_bits(x["cache_v"], cfg.dtype)
        assert oracle.paged_append(ck, cv, kp, vp, x["block_table"], zeros) == 0
    x["k_pool"], x["v_pool"] = kp, vp
    return x


def oracle_chunk(x, rows=None, scale=None):
    return oracle.chunk_relattn(x["q"], x["cache_k"], x["cache_v"], x["k_new"], x["v_new"],
                                x["pos_bias_u"], x["pos_bias_v"], x["rel"], scale=scale,
                                rows=rows)


def check_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    """Assert the parity gates; returns (max_abs, rms_rel) for reporting."""
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    rms_ref = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 1.0
    rms_rel = float(np.sqrt(np.mean(err ** 2)) / max(rms_ref, 1e-30)) if err.size else 0.0
    if dtype == "f32":
        assert max_abs <= TOL_F32, f"{what}: max abs err {max_abs:.3e} > {TOL_F32}"
    else:
        assert max_abs <= TOL_BF16, f"{what}: max abs err {max_abs:.3e} > {TOL_BF16}"
        assert max_abs <= TOL_BF16_INTERNAL, f"{what}: max abs err {max_abs:.3e} > internal gate"
        assert rms_rel <= TOL_BF16_RMS_REL, f"{what}: rms-relative err {rms_rel:.3e}"
    return max_abs, rms_rel


def gpu_stream_inputs(x, dtype):
    """Device tensors for one streaming step."""
    d = {k: dev(x[k], dtype) for k in ("q", "k_new", "v_new", "pos_bias_u", "pos_bias_v", "rel")}
    d["k_pool"] = dev_pool(x["k_pool"], dtype)
    d["v_pool"] = dev_pool(x["v_pool"], dtype)
    d["block_table"] = torch.from_numpy(x["block_table"]).cuda()
    d["cache_seqlens"] = torch.from_numpy(x["cache_seqlens"]).cuda()
    return d


def sample_rows(rng, B, T, H, n):
    """n distinct (b, i, h) triples."""
    n = min(n, B * T * H)
    flat = rng.choice(B * T * H, size=n, replace=False)
    h = flat % H
    i = (flat // H) % T
    b = flat // (H * T)
    return np.stack([b, i, h], axis=1).astype(np.int32)
