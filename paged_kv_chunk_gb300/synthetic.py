"""Seeded synthetic inputs for the chunk attention workloads.

This module only draws random numbers and lays them out: it holds none of the
attention arithmetic, and both the CUDA path (tests, benchmark) and the CPU oracle
consume what it returns.  It imports nothing else from this package.

Value recipe: every float tensor (q, chunk K/V, cached K/V, pos_bias_u/v and the
rel-pos table) is drawn as N(0, 1) / 8 in float32 with numpy's PCG64 generator and,
for bf16 workloads, rounded to bf16 (round-to-nearest-even) by torch; the arrays
returned are float32 holding exactly those stored values.  Block tables are a
seeded permutation of the pool's block ids, so a stream's pages are scattered
across the pool.  Packed segment lengths are integers drawn uniformly from a range.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

SIGMA = 1.0 / 8.0


@dataclasses.dataclass(frozen=True)
class StreamingConfig:
    """One lockstep cohort: B streams, all with cache length C, appending T frames."""
    name: str
    B: int
    H: int
    D: int
    T: int
    C: int
    block_size: int
    dtype: str                  # "bf16" or "f32"
    seed: int
    num_blocks: int | None = None          # default: twice the demand
    max_blocks_per_seq: int | None = None  # default: pages needed for C + T keys
    window: int = 0                        # > 0: trained window (frames); steps commit with eviction
    hetero: bool = False                   # per-stream cache lengths U{0..C} (cache_lengths)

    @property
    def K(self) -> int:
        return self.C + self.T

    @property
    def R(self) -> int:
        return self.C + 2 * self.T - 1

    @property
    def pages_per_seq(self) -> int:
        return -(-self.K // self.block_size)

    @property
    def mbps(self) -> int:
        return self.max_blocks_per_seq or self.pages_per_seq

    @property
    def pool_blocks(self) -> int:
        return self.num_blocks or 2 * self.B * self.pages_per_seq


@dataclasses.dataclass(frozen=True)
class PackedConfig:
    """Offline packed row: num_seqs utterances of lengths U{min_len..max_len}."""
    name: str
    num_seqs: int
    min_len: int
    max_len: int
    H: int
    D: int
    dtype: str
    seed: int

    @property
    def R(self) -> int:
        return 2 * self.max_len - 1


# The five workloads: a tiny fp32 cohort, the Conformer-small and Conformer-large
# streaming cohorts, the chunk-size sweep, and the offline packed row.
TINY = StreamingConfig("tiny", B=2, H=4, D=64, T=16, C=64, block_size=16, dtype="f32",
                       seed=1000, num_blocks=16, max_blocks_per_seq=8)
SMALL = StreamingConfig("conformer_small", B=64, H=4, D=64, T=16, C=256, block_size=16,
                        dtype="bf16", seed=1001)
LARGE = StreamingConfig("conformer_large", B=256, H=8, D=64, T=16, C=512, block_size=32,
                        dtype="bf16", seed=1002)
SWEEP = tuple(StreamingConfig(f"sweep_T{T}", B=128, H=8, D=64, T=T, C=16 * T, block_size=16,
                              dtype="bf16", seed=1003 + T) for T in (4, 8, 16, 32, 64))
PACKED = PackedConfig("packed_varlen", num_seqs=256, min_len=50, max_len=1500, H=8, D=64,
                      dtype="bf16", seed=1004)

# A trained-window cohort paged by chunk (the pages' Nemotron sizing: 32 streams, 5 pages of
# one 16-frame chunk each, i.e. a 64-frame window plus the chunk being appended); every step
# commits with eviction, so the cache length stays at the window.
WINDOW_RING = StreamingConfig("window_ring", B=32, H=8, D=64, T=16, C=64, block_size=16,
                              dtype="bf16", seed=1010, window=64)

# The Conformer-small cohort at heterogeneous offsets (streams that joined at different
# times, one launch): stream b's cache length is drawn from U{0..256}, one table for all.
HETERO = StreamingConfig("hetero_small", B=64, H=4, D=64, T=16, C=256, block_size=16,
                         dtype="bf16", seed=1011, hetero=True)

STREAMING_CONFIGS = {c.name: c for c in (TINY, SMALL, LARGE, WINDOW_RING, HETERO) + SWEEP}


def cache_lengths(cfg: StreamingConfig) -> np.ndarray:
    """int32 [B]: every stream's cache length (C, or U{0..C} per stream for a heterogeneous
    cohort, seeded by the config)."""
    if not cfg.hetero:
        return np.full((cfg.B,), cfg.C, np.int32)
    return np.random.default_rng(cfg.seed + 17).integers(0, cfg.C + 1, cfg.B).astype(np.int32)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the storage dtype and return them as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    raise ValueError(f"unknown dtype {dtype!r}")


def normal(rng: np.random.Generator, shape, dtype: str, sigma: float = SIGMA) -> np.ndarray:
    return round_to(rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma), dtype)


def quarters(rng: np.random.Generator, shape, amp: int = 4) -> np.ndarray:
    """Integers drawn uniformly from [-amp, amp], divided by 4, as float32.  With amp <= 4 the
    values, their sums with another such tensor and their products by powers of two up to 16
    are exact in bf16, and dot products of 64 of them are exact in fp32: inputs for which a
    score carries no rounding in any precision."""
    return (rng.integers(-amp, amp + 1, size=shape).astype(np.float32) / np.float32(4.0))


def block_table(rng: np.random.Generator, B: int, mbps: int, num_blocks: int) -> np.ndarray:
    """Each stream gets mbps distinct pool blocks from one seeded permutation."""
    if B * mbps > num_blocks:
        raise ValueError("pool too small for the block tables")
    perm = rng.permutation(num_blocks).astype(np.int32)
    return np.ascontiguousarray(perm[: B * mbps].reshape(B, mbps))


def streaming_inputs(cfg: StreamingConfig, seed: int | None = None, *, R: int | None = None):
    """All inputs of one streaming step, as float32 (dtype-exact) numpy arrays.

    Returns a dict with q, k_new, v_new [B,T,H,D]; cache_k, cache_v [B,C,H,D]
    (the history, un-paged); pos_bias_u, pos_bias_v [H,D]; rel [R,H,D];
    block_table int32 [B, mbps]; cache_seqlens int32 [B] (all C); num_blocks.
    """
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    B, H, D, T, C = cfg.B, cfg.H, cfg.D, cfg.T, cfg.C
    R = cfg.R if R is None else R
    out = {
        "q": normal(rng, (B, T, H, D), cfg.dtype),
        "k_new": normal(rng, (B, T, H, D), cfg.dtype),
        "v_new": normal(rng, (B, T, H, D), cfg.dtype),
        "cache_k": normal(rng, (B, C, H, D), cfg.dtype),
        "cache_v": normal(rng, (B, C, H, D), cfg.dtype),
        "pos_bias_u": normal(rng, (H, D), cfg.dtype),
        "pos_bias_v": normal(rng, (H, D), cfg.dtype),
        "rel": normal(rng, (R, H, D), cfg.dtype),
    }
    out["block_table"] = block_table(rng, B, cfg.mbps, cfg.pool_blocks)
    out["cache_seqlens"] = np.full((B,), C, dtype=np.int32)
    out["num_blocks"] = cfg.pool_blocks
    return out


def packed_lengths(cfg: PackedConfig, rng: np.random.Generator) -> np.ndarray:
    return rng.integers(cfg.min_len, cfg.max_len + 1, size=cfg.num_seqs).astype(np.int32)


def packed_inputs(cfg: PackedConfig, seed: int | None = None, lengths=None):
    """All inputs of one packed offline call.

    Returns q, k, v [total,H,D]; cu_seqlens int32 [num_seqs+1]; lengths;
    pos_bias_u, pos_bias_v [H,D]; rel [2*max_len-1, H, D]; max_seqlen.
    """
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    lengths = packed_lengths(cfg, rng) if lengths is None else np.asarray(lengths, np.int32)
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    total = int(cu[-1])
    H, D = cfg.H, cfg.D
    R = 2 * max(cfg.max_len, int(lengths.max()) if len(lengths) else 1) - 1
    return {
        "q": normal(rng, (total, H, D), cfg.dtype),
        "k": normal(rng, (total, H, D), cfg.dtype),
        "v": normal(rng, (total, H, D), cfg.dtype),
        "cu_seqlens": cu,
        "lengths": lengths,
        "pos_bias_u": normal(rng, (H, D), cfg.dtype),
        "pos_bias_v": normal(rng, (H, D), cfg.dtype),
        "rel": normal(rng, (R, H, D), cfg.dtype),
        "max_seqlen": int(lengths.max()) if len(lengths) else 0,
    }


def canary_pool(num_blocks: int, block_size: int, H: int, D: int, dtype: str) -> np.ndarray:
    """A pool whose every element is a quiet NaN (stray reads poison results,
    untouched slots stay recognisable).  bf16 pools are returned as uint16 bits."""
    if dtype == "bf16":
        return np.full((num_blocks, block_size, H, D), 0x7FC1, dtype=np.uint16)
    return np.full((num_blocks, block_size, H, D), np.nan, dtype=np.float32)


def random_pool(rng: np.random.Generator, num_blocks: int, block_size: int, H: int, D: int,
                dtype: str) -> np.ndarray:
    """A pool filled with N(0,1)/8 values (used where only timing matters)."""
    return normal(rng, (num_blocks, block_size, H, D), dtype)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """float32 (dtype-exact) array -> raw storage array (uint16 bf16 bits, or float32)."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def from_bits(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Raw storage array -> float32 values."""
    if dtype == "f32":
        return np.asarray(bits, dtype=np.float32)
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)

