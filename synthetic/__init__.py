"""Seeded synthetic workloads for the OSCAR INT2 paged KV-cache path.

This module only draws random numbers and formats them (shapes, BF16 storage
rounding of inputs, ragged lengths, page permutations).  It holds none of the
method's arithmetic: no rotation, covariance, clipping, quantisation, packing
or attention.  Both the CPU oracle and the CUDA path take their inputs from
here, so neither has to import the other.

Distribution (a stand-in for the Qwen3-shaped activations the OSCAR pages
evaluate on; the real models and datasets are not available):

* every channel c of K, V and q is N(0, sigma_c^2) with
  sigma_c ~ LogNormal(0, 0.5), drawn per (layer, head, channel);
* two outlier channels per head, chosen at random, have sigma multiplied by 20;
* workload values use ``seed``; calibration samples use ``seed + 1000`` with
  the same per-channel sigmas.

Every stream is ``numpy.random.default_rng([seed, layer, stream])`` so that a
layer or a tensor can be regenerated on its own.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

# stream ids for default_rng([seed, layer, stream])
_S_SIG_K, _S_SIG_V, _S_SIG_Q = 1, 2, 3
_S_K, _S_V, _S_Q = 11, 12, 13
_S_KNEW, _S_VNEW, _S_QSTEP = 21, 22, 23
_S_LENS, _S_PAGES = 31, 32

CALIB_SEED_OFFSET = 1000
OUTLIER_CHANNELS = 2
OUTLIER_FACTOR = 20.0
LOGNORMAL_SIGMA = 0.5


@dataclass(frozen=True)
class Shape:
    """Attention-layer and cache shape of one workload."""

    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    group_size: int = 32
    sink: int = 4
    recent: int = 128
    num_layers: int = 1


@dataclass
class Workload:
    """A named synthetic workload: a shape plus per-request lengths."""

    name: str
    shape: Shape
    seq_lens: List[int]
    seed: int
    dtype: str = "bf16"  # storage type of K, V, q inputs: "bf16" or "f32"
    notes: str = ""
    extra: dict = field(default_factory=dict)


# --------------------------------------------------------------------------
# the workloads (sizes of the OSCAR pages' Qwen3-shaped attention layers)
# --------------------------------------------------------------------------
def tiny() -> Workload:
    """1 layer, batch 1, 4 q / 2 kv heads, d=64, n=512 = 4 sink + 32 recent + 476 INT2, P=16, fp32 inputs."""
    return Workload("tiny", Shape(4, 2, 64, 16, 32, 4, 32, 1), [512], seed=0, dtype="f32")


def batch1_32k(num_layers: int = 1) -> Workload:
    """Qwen3-8B-shaped layer: 32 q / 8 kv heads, d=128, n=32768 = 4 + 128 + 32636 INT2, P=64."""
    return Workload("batch1_32k", Shape(32, 8, 128, 64, 32, 4, 128, num_layers), [32768], seed=1)


def batched_ragged(batch: int, num_layers: int = 1) -> Workload:
    """Qwen3-32B-shaped layer: 64 q / 8 kv heads, d=128, ragged n ~ U[8K, 32K], P=64, shuffled pages."""
    rng = np.random.default_rng([2, 0, _S_LENS, batch])
    lens = [int(x) for x in rng.integers(8192, 32769, size=batch)]
    return Workload(f"batched_ragged_b{batch}", Shape(64, 8, 128, 64, 32, 4, 128, num_layers), lens, seed=2)


def long_131k() -> Workload:
    """Batch 1 at 131,072 tokens, 32 q / 8 kv heads, d=128, P=64."""
    return Workload("long_131k", Shape(32, 8, 128, 64, 32, 4, 128, 1), [131072], seed=3)


def capacity_28x100k(num_layers: int = 64) -> Workload:
    """28 requests x 100,000 tokens x 64 layers, 64 q / 8 kv heads, d=128, P=64."""
    return Workload("capacity_28x100k", Shape(64, 8, 128, 64, 32, 4, 128, num_layers), [100000] * 28, seed=4)


def write_prefill(batch: int = 8, n: int = 32768) -> Workload:
    """Write path: prefill batch x n tokens, 8 kv heads, d=128, P=64; then 256 appends; 4 requests share a 16K prefix."""
    return Workload(f"write_prefill_{batch}x{n}", Shape(8, 8, 128, 64, 32, 4, 128, 1), [n] * batch, seed=5,
                    extra={"appends": 256, "prefix_tokens": 16384, "prefix_sharers": 4})


# --------------------------------------------------------------------------
# generators
# --------------------------------------------------------------------------
def _rng(seed: int, layer: int, stream: int, *more: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(layer), int(stream), *[int(m) for m in more]])


def channel_sigmas(seed: int, layer: int, which: str, n_heads: int, d: int) -> np.ndarray:
    """Per-(head, channel) standard deviations, float64 [n_heads, d]."""
    stream = {"k": _S_SIG_K, "v": _S_SIG_V, "q": _S_SIG_Q}[which]
    rng = _rng(seed, layer, stream)
    sig = rng.lognormal(mean=0.0, sigma=LOGNORMAL_SIGMA, size=(n_heads, d))
    for h in range(n_heads):
        idx = rng.choice(d, size=OUTLIER_CHANNELS, replace=False)
        sig[h, idx] *= OUTLIER_FACTOR
    return sig


def draw(seed: int, layer: int, which: str, n_tokens: int, n_heads: int, d: int,
         stream_override: Optional[int] = None, sub: int = 0, calib: bool = False,
         scale: float = 1.0) -> np.ndarray:
    """Gaussian activations with the per-channel sigmas, float32 [n_tokens, n_heads, d]."""
    sig = channel_sigmas(seed, layer, which, n_heads, d).astype(np.float32)
    stream = stream_override if stream_override is not None else {"k": _S_K, "v": _S_V, "q": _S_Q}[which]
    vseed = seed + CALIB_SEED_OFFSET if calib else seed
    rng = _rng(vseed, layer, stream, sub)
    x = rng.standard_normal(size=(n_tokens, n_heads, d), dtype=np.float32)
    x *= sig[None, :, :] * np.float32(scale)
    return x


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest even), return the uint16 bit patterns.

    Input formatting only (activations arrive in BF16 storage); NaN is not expected.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def as_input(x: np.ndarray, dtype: str) -> np.ndarray:
    """The exact float32 values the path receives for storage type ``dtype``."""
    if dtype == "bf16":
        return bf16_bits_to_f32(to_bf16_bits(x))
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(dtype)


def kv_tokens(w: Workload, layer: int, n_tokens: int, sub: int = 0, calib: bool = False):
    """K and V inputs [n_tokens, Hkv, d] as float32 values (BF16-representable if dtype is bf16)."""
    s = w.shape
    k = draw(w.seed, layer, "k", n_tokens, s.n_kv_heads, s.head_dim, sub=sub, calib=calib)
    v = draw(w.seed, layer, "v", n_tokens, s.n_kv_heads, s.head_dim, sub=sub, calib=calib)
    return as_input(k, w.dtype), as_input(v, w.dtype)


def queries(w: Workload, layer: int, n_rows: int, sub: int = 0, calib: bool = False, scale: float = 1.0):
    """Queries [n_rows, Hq, d] as float32 values (BF16-representable if dtype is bf16)."""
    s = w.shape
    q = draw(w.seed, layer, "q", n_rows, s.n_q_heads, s.head_dim, sub=sub, calib=calib, scale=scale)
    return as_input(q, w.dtype)


def page_permutation(seed: int, num_pages: int, shuffle: bool = True) -> np.ndarray:
    """Order in which physical pages are handed out (shuffled: non-contiguous block tables)."""
    ids = np.arange(num_pages, dtype=np.int32)
    if shuffle:
        _rng(seed, 0, _S_PAGES).shuffle(ids)
    return ids


def pages_for(n_tokens: int, page_size: int) -> int:
    return (n_tokens + page_size - 1) // page_size
