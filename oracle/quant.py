"""Per-group asymmetric INT2 quantiser and packed code layouts, float64 (test infrastructure only).

The pages fix only "INT2" with four levels (gist.science summaries, section 1)
and that history is stored in INT2 after the fixed rotation and clipping
(section 2.2 B, "mixed-precision layout").  The quantiser details are fixed by
the workload definition: per token, per head, per group of 32 consecutive
channels of the rotated vector, asymmetric min/max, BF16 scale and zero.

Readings: zero z = bf16(min) (a float minimum, not an integer zero-point);
scale s = bf16((max - min) / 3); code = clamp(rne((y - z) / s), 0, 3) using the
BF16-rounded z and s; s = 0 gives all-zero codes; dequantised value z + code*s.
BF16 rounding here is round-to-nearest-even directly from float64.

Code layouts (ours; the pages give none).  A token's codes for one head fill a
row of d/4 bytes, read as little-endian 32-bit words.  Both layouts are fixed
bijections channel -> 2-bit field:

K row (d/64 words per "lane" tig in 0..3):
    word index  = tig*(d/64) + w,  w in [0, d/64)
    slot x in 0..7 holds two channels: bits 2x  <- channel c,
                                       bits 16+2x <- channel c+1,
    with P = 8w + x, g = P>>2, kt = (P>>1)&1, h = P&1,
         c = 32g + 16kt + 8h + 2*tig.
V row (d/8 little-endian 16-bit half-words):
    half-word hw, slot s in 0..7 at bits 2s of that half-word holds channel
    64*(hw mod (d/64)) + 8s + hw div (d/64).
"""
from __future__ import annotations

import numpy as np

LEVELS = 4  # INT2


# ---------------------------------------------------------------- BF16
def bf16_round(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even), returned as float64.

    bfloat16 keeps 8 significant bits and float32's exponent range; its
    subnormal spacing is 2**-133.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    q_exp = np.maximum(e - 8, -133)
    return np.ldexp(np.rint(np.ldexp(x, -q_exp)), q_exp)


def bf16_to_bits(x_bf16_valued) -> np.ndarray:
    """uint16 bit pattern of values that are exactly representable in bfloat16."""
    f = np.asarray(x_bf16_valued, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bits_to_f64(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- quantiser
def quantize_groups(y, group: int):
    """Quantise the last axis of y (already clipped, float64) in groups of ``group`` channels.

    Returns (codes uint8 [..., d], scale [..., d/G], zero [..., d/G], mn, rng3)
    where scale and zero are BF16-valued float64 and mn / rng3 are the
    pre-rounding group minimum and (max - min)/3.
    """
    y = np.asarray(y, dtype=np.float64)
    d = y.shape[-1]
    yg = y.reshape(y.shape[:-1] + (d // group, group))
    mn = yg.min(axis=-1)
    mx = yg.max(axis=-1)
    rng3 = (mx - mn) / 3.0
    zero = bf16_round(mn)
    scale = bf16_round(rng3)
    codes = quantize_with(y, scale, zero, group)
    return codes, scale, zero, mn, rng3


def quantize_with(y, scale, zero, group: int) -> np.ndarray:
    """Codes of y for given (BF16-valued) per-group scale and zero: clamp(rne((y-z)/s), 0, 3)."""
    y = np.asarray(y, dtype=np.float64)
    d = y.shape[-1]
    yg = y.reshape(y.shape[:-1] + (d // group, group))
    s = np.asarray(scale, dtype=np.float64)[..., None]
    z = np.asarray(zero, dtype=np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (yg - z) / s
        c = np.clip(np.rint(t), 0, LEVELS - 1)
    c = np.where(s > 0, c, 0.0)
    return c.astype(np.uint8).reshape(y.shape)


def dequantize(codes, scale, zero, group: int) -> np.ndarray:
    """y_hat = z + code * s per group, float64."""
    c = np.asarray(codes, dtype=np.float64)
    d = c.shape[-1]
    cg = c.reshape(c.shape[:-1] + (d // group, group))
    out = np.asarray(zero, dtype=np.float64)[..., None] + cg * np.asarray(scale, dtype=np.float64)[..., None]
    return out.reshape(c.shape)


# ---------------------------------------------------------------- layouts
def k_bit_offsets(d: int) -> np.ndarray:
    """Bit offset (from the start of the K code row) of each channel's 2-bit code."""
    if d % 64:
        raise ValueError("head_dim must be a multiple of 64")
    wpl = d // 64
    off = np.full(d, -1, dtype=np.int64)
    for tig in range(4):
        for w in range(wpl):
            word = tig * wpl + w
            for x in range(8):
                p = 8 * w + x
                g, kt, h = p >> 2, (p >> 1) & 1, p & 1
                c = 32 * g + 16 * kt + 8 * h + 2 * tig
                off[c] = 32 * word + 2 * x
                off[c + 1] = 32 * word + 16 + 2 * x
    assert (off >= 0).all()
    return off


def v_bit_offsets(d: int) -> np.ndarray:
    """Bit offset (from the start of the V code row) of each channel's 2-bit code."""
    if d % 64:
        raise ValueError("head_dim must be a multiple of 64")
    per = d // 64
    off = np.full(d, -1, dtype=np.int64)
    for hw in range(d // 8):
        for s in range(8):
            c = 64 * (hw % per) + 8 * s + hw // per
            off[c] = 16 * hw + 2 * s
    assert (off >= 0).all()
    return off


def pack_rows(codes, bit_offsets) -> np.ndarray:
    """Pack codes [..., d] (values 0..3) into rows of d/4 bytes following ``bit_offsets``."""
    c = np.asarray(codes, dtype=np.uint8)
    d = c.shape[-1]
    out = np.zeros(c.shape[:-1] + (d // 4,), dtype=np.uint8)
    for j in range(d):
        o = int(bit_offsets[j])
        out[..., o >> 3] |= (c[..., j] & 3) << (o & 7)
    return out


def unpack_rows(rows, bit_offsets) -> np.ndarray:
    """Inverse of pack_rows: bytes [..., d/4] -> codes [..., d]."""
    r = np.asarray(rows, dtype=np.uint8)
    d = r.shape[-1] * 4
    out = np.zeros(r.shape[:-1] + (d,), dtype=np.uint8)
    for j in range(d):
        o = int(bit_offsets[j])
        out[..., j] = (r[..., o >> 3] >> (o & 7)) & 3
    return out
