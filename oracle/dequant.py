"""Float64 oracle for the W4A16-G128 weight dequantisation.

TEST INFRASTRUCTURE ONLY: imported by tests/ and the benchmark's CPU legs;
never by the product library.

What it restates (s1nh.org post on upgrading nano-vllm to big-vLLM, section
"add quantisation"): a quantised weight is stored as an int32 tensor in which
every int32 packs eight 4-bit values; dequantisation is int32 -> u4 unpack
-> s4 reconstruct -> float x weight_scale, with one scale per group of 128
weights ("G128").

Readings where the post is silent (each listed in the design notes):
  * value i of a word (i = 0..7) is bits 4i..4i+3: the lowest nibble first;
  * s4 = u4 - 8 (the unsigned nibble is an offset-binary signed value, giving
    the range -8..7);
  * weight W [N, K] (K, the input dimension, is the packed one): packed
    [N, K/8] int32, scales [N, K/128] bf16, group g of row n covering
    columns 128g .. 128g+127;
  * the result is bf16 (round to nearest even), the activations' type.

s4 * scale is exact in float64 (and in float32: at most 12 significant
bits), so rounding it once to bf16 is the whole answer and a kernel that
multiplies in fp32 and rounds once must match it bit for bit.
"""
from __future__ import annotations

import numpy as np

GROUP = 128  # weights per scale ("G128")


def unpack_u4(packed: np.ndarray) -> np.ndarray:
    """int32 words [..., W] -> unsigned nibbles [..., 8W], lowest nibble first."""
    words = np.asarray(packed).astype(np.int64) & 0xFFFFFFFF
    shifts = 4 * np.arange(8, dtype=np.int64)
    nib = (words[..., :, None] >> shifts) & 0xF          # [..., W, 8]
    return nib.reshape(*words.shape[:-1], words.shape[-1] * 8)


def s4_from_u4(u4: np.ndarray) -> np.ndarray:
    """Offset-binary reconstruction: u4 in 0..15 -> s4 in -8..7."""
    return np.asarray(u4, dtype=np.int64) - 8


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite float64 values to bf16, nearest-even, returning bit patterns.

    Done on the exact binary value: keep the top 8 significand bits of the
    float32 image and round the dropped 16 bits half-to-even.  (Used only on
    values that float32 holds exactly.)"""
    f = np.asarray(x, dtype=np.float64)
    f32 = f.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), f), "value not exact in float32"
    u = f32.view(np.uint32).astype(np.uint64)
    hi = u >> 16
    lo = u & 0xFFFF
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 1))
    return (hi + up.astype(np.uint64)).astype(np.uint16)


def w4a16_dequant(packed: np.ndarray, scales_bits: np.ndarray, group: int = GROUP) -> np.ndarray:
    """Dequantised weights as exact float64: W[n, k] = s4[n, k] * scale[n, k // group].

    packed [N, K/8] int32; scales_bits [N, K/group] bf16 bit patterns."""
    s4 = s4_from_u4(unpack_u4(packed)).astype(np.float64)        # [N, K]
    n, k = s4.shape
    scale = bf16_bits_to_f64(scales_bits)                        # [N, K/group]
    assert scale.shape == (n, k // group)
    return s4 * np.repeat(scale, group, axis=1)


def w4a16_dequant_bf16(packed: np.ndarray, scales_bits: np.ndarray, group: int = GROUP) -> np.ndarray:
    """The same, rounded once to bf16 (uint16 bit patterns [N, K])."""
    return f64_to_bf16_bits(w4a16_dequant(packed, scales_bits, group))
