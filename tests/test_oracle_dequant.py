"""Pins of the W4A16-G128 dequantisation oracle (CPU).

The post gives the pipeline (int32 -> u4 unpack -> s4 reconstruct -> x scale,
8 nibbles per int32, one scale per 128 weights) but no worked example; these
tests fix the oracle to hand-computed values under the stated readings
(lowest nibble first, s4 = u4 - 8) and to properties any correct
implementation has, so that a swapped nibble order, a sign rule of two's
complement, a group index off by one or a wrong rounding all fail."""
import numpy as np
import pytest

import oracle


def words(*vals):
    return np.array([v - (1 << 32) if v >= 1 << 31 else v for v in vals], dtype=np.int32)


def test_nibble_order_lowest_first():
    assert oracle.unpack_u4(words(0x76543210)).tolist() == [0, 1, 2, 3, 4, 5, 6, 7]
    assert oracle.unpack_u4(words(0xFEDCBA98)).tolist() == [8, 9, 10, 11, 12, 13, 14, 15]
    assert oracle.unpack_u4(words(0x0000000F)).tolist() == [15, 0, 0, 0, 0, 0, 0, 0]


def test_words_with_the_sign_bit_set():
    # int32 -1 and INT32_MIN: the sign bit is just the top nibble's high bit
    assert oracle.unpack_u4(words(0xFFFFFFFF)).tolist() == [15] * 8
    assert oracle.unpack_u4(words(0x80000000)).tolist() == [0] * 7 + [8]


def test_offset_binary_reconstruction():
    # u4 0..15 -> s4 -8..7; 8 is zero, 0 the most negative (two's complement
    # would map 15 to -1 instead)
    assert oracle.s4_from_u4(np.arange(16)).tolist() == list(range(-8, 8))


def test_unit_scale_gives_the_signed_nibbles():
    one = np.full((1, 1), 0x3F80, dtype=np.uint16)  # bf16 1.0
    row = np.tile(words(0x76543210, 0xFEDCBA98), 8)[None, :]  # 16 words = 128 weights
    w = oracle.w4a16_dequant(row, one)
    assert w.shape == (1, 128)
    assert w[0, :16].tolist() == list(range(-8, 8))
    assert w[0, 112:].tolist() == list(range(-8, 8))


def test_group_boundaries():
    # two groups with scales 1.0 and -2.0: columns 127 and 128 straddle them
    scales = np.array([[0x3F80, 0xC000]], dtype=np.uint16)
    row = np.full((1, 32), words(0xFFFFFFFF)[0], dtype=np.int32)  # every s4 = 7
    w = oracle.w4a16_dequant(row, scales)
    assert w[0, 0] == 7.0 and w[0, 127] == 7.0
    assert w[0, 128] == -14.0 and w[0, 255] == -14.0


def test_rounding_to_bf16_is_nearest_even():
    # 1 + 2^-8 lies halfway between bf16 1.0 (0x3F80) and 1 + 2^-7 (0x3F81):
    # ties go to the even one, 0x3F80; 1 + 3*2^-8 is halfway between 0x3F81 and
    # 0x3F82 and goes to 0x3F82; 1 + 2^-8 + 2^-20 is above halfway: 0x3F81.
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -20, -7.0])
    assert oracle.f64_to_bf16_bits(x).tolist() == [0x3F80, 0x3F82, 0x3F81, 0xC0E0]


def test_products_round_once():
    # scale 1.0078125 (bf16 0x3F81) times 7 = 7.0546875, exactly between no bf16
    # pair's midpoint: bf16 values near 7 are 1/32 apart (7.03125, 7.0625);
    # 7.0546875 is nearer 7.0625 (0x40E2)
    scales = np.array([[0x3F81]], dtype=np.uint16)
    row = np.full((1, 16), words(0xFFFFFFFF)[0], dtype=np.int32)
    assert oracle.w4a16_dequant(row, scales)[0, 0] == 7.0546875
    assert int(oracle.w4a16_dequant_bf16(row, scales)[0, 0]) == 0x40E2


def test_pack_then_dequant_round_trips():
    # packing signed values by the stated layout and dequantising gives them back
    rng = np.random.default_rng(0)
    s4 = rng.integers(-8, 8, size=(3, 256))
    u4 = (s4 + 8).astype(np.int64).reshape(3, 32, 8)
    packed = np.zeros((3, 32), dtype=np.int64)
    for i in range(8):
        packed |= u4[:, :, i] << (4 * i)
    packed = np.where(packed >= 1 << 31, packed - (1 << 32), packed).astype(np.int32)
    one = np.full((3, 2), 0x3F80, dtype=np.uint16)
    assert np.array_equal(oracle.w4a16_dequant(packed, one), s4.astype(np.float64))


def test_rejects_values_float32_cannot_hold():
    with pytest.raises(AssertionError):
        oracle.f64_to_bf16_bits(np.array([1.0 + 2.0 ** -40]))
