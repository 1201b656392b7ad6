"""W4A16-G128 dequantisation on the GPU: bit-exact against the oracle (the
product is exact in fp32 and both sides round it once to bf16)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import bits

pytestmark = pytest.mark.gpu


def run(lib, w, offset_elems=0):
    n, k = w.shape
    packed = torch.from_numpy(w.packed).cuda()
    scales = torch.from_numpy(w.scales.view(np.int16)).view(torch.bfloat16).cuda()
    buf = torch.full((n * k + offset_elems,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = buf[offset_elems:].view(n, k)
    lib.w4a16_dequant(out, packed, scales)
    torch.cuda.synchronize()
    return out, buf


@pytest.mark.parametrize("shape", [(1, 128), (3, 384), (5, 1024), (7, 4096), (64, 128 * 33)])
def test_dequant_bit_exact(lib, shape):
    w = wl.w4a16_weight("t", 20 + shape[0], *shape)
    out, _ = run(lib, w)
    assert np.array_equal(bits(out), oracle.w4a16_dequant_bf16(w.packed, w.scales))


def test_dequant_every_nibble_value_and_sign(lib):
    # words cycling through all 16 nibble values in every position, scales
    # of both signs and a range of exponents
    n, k = 4, 256
    base = np.array([0x76543210, 0xFEDCBA98, 0x89ABCDEF, 0x01234567], dtype=np.int64)
    packed = np.resize(base, (n, k // 8))
    packed = np.where(packed >= 1 << 31, packed - (1 << 32), packed).astype(np.int32)
    scales = np.array([[0x3F80, 0xBF80], [0x0080, 0x7D00], [0x3C23, 0xC123], [0x4000, 0x3E80]],
                      dtype=np.uint16)
    w = wl.W4A16Weight("signs", packed, scales)
    out, _ = run(lib, w)
    assert np.array_equal(bits(out), oracle.w4a16_dequant_bf16(packed, scales))


def test_dequant_out_only_16_byte_aligned(lib):
    # 32-byte stores when out allows them, 16-byte stores otherwise
    w = wl.w4a16_weight("align", 30, 6, 512)
    out, buf = run(lib, w, offset_elems=8)
    assert out.data_ptr() % 32 == 16
    assert np.array_equal(bits(out), oracle.w4a16_dequant_bf16(w.packed, w.scales))
    assert torch.isnan(buf[:8].float()).all()  # nothing written before out


def test_dequant_full_size_sampled_rows(lib):
    w = wl.dequant()
    out, _ = run(lib, w)
    rows = np.random.default_rng(5).choice(w.shape[0], size=48, replace=False)
    got = bits(out[torch.as_tensor(rows, device="cuda")])
    assert np.array_equal(got, oracle.w4a16_dequant_bf16(w.packed[rows], w.scales[rows]))
