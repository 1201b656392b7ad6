"""kv_store on the GPU: bit-exact against the oracle's scatter, untouched slots
unchanged, padding and bad slots handled."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import DeviceBatch, bf16, bits, i32, oracle_caches

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("make", [wl.tiny, wl.decode, wl.prefill, wl.prefix])
def test_kv_store_bit_exact(lib, make):
    b = make()
    db = DeviceBatch(lib, b)
    ekc, evc = oracle_caches(b)
    assert np.array_equal(bits(db.k_cache), ekc)
    assert np.array_equal(bits(db.v_cache), evc)
    assert db.status_value() == 0


def test_kv_store_sentinel_padding_and_strided_rows(lib):
    rng = np.random.default_rng(3)
    NB, BS, Hkv, D, T = 6, 64, 2, 64, 40
    kc0 = np.full((NB, BS, Hkv, D), 0xAAAA, np.uint16)
    vc0 = np.full((NB, BS, Hkv, D), 0x5555, np.uint16)
    # k and v come from one fused qkv-like buffer: rows are strided
    fused = wl.normal_bf16(rng, (T, 3, Hkv, D))
    slots = rng.permutation(NB * BS)[:T].astype(np.int32)
    slots[::7] = -1  # padding tokens
    kc, vc = bf16(kc0), bf16(vc0)
    f = bf16(fused)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kv_store(f[:, 1], f[:, 2], kc, vc, i32(slots), status)
    ekc, evc = oracle.kv_store(kc0, vc0, fused[:, 1], fused[:, 2], slots)
    assert np.array_equal(bits(kc), ekc) and np.array_equal(bits(vc), evc)
    assert int(status.item()) == 0


def test_kv_store_flags_out_of_range_slot_and_skips_it(lib):
    rng = np.random.default_rng(4)
    NB, BS, Hkv, D = 2, 64, 1, 64
    kc0 = np.full((NB, BS, Hkv, D), 0x1234, np.uint16)
    k = wl.normal_bf16(rng, (3, Hkv, D))
    slots = np.array([5, NB * BS, -7], np.int32)  # valid, one past the end, negative
    kc, vc = bf16(kc0), bf16(kc0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kv_store(bf16(k), bf16(k), kc, vc, i32(slots), status)
    torch.cuda.synchronize()
    assert int(status.item()) & lib.DEV_BAD_SLOT
    want, _ = oracle.kv_store(kc0, kc0, k[:1], k[:1], slots[:1])
    assert np.array_equal(bits(kc), want)
