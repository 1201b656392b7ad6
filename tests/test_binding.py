"""The Python binding only marshals device tensors: host tensors, wrong dtypes
or ranks and inconsistent shapes are refused before the library is called,
so there is no path that computes on the CPU (no GPU needed)."""
import pytest
import torch

import paged_kv_cache_241_gb300 as pkv

bf16, i32 = torch.bfloat16, torch.int32


def host_decode_args(S=2, Hq=4, Hkv=2, D=64, NB=8, BS=256, maxb=2):
    return dict(out=torch.zeros(S, Hq, D, dtype=bf16), q=torch.zeros(S, Hq, D, dtype=bf16),
                k_cache=torch.zeros(NB, BS, Hkv, D, dtype=bf16),
                v_cache=torch.zeros(NB, BS, Hkv, D, dtype=bf16),
                block_tables=torch.zeros(S, maxb, dtype=i32),
                context_lens=torch.ones(S, dtype=i32), scale=0.125,
                workspace=torch.zeros(4096, dtype=torch.uint8), max_total_blocks=4)


def test_decode_refuses_host_tensors():
    with pytest.raises(ValueError, match="CUDA"):
        pkv.paged_decode_attn(**host_decode_args())


def test_decode_refuses_a_wrong_dtype():
    # (each argument's dtype is checked before its device)
    a = host_decode_args()
    a["out"] = a["out"].float()
    with pytest.raises(TypeError, match="out"):
        pkv.paged_decode_attn(**a)


def test_prefill_refuses_host_tensors():
    T, Hq, Hkv, D = 5, 4, 2, 64
    with pytest.raises(ValueError, match="CUDA"):
        pkv.paged_prefill_attn(torch.zeros(T, Hq, D, dtype=bf16), torch.zeros(T, Hq, D, dtype=bf16),
                               torch.zeros(4, 256, Hkv, D, dtype=bf16),
                               torch.zeros(4, 256, Hkv, D, dtype=bf16),
                               torch.zeros(1, 1, dtype=i32), torch.tensor([0, T], dtype=i32),
                               torch.tensor([0, T], dtype=i32), T, 0.125)


def test_kv_store_refuses_host_tensors():
    k = torch.zeros(3, 2, 64, dtype=bf16)
    with pytest.raises(ValueError, match="CUDA"):
        pkv.kv_store(k, k.clone(), torch.zeros(4, 256, 2, 64, dtype=bf16),
                     torch.zeros(4, 256, 2, 64, dtype=bf16), torch.zeros(3, dtype=i32))


def test_dequant_refuses_host_tensors_and_a_wrong_dtype():
    with pytest.raises(ValueError, match="CUDA"):
        pkv.w4a16_dequant(torch.zeros(4, 128, dtype=bf16), torch.zeros(4, 16, dtype=i32),
                          torch.zeros(4, 1, dtype=bf16))
    with pytest.raises(TypeError, match="out"):
        pkv.w4a16_dequant(torch.zeros(4, 128, dtype=torch.float16), torch.zeros(4, 16, dtype=i32),
                          torch.zeros(4, 1, dtype=bf16))
