"""CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline / reference leg may import this package.  The CUDA library never
calls it, and it shares no code with the CUDA path.

It is a plain, slow, obviously-correct restatement of what the path computes,
in float64 (see `attention.py`; the W4A16-G128 dequantisation in `dequant.py`).
"""
from .attention import (  # noqa: F401
    BLOCK_SIZE,
    allocation_points,
    attend,
    bf16_bits_to_f64,
    blocks_for_length,
    gather_sequence,
    kv_head_of,
    kv_store,
    paged_decode_attn,
    paged_prefill_attn,
    slot_of,
)
from .dequant import (  # noqa: F401
    GROUP,
    f64_to_bf16_bits,
    s4_from_u4,
    unpack_u4,
    w4a16_dequant,
    w4a16_dequant_bf16,
)
