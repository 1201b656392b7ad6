"""CPU oracle for attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline / reference leg may import this package.  The CUDA library never
calls it, and it shares no code with the CUDA path.

It is a plain, slow, obviously-correct restatement of what the path computes,
in float64 (see `attention.py`).
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
