"""Seeded synthetic inputs for paged KV-cache attention.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It holds no attention arithmetic: only random draws, the rounding of
those draws to bf16 bit patterns, the assignment of physical blocks to
sequences, and the slot bookkeeping that an engine's block manager hands to the
kernels (the 256-token blocks of the nano-vllm hub page, "KV Cache block
manager"; the block table of the CSDN essay "from nanoVLLM to vLLM",
Mountain 1).

All tensors are numpy arrays.  bf16 values are carried as their uint16 bit
patterns so that every consumer reads identical bits.

Layouts (the pages give none; these are the readings used everywhere):
  q            [T_q, Hq, D]             bf16 bits
  k, v         [T_new, Hkv, D]          bf16 bits (this step's new tokens)
  k/v_cache    [NB, block_size, Hkv, D] bf16 bits (one slot = Hkv*D values)
  slot_mapping [T_new] int32, -1 = padding (skip)
  block_tables [S, max_blocks] int32, padded with -1
  context_lens [S] int32 (tokens visible, including this step's new ones)
  cu_seqlens_q [S+1] int32, cu_seqlens_k [S+1] int32
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BLOCK_SIZE = 256  # fixed-size KV blocks of 256 tokens (nano-vllm hub page, block manager)

# bf16 bit pattern of a quiet NaN; used to poison cache slots nobody may read.
BF16_QNAN = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 with round-to-nearest-even; return uint16 bits.

    Inputs are finite draws (no NaN/Inf handling is needed for them)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) draws in fp32, rounded to bf16 bits."""
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def blocks_for(length: int, block_size: int = BLOCK_SIZE) -> int:
    return -(-int(length) // block_size)


@dataclass
class PagedBatch:
    """One step's inputs for kv_store followed by decode or prefill attention."""

    name: str
    kind: str  # "decode" (one query per sequence) or "prefill"
    seed: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    cached_lens: np.ndarray  # int64 [S]: tokens already in the cache
    new_lens: np.ndarray  # int64 [S]: tokens stored by this step
    block_tables: np.ndarray  # int32 [S, max_blocks], -1 padded
    slot_mapping: np.ndarray  # int32 [T_new]
    q: np.ndarray  # uint16 [T_q, Hq, D]
    k: np.ndarray  # uint16 [T_new, Hkv, D]
    v: np.ndarray  # uint16 [T_new, Hkv, D]
    k_cache: Optional[np.ndarray]  # uint16 [NB, BS, Hkv, D] before the store
    v_cache: Optional[np.ndarray]
    scale: float
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.cached_lens.shape[0])

    @property
    def context_lens(self) -> np.ndarray:
        return (self.cached_lens + self.new_lens).astype(np.int32)

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        lens = np.ones_like(self.new_lens) if self.kind == "decode" else self.new_lens
        return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)

    @property
    def cu_seqlens_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.context_lens)]).astype(np.int32)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def total_blocks_used(self) -> int:
        return int(sum(blocks_for(L, self.block_size) for L in self.context_lens))


def build_batch(
    name: str,
    kind: str,
    seed: int,
    cached_lens,
    new_lens,
    num_q_heads: int,
    num_kv_heads: int,
    head_dim: int,
    block_size: int = BLOCK_SIZE,
    num_blocks: Optional[int] = None,
    fill_cache: bool = True,
    stale: str = "normal",
    rng: Optional[np.random.Generator] = None,
    max_blocks_pad: int = 0,
) -> PagedBatch:
    """Assemble a batch: shuffled block pool, block tables, slots and bf16 data.

    cached_lens[s] tokens of sequence s are already in the cache (random data);
    new_lens[s] tokens are this step's new K/V, stored through slot_mapping.
    Each sequence holds ceil((cached+new)/block_size) blocks drawn, in order,
    from a seeded permutation of the pool.  `stale` sets what fills cache slots
    at or beyond a sequence's context length: "normal" (random) or "nan".
    `max_blocks_pad` adds that many extra -1 columns to the block table.
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    cached = np.asarray(cached_lens, dtype=np.int64)
    new = np.asarray(new_lens, dtype=np.int64)
    assert cached.shape == new.shape
    if kind == "decode":
        assert np.all(new == 1), "decode steps store exactly one token per sequence"
    ctx = cached + new
    nblk = np.array([blocks_for(L, block_size) for L in ctx], dtype=np.int64)
    used = int(nblk.sum())
    if num_blocks is None:
        num_blocks = used
    assert used <= num_blocks, "pool too small for the contexts"
    S = cached.shape[0]
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_blocks = int(nblk.max()) + max_blocks_pad if S else 1
    block_tables = np.full((S, max(max_blocks, 1)), -1, dtype=np.int32)
    off = 0
    for s in range(S):
        block_tables[s, : nblk[s]] = perm[off : off + nblk[s]]
        off += nblk[s]

    T_new = int(new.sum())
    T_q = S if kind == "decode" else T_new
    q = normal_bf16(rng, (T_q, num_q_heads, head_dim))
    k = normal_bf16(rng, (T_new, num_kv_heads, head_dim))
    v = normal_bf16(rng, (T_new, num_kv_heads, head_dim))

    slot_mapping = np.empty(T_new, dtype=np.int32)
    t = 0
    for s in range(S):
        for i in range(int(new[s])):
            pos = int(cached[s]) + i
            slot_mapping[t] = int(block_tables[s, pos // block_size]) * block_size + pos % block_size
            t += 1

    k_cache = v_cache = None
    if fill_cache:
        shape = (num_blocks, block_size, num_kv_heads, head_dim)
        k_cache = np.zeros(shape, dtype=np.uint16)
        v_cache = np.zeros(shape, dtype=np.uint16)
        for cache in (k_cache, v_cache):
            for s in range(S):
                ids = block_tables[s, : nblk[s]]
                cache[ids] = normal_bf16(rng, (len(ids), block_size, num_kv_heads, head_dim))
                if stale == "nan":
                    for p in range(int(ctx[s]), int(nblk[s]) * block_size):
                        cache[ids[p // block_size], p % block_size] = BF16_QNAN
    return PagedBatch(
        name=name,
        kind=kind,
        seed=seed,
        num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads,
        head_dim=head_dim,
        block_size=block_size,
        num_blocks=num_blocks,
        cached_lens=cached,
        new_lens=new,
        block_tables=block_tables,
        slot_mapping=slot_mapping,
        q=q,
        k=k,
        v=v,
        k_cache=k_cache,
        v_cache=v_cache,
        scale=1.0 / float(np.sqrt(head_dim)),
    )


# ---------------------------------------------------------------------------
# The five named workloads.  Seeds are the workload index (tiny=1 ... prefix=5).
# ---------------------------------------------------------------------------

def tiny(fill_cache: bool = True) -> PagedBatch:
    """2 sequences with context 5 and 300 (crosses the 256->257 block boundary),
    4 q heads / 2 kv heads, D=64, an 8-block pool in seeded random order; one
    new token per sequence stored, then decode."""
    return build_batch("tiny", "decode", 1, [4, 299], [1, 1], 4, 2, 64, num_blocks=8,
                       fill_cache=fill_cache)


def decode(fill_cache: bool = True) -> PagedBatch:
    """64 sequences, context ~ U[128, 2048], 16 q / 8 kv heads, D=128, a
    1024-block pool with permuted block tables; one store per sequence, then decode."""
    rng = np.random.default_rng(2)
    L = rng.integers(128, 2048, size=64, endpoint=True)
    return build_batch("decode", "decode", 2, L - 1, np.ones(64, np.int64), 16, 8, 128,
                       num_blocks=1024, fill_cache=fill_cache, rng=rng)


def longdecode_lengths(rng: np.random.Generator, n: int = 256) -> np.ndarray:
    """Context lengths ~ lognormal with median 1024 (sigma 1 in log space),
    rounded, clamped to [1, 32768]."""
    L = np.rint(rng.lognormal(mean=np.log(1024.0), sigma=1.0, size=n))
    return np.clip(L, 1, 32768).astype(np.int64)


def longdecode(fill_cache: bool = True) -> PagedBatch:
    """256 sequences with lognormal contexts capped at 32768, 32 q / 8 kv
    heads, D=128, a shuffled pool sized exactly to the contexts."""
    rng = np.random.default_rng(3)
    L = longdecode_lengths(rng)
    return build_batch("longdecode", "decode", 3, L - 1, np.ones(L.shape[0], np.int64), 32, 8,
                       128, fill_cache=fill_cache, rng=rng)


def prefill(fill_cache: bool = True) -> PagedBatch:
    """16 prompts with lengths ~ U[64, 4096] packed by cu_seqlens, 16 q / 8 kv
    heads, D=128; K/V stored into a shuffled pool via slot_mapping, then causal
    attention over the cache."""
    rng = np.random.default_rng(4)
    n = rng.integers(64, 4096, size=16, endpoint=True)
    return build_batch("prefill", "prefill", 4, np.zeros(16, np.int64), n, 16, 8, 128,
                       fill_cache=fill_cache, rng=rng)


def prefix(fill_cache: bool = True) -> PagedBatch:
    """32 sequences with k*256 cached tokens (k in {0,1,2,4}) plus U[1, 512]
    new tokens, 16 q / 8 kv heads, D=128, shuffled blocks; the causal mask is
    offset by the cached length."""
    rng = np.random.default_rng(5)
    c = 256 * rng.choice(np.array([0, 1, 2, 4]), size=32)
    n = rng.integers(1, 512, size=32, endpoint=True)
    return build_batch("prefix", "prefill", 5, c, n, 16, 8, 128, fill_cache=fill_cache, rng=rng)


def mixed(fill_cache: bool = True) -> PagedBatch:
    """One engine step of chunked prefill mixed with decode: 48 decode rows
    (one new token, contexts ~ U[128, 2048]) and 8 prompt chunks of
    U[256, 1024] new tokens after U[0, 2048] cached ones, 16 q / 8 kv heads,
    D=128, served by one prefill launch."""
    rng = np.random.default_rng(6)
    dec_ctx = rng.integers(128, 2048, size=48, endpoint=True)
    chunk_new = rng.integers(256, 1024, size=8, endpoint=True)
    chunk_cached = rng.integers(0, 2048, size=8, endpoint=True)
    cached = np.concatenate([dec_ctx - 1, chunk_cached])
    new = np.concatenate([np.ones(48, np.int64), chunk_new])
    return build_batch("mixed", "prefill", 6, cached, new, 16, 8, 128, fill_cache=fill_cache,
                       rng=rng)


WORKLOADS = {"tiny": tiny, "decode": decode, "longdecode": longdecode, "prefill": prefill,
             "prefix": prefix, "mixed": mixed}


# ------------------------------------------------ W4A16-G128 weight inputs

@dataclass
class W4A16Weight:
    """A quantised weight [n, k]: packed int32 words [n, k/8] (8 nibbles each)
    and bf16 scale bits [n, k/128] (one per 128 weights)."""
    name: str
    packed: np.ndarray
    scales: np.ndarray

    @property
    def shape(self):
        return self.packed.shape[0], self.packed.shape[1] * 8


def w4a16_weight(name: str, seed: int, n: int, k: int) -> W4A16Weight:
    """Uniformly random words (every nibble value equally likely) and scales
    drawn from N(0, 0.02^2) rounded to bf16, a typical magnitude for the
    per-group scales of a 4-bit linear layer."""
    assert k % 128 == 0
    rng = np.random.default_rng(seed)
    packed = rng.integers(-(1 << 31), 1 << 31, size=(n, k // 8), dtype=np.int64).astype(np.int32)
    scales = f32_to_bf16_bits(0.02 * rng.standard_normal(size=(n, k // 128), dtype=np.float32))
    return W4A16Weight(name, packed, scales)


def dequant_small() -> W4A16Weight:
    """3 rows x 384 inputs (three groups per row): parity-test size."""
    return w4a16_weight("dequant_small", 11, 3, 384)


def dequant() -> W4A16Weight:
    """One 4096 x 14336 projection (58.7M weights: 29 MB packed, 117 MB out),
    the size of an MLP up-projection of a mid-size model."""
    return w4a16_weight("dequant", 12, 4096, 14336)
