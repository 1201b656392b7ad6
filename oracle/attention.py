"""Float64 oracle for the paged KV-cache attention hot path.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline / reference leg; never by the product library.

What it restates, and where the pages state it:

* Fixed blocks of 256 tokens, managed by a block manager
  (nano-vllm hub page, pomoai.com, "core tech 4: KV Cache block manager").
* A block table maps a sequence's logical blocks to physical blocks, and a new
  block is allocated when the length reaches a multiple of 256 plus one
  (257, 513, ...)  (CSDN essay "from nanoVLLM to vLLM", Mountain 1: KV cache).
* New keys/values are written into the preallocated cache blocks through a
  slot mapping (nano-vllm hub page, "core tech 2: Attention + Triton kernel").
* The attention result is that of standard attention: FlashAttention only
  reorders the computation so tiles stay on chip (CSDN essay, Mountain 3:
  attention).  So the oracle is the plain definition softmax(q K^T * scale) V,
  evaluated on the gathered (unpaged) keys and values.

Readings where the pages are silent (each listed in the design notes):
  cache layout [NB, block_size, Hkv, D]; slot = block_table[p // bs] * bs + p % bs;
  slot -1 means "skip"; context_lens include the token(s) just stored; query
  head h reads kv head h // (Hq / Hkv); a prefill query i of a sequence with c
  cached tokens sits at absolute position c + i and sees keys 0..c+i; the
  softmax base is e and the logits are multiplied by `scale`.

bf16 inputs are uint16 bit patterns; the oracle widens them exactly to float64
and never rounds its result back to bf16.
"""
from __future__ import annotations

import numpy as np

BLOCK_SIZE = 256


# ---------------------------------------------------------------- data types

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns: bf16 is the top half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ------------------------------------------------------- block bookkeeping

def blocks_for_length(length: int, block_size: int = BLOCK_SIZE) -> int:
    """Blocks a sequence of `length` tokens occupies: ceil(length / block_size)."""
    return (int(length) + block_size - 1) // block_size


def allocation_points(max_len: int, block_size: int = BLOCK_SIZE) -> list[int]:
    """Lengths at which appending one token at a time allocates a new block.

    Simulates a sequence growing from 0 to max_len tokens; a block is taken
    whenever the token being appended does not fit in the blocks already held
    (CSDN essay, Mountain 1: a new block appears at 257, 513, ...)."""
    held = 0
    points = []
    for length in range(1, max_len + 1):
        if length > held * block_size:
            held += 1
            points.append(length)
    return points


def slot_of(block_table_row: np.ndarray, pos: int, block_size: int = BLOCK_SIZE) -> int:
    """Physical slot of logical token `pos`: its block's id times block_size
    plus the offset inside the block."""
    return int(block_table_row[pos // block_size]) * block_size + pos % block_size


def kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """GQA: consecutive groups of Hq/Hkv query heads share one kv head."""
    return h // (num_q_heads // num_kv_heads)


# ----------------------------------------------------------------- kv_store

def kv_store(k_cache, v_cache, k, v, slot_mapping):
    """Scatter each new token's K and V row into its slot (bit copy).

    k_cache/v_cache: uint16 [NB, BS, Hkv, D]; k/v: uint16 [T, Hkv, D];
    slot_mapping: [T], -1 = skip.  Returns new arrays; the inputs are untouched.
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    nb, bs = kc.shape[0], kc.shape[1]
    for t in range(len(slot_mapping)):
        slot = int(slot_mapping[t])
        if slot < 0:
            continue
        assert slot < nb * bs, "slot outside the cache"
        kc[slot // bs, slot % bs] = k[t]
        vc[slot // bs, slot % bs] = v[t]
    return kc, vc


def gather_sequence(cache: np.ndarray, block_table_row: np.ndarray, length: int) -> np.ndarray:
    """Walk the block table and return the sequence's rows in logical order:
    [length, Hkv, D], row p taken from block block_table_row[p // bs], offset p % bs."""
    bs = cache.shape[1]
    out = np.empty((length,) + cache.shape[2:], dtype=cache.dtype)
    for p in range(length):
        out[p] = cache[int(block_table_row[p // bs]), p % bs]
    return out


# ---------------------------------------------------------------- attention

def attend(q_vec: np.ndarray, keys: np.ndarray, values: np.ndarray, scale: float) -> np.ndarray:
    """Standard attention of one query over n keys, float64.

    s_p = scale * <q, k_p>;  w = exp(s - max s) / sum exp(s - max s);  out = sum_p w_p v_p.
    """
    s = scale * (keys @ q_vec)
    w = np.exp(s - s.max())
    w /= w.sum()
    return w @ values


def paged_decode_attn(q, k_cache, v_cache, block_tables, context_lens, scale,
                      num_kv_heads=None, seqs=None):
    """Decode attention: the single query of sequence s attends to all
    context_lens[s] tokens of its paged K/V.

    q: uint16 [S, Hq, D].  Returns float64 [S, Hq, D] (rows of sequences not in
    `seqs`, when given, are left NaN)."""
    S, Hq, D = q.shape
    Hkv = k_cache.shape[2] if num_kv_heads is None else num_kv_heads
    out = np.full((S, Hq, D), np.nan)
    for s in (range(S) if seqs is None else seqs):
        L = int(context_lens[s])
        K = bf16_bits_to_f64(gather_sequence(k_cache, block_tables[s], L))
        V = bf16_bits_to_f64(gather_sequence(v_cache, block_tables[s], L))
        qs = bf16_bits_to_f64(q[s])
        for h in range(Hq):
            j = kv_head_of(h, Hq, Hkv)
            out[s, h] = attend(qs[h], K[:, j, :], V[:, j, :], scale)
    return out


def paged_prefill_attn(q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k, scale,
                       rows=None):
    """Causal prefill over a paged cache with an optional cached prefix.

    For sequence s with n = cu_q[s+1]-cu_q[s] new queries and len_k =
    cu_k[s+1]-cu_k[s] keys (c = len_k - n of them cached before this step),
    query i sits at absolute position c + i and attends to keys 0..c+i.

    q: uint16 [T_q, Hq, D].  Returns float64 [T_q, Hq, D]; when `rows` (global
    query indices) is given only those rows are computed, the rest stay NaN.
    """
    T, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    out = np.full((T, Hq, D), np.nan)
    wanted = None if rows is None else set(int(r) for r in rows)
    S = len(cu_seqlens_q) - 1
    for s in range(S):
        q0, q1 = int(cu_seqlens_q[s]), int(cu_seqlens_q[s + 1])
        n = q1 - q0
        len_k = int(cu_seqlens_k[s + 1]) - int(cu_seqlens_k[s])
        c = len_k - n
        todo = [r for r in range(q0, q1) if wanted is None or r in wanted]
        if not todo:
            continue
        K = bf16_bits_to_f64(gather_sequence(k_cache, block_tables[s], len_k))
        V = bf16_bits_to_f64(gather_sequence(v_cache, block_tables[s], len_k))
        for r in todo:
            i = r - q0
            visible = c + i + 1
            qr = bf16_bits_to_f64(q[r])
            for h in range(Hq):
                j = kv_head_of(h, Hq, Hkv)
                out[r, h] = attend(qr[h], K[:visible, j, :], V[:visible, j, :], scale)
    return out
