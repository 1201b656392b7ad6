"""The synthetic workloads have the shapes, sizes and structure of the
stated configurations (tiny decode+store, decode batch, long skewed decode,
varlen prefill, prefix-cached prefill, the mixed step), are reproducible from
their seeds, and every sequence's blocks are distinct blocks of the pool."""
import numpy as np
import pytest

import workloads as wl


def built(name):
    return wl.WORKLOADS[name](fill_cache=False)


def check_structure(b):
    S = b.num_seqs
    L = b.cached_lens + b.new_lens
    nb = np.array([wl.blocks_for(int(x), b.block_size) for x in L])
    used = np.concatenate([b.block_tables[s, :nb[s]] for s in range(S)])
    assert (used >= 0).all() and (used < b.num_blocks).all()
    assert len(np.unique(used)) == len(used), "a block is shared by two sequences"
    for s in range(S):
        assert (b.block_tables[s, nb[s]:] == -1).all()
    assert b.slot_mapping.shape[0] == int(b.new_lens.sum())
    assert len(np.unique(b.slot_mapping)) == b.slot_mapping.shape[0]
    assert b.q.dtype == np.uint16 and b.k.shape == (int(b.new_lens.sum()), b.num_kv_heads,
                                                    b.head_dim)
    assert b.scale == pytest.approx(1.0 / np.sqrt(b.head_dim))


def test_tiny():
    b = built("tiny")
    assert list(b.cached_lens + b.new_lens) == [5, 300] and list(b.new_lens) == [1, 1]
    assert (b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size) == (4, 2, 64, 256)
    assert b.num_blocks == 8
    check_structure(b)


def test_decode_batch():
    b = built("decode")
    L = b.cached_lens + b.new_lens
    assert b.num_seqs == 64 and (b.new_lens == 1).all()
    assert L.min() >= 128 and L.max() <= 2048
    assert (b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size) == (16, 8, 128, 256)
    assert b.num_blocks == 1024
    check_structure(b)


def test_long_skewed_decode():
    b = built("longdecode")
    L = b.cached_lens + b.new_lens
    assert b.num_seqs == 256 and (b.new_lens == 1).all()
    assert L.min() >= 1 and L.max() <= 32768
    assert 700 <= np.median(L) <= 1400  # lognormal with median 1024
    assert (b.num_q_heads, b.num_kv_heads, b.head_dim) == (32, 8, 128)
    # a pool sized exactly to the contexts
    assert b.num_blocks == sum(wl.blocks_for(int(x)) for x in L)
    check_structure(b)


def test_varlen_prefill():
    b = built("prefill")
    assert b.num_seqs == 16 and (b.cached_lens == 0).all()
    assert b.new_lens.min() >= 64 and b.new_lens.max() <= 4096
    assert list(b.cu_seqlens_q) == [0] + list(np.cumsum(b.new_lens))
    assert (b.num_q_heads, b.num_kv_heads, b.head_dim) == (16, 8, 128)
    check_structure(b)


def test_prefix_cached_prefill():
    b = built("prefix")
    assert b.num_seqs == 32
    assert set(np.unique(b.cached_lens // 256)) <= {0, 1, 2, 4} and (b.cached_lens % 256 == 0).all()
    assert b.new_lens.min() >= 1 and b.new_lens.max() <= 512
    assert list(b.cu_seqlens_k) == [0] + list(np.cumsum(b.cached_lens + b.new_lens))
    check_structure(b)


def test_mixed_step():
    b = built("mixed")
    assert b.num_seqs == 56
    assert (b.new_lens[:48] == 1).all()
    ctx = b.cached_lens[:48] + 1
    assert ctx.min() >= 128 and ctx.max() <= 2048
    assert b.new_lens[48:].min() >= 256 and b.new_lens[48:].max() <= 1024
    assert b.cached_lens[48:].max() <= 2048
    check_structure(b)


@pytest.mark.parametrize("name", ["tiny", "decode", "prefix", "mixed"])
def test_seeded_and_reproducible(name):
    a, b = built(name), built(name)
    for f in ("cached_lens", "new_lens", "block_tables", "slot_mapping", "q", "k", "v"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
