"""Paged decode attention on the GPU against the fp64 oracle.

Tolerance: |gpu - oracle| <= 8e-3 + 1e-2 |oracle| elementwise (bf16 inputs,
fp32 accumulation, bf16 output)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import DeviceBatch, assert_close, bf16, bits, i32, oracle_caches

pytestmark = pytest.mark.gpu


def check_decode(lib, b, seqs=None, max_total_blocks=None):
    db = DeviceBatch(lib, b)
    out = db.decode(max_total_blocks)
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle.paged_decode_attn(b.q, ekc, evc, b.block_tables, b.context_lens, b.scale,
                                    seqs=seqs)
    got = out.double().cpu().numpy()
    rows = slice(None) if seqs is None else list(seqs)
    assert_close(got[rows], want[rows], f"decode {b.name}")
    return db, out


def test_decode_tiny(lib):
    check_decode(lib, wl.tiny())


def test_decode_batch_full_size(lib):
    check_decode(lib, wl.decode())


def test_longdecode_every_sequence(lib):
    # 256 sequences, lognormal contexts up to 32768, 32 q / 8 kv heads
    check_decode(lib, wl.longdecode())


def counter_batch(G, seed):
    """Many items per CTA (about 14K (sequence, kv head, 64-token block)
    items): the kernel then hands items out through its workspace counter."""
    rng = np.random.default_rng(seed)
    L = rng.integers(3000, 4000, size=128, endpoint=True)
    return wl.build_batch("counter", "decode", seed, L - 1, np.ones(128, np.int64), 2 * G, 2, 64,
                          block_size=64, rng=rng)


@pytest.mark.parametrize("G", [2, 4])  # 4-deep ring (TMA + cp.async), 3-deep ring (TMA)
def test_decode_items_handed_out_by_the_counter(lib, G):
    b = counter_batch(G, 49 + G)
    db, out = check_decode(lib, b)


def span_batch(G, seed):
    """About 20K (sequence, kv head, block) triples over 160 sequences and 4
    kv heads: items then span two blocks of their sequence (and the merge
    reads the partials' prefix the split-K grid publishes)."""
    rng = np.random.default_rng(seed)
    L = rng.integers(1500, 2500, size=160, endpoint=True)
    L[:3] = [64, 65, 129]  # one block, two blocks (one item), three blocks (two items)
    return wl.build_batch("span", "decode", seed, L - 1, np.ones(160, np.int64), 4 * G, 4, 64,
                          block_size=64, rng=rng)


@pytest.mark.parametrize("G", [2, 4])
def test_decode_items_of_two_blocks(lib, G):
    check_decode(lib, span_batch(G, 57 + G))


def test_decode_batch_of_4096_sequences(lib):
    # A large batch: every CTA keeps all 4096 sequences' block offsets and
    # lengths in shared memory, and the items are handed out by the counter.
    rng = np.random.default_rng(48)
    L = rng.integers(1, 200, size=4096, endpoint=True)
    b = wl.build_batch("big", "decode", 48, L - 1, np.ones(4096, np.int64), 4, 2, 128,
                       block_size=64, rng=rng)
    check_decode(lib, b)


def test_decode_merge_paths_agree_at_the_batch_size_boundary(lib):
    # Up to 128 sequences the merge finds each sequence's partials from
    # context_lens itself; from 129 on it reads the prefix the split-K grid
    # publishes.  The first 128 sequences must come out bit-identical.
    rng = np.random.default_rng(47)
    L = rng.integers(1, 1200, size=129, endpoint=True)
    b = wl.build_batch("edge129", "decode", 47, L - 1, np.ones(129, np.int64), 4, 2, 128, rng=rng)
    db129, out129 = check_decode(lib, b)
    mtb = int(b.total_blocks_used)
    ws = lib.decode_workspace(128, b.num_q_heads, b.num_kv_heads, b.head_dim, mtb, db129.dev)
    out128 = torch.empty((128, b.num_q_heads, b.head_dim), dtype=torch.bfloat16, device=db129.dev)
    lib.paged_decode_attn(out128, db129.q[:128], db129.k_cache, db129.v_cache,
                          db129.block_tables[:128].contiguous(), db129.context_lens[:128].contiguous(),
                          b.scale, ws, mtb, db129.status)
    assert db129.status_value() == 0
    assert np.array_equal(bits(out128), bits(out129[:128]))


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_decode_edge_lengths(lib, D, G):
    lens = [1, 2, 63, 64, 65, 255, 256, 257, 511, 512, 513, 1000]
    Hkv = 2
    b = wl.build_batch("edge", "decode", 10 + G + D, [L - 1 for L in lens], [1] * len(lens),
                       G * Hkv, Hkv, D, num_blocks=40, max_blocks_pad=3)
    check_decode(lib, b)


@pytest.mark.parametrize("scale", [0.0, -1.0 / np.sqrt(128.0)])
@pytest.mark.parametrize("G", [2, 4])
def test_decode_zero_and_negative_scale(lib, scale, G):
    # A negative scale puts each row's largest scaled logit at its smallest
    # q.k; zero gives the mean of the context's values.  Contexts across the
    # 64-token tile and 256-token block boundaries, NaN in stale slots.
    L = np.array([1, 63, 64, 65, 255, 256, 257, 700, 1500, 2048])
    b = wl.build_batch("dscale", "decode", 17 + G, L - 1, np.ones(len(L), np.int64), 4 * G, 4,
                       128, stale="nan")
    b = dataclasses.replace(b, scale=float(scale))
    db, out = check_decode(lib, b)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("bs", [64, 128, 512])
def test_decode_other_block_sizes(lib, bs):
    lens = [1, bs - 1, bs, bs + 1, 3 * bs + 5, 700]
    b = wl.build_batch("bs", "decode", 30 + bs, [L - 1 for L in lens], [1] * len(lens), 8, 2, 128,
                       block_size=bs)
    check_decode(lib, b)


def test_decode_never_reads_stale_slots(lib):
    lens = [3, 256, 257, 300, 700]
    b = wl.build_batch("nan", "decode", 41, [L - 1 for L in lens], [1] * len(lens), 8, 2, 128,
                       stale="nan")
    db, out = check_decode(lib, b)
    assert torch.isfinite(out.float()).all()


def test_decode_context_of_one_returns_v_bits(lib):
    b = wl.build_batch("one", "decode", 42, [0, 0, 0], [1, 1, 1], 8, 4, 128)
    db = DeviceBatch(lib, b)
    out = bits(db.decode())
    for s in range(3):
        for h in range(8):
            assert np.array_equal(out[s, h], b.v[s, h // 2])


def test_decode_workspace_reuse_gives_identical_results(lib):
    b = wl.build_batch("reuse", "decode", 43, [700, 2000, 40], [1, 1, 1], 16, 8, 128)
    db = DeviceBatch(lib, b)
    mtb = b.total_blocks_used
    ws = lib.decode_workspace(b.num_seqs, 16, 8, 128, mtb)
    outs = []
    for _ in range(3):
        out = torch.empty((3, 16, 128), dtype=torch.bfloat16, device="cuda")
        lib.paged_decode_attn(out, db.q, db.k_cache, db.v_cache, db.block_tables,
                              db.context_lens, b.scale, ws, mtb, db.status)
        outs.append(bits(out))
    assert db.status_value() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_decode_workspace_needs_only_its_counter_zeroed(lib):
    # The first 256 bytes (the work counter) must start at zero and every call
    # leaves them at zero; the split-K scratch after them needs no
    # initialisation.
    b = wl.build_batch("dirty", "decode", 45, [700, 2000, 40, 5000], [1, 1, 1, 1], 16, 8, 128)
    db = DeviceBatch(lib, b)
    mtb = b.total_blocks_used
    clean = lib.decode_workspace(b.num_seqs, 16, 8, 128, mtb)
    dirty = torch.full_like(clean, 0xFF)  # scratch bytes 0xFF: NaN floats, -1 ints
    dirty[:256] = 0
    outs = []
    for ws in (clean, dirty, dirty):
        out = torch.empty((b.num_seqs, 16, 128), dtype=torch.bfloat16, device="cuda")
        lib.paged_decode_attn(out, db.q, db.k_cache, db.v_cache, db.block_tables,
                              db.context_lens, b.scale, ws, mtb, db.status)
        outs.append(bits(out))
        torch.cuda.synchronize()
        assert int(ws[:256].count_nonzero().item()) == 0
    assert db.status_value() == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_decode_flags_bad_context_block_and_workspace(lib):
    b = wl.build_batch("err", "decode", 44, [10, 300], [1, 1], 4, 2, 64, num_blocks=6)
    db = DeviceBatch(lib, b)
    # a zero-length context
    db.context_lens[0] = 0
    db.decode()
    assert db.status_value() & lib.DEV_BAD_CONTEXT
    # a block id outside the pool
    db = DeviceBatch(lib, b)
    db.block_tables[1, 1] = 1000
    db.decode()
    assert db.status_value() & lib.DEV_BAD_BLOCK
    # more blocks than the workspace bound
    db = DeviceBatch(lib, b)
    db.decode(max_total_blocks=1)
    assert db.status_value() & lib.DEV_WORKSPACE


def test_decode_step_replays_from_a_cuda_graph(lib):
    """kv_store + paged decode (split-K and its dependent merge launch) have no
    host synchronisation, so a decode step can be captured once and replayed;
    a replay reads the buffers' current contents."""
    lens = [1, 300, 1000, 2048, 513]
    b = wl.build_batch("graph", "decode", 46, [L - 1 for L in lens], [1] * len(lens), 16, 8, 128)
    db = DeviceBatch(lib, b, store=False)
    mtb = b.total_blocks_used
    ws = lib.decode_workspace(b.num_seqs, 16, 8, 128, mtb)
    out = torch.empty((b.num_seqs, 16, 128), dtype=torch.bfloat16, device="cuda")

    def step():
        lib.kv_store(db.k, db.v, db.k_cache, db.v_cache, db.slot_mapping, db.status)
        lib.paged_decode_attn(out, db.q, db.k_cache, db.v_cache, db.block_tables,
                              db.context_lens, b.scale, ws, mtb, db.status)

    step()
    eager = bits(out)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), eager)
    # new queries in the same buffer: the replay follows them
    q2 = wl.normal_bf16(np.random.default_rng(7), b.q.shape)
    db.q.copy_(bf16(q2))
    graph.replay()
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle.paged_decode_attn(q2, ekc, evc, b.block_tables, b.context_lens, b.scale)
    assert_close(out.double().cpu().numpy(), want, "graph replay with new q")


@pytest.mark.parametrize("make", [wl.tiny, wl.decode, lambda: span_batch(2, 61),
                                  lambda: span_batch(4, 62)],
                         ids=["tiny", "decode", "span_g2", "span_g4"])
def test_fused_store_and_decode_match_the_two_calls_bit_for_bit(lib, make):
    b = make()
    two = DeviceBatch(lib, b)            # kv_store, then decode
    ref = bits(two.decode())
    fused = DeviceBatch(lib, b, store=False)
    mtb = b.total_blocks_used
    ws = lib.decode_workspace(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim, mtb)
    out = torch.empty_like(fused.q)
    lib.paged_decode_store_attn(out, fused.q, fused.k, fused.v, fused.slot_mapping,
                                fused.k_cache, fused.v_cache, fused.block_tables,
                                fused.context_lens, b.scale, ws, mtb, fused.status)
    assert fused.status_value() == 0
    assert np.array_equal(bits(out), ref)
    ekc, evc = oracle_caches(b)
    assert np.array_equal(bits(fused.k_cache), ekc) and np.array_equal(bits(fused.v_cache), evc)


def test_fused_store_never_reads_the_new_slot_from_the_cache(lib):
    # stale NaN everywhere past the old context, including the new token's slot
    lens = [1, 256, 257, 700, 2049]
    b = wl.build_batch("fnan", "decode", 47, [L - 1 for L in lens], [1] * len(lens), 8, 2, 128,
                       stale="nan")
    for s_, L in enumerate(lens):  # poison the slot the new token goes to
        slot = int(b.slot_mapping[s_])
        b.k_cache[slot // 256, slot % 256] = 0x7FC0
        b.v_cache[slot // 256, slot % 256] = 0x7FC0
    db = DeviceBatch(lib, b, store=False)
    mtb = b.total_blocks_used
    ws = lib.decode_workspace(b.num_seqs, 8, 2, 128, mtb)
    out = torch.empty_like(db.q)
    lib.paged_decode_store_attn(out, db.q, db.k, db.v, db.slot_mapping, db.k_cache, db.v_cache,
                                db.block_tables, db.context_lens, b.scale, ws, mtb, db.status)
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle.paged_decode_attn(b.q, ekc, evc, b.block_tables, b.context_lens, b.scale)
    assert_close(out.double().cpu().numpy(), want, "fused decode")
    assert np.array_equal(bits(db.k_cache), ekc) and np.array_equal(bits(db.v_cache), evc)
