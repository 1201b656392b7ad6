"""Batch shapes an engine produces beyond plain decode or prefill batches:

* mixed batches: decode is the n = 1 case of prefill with a cached prefix, so
  one prefill launch serves decode rows and prompt chunks together (the
  chunked-prefill-with-decode scheduling the CSDN essay says nano-vllm lacks,
  Mountain 2);
* shared prefix blocks: reference-counted blocks (nano-vllm hub page, "core
  tech 4") let sequences point at the same physical blocks, here also as
  handed out by the library's block manager (prefix caching).
All run on the unchanged kernels; results are checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import (DeviceBatch, assert_close, bf16, bits, i32, oracle_caches,
                      oracle_prefill_all_rows)

pytestmark = pytest.mark.gpu


def test_mixed_decode_rows_and_prompt_chunks_in_one_prefill_launch(lib):
    cached = [1500, 0, 700, 256, 3000, 40]
    new = [1, 333, 1, 129, 1, 64]  # three decode rows, three prompt chunks
    b = wl.build_batch("mixed", "prefill", 71, cached, new, 16, 8, 128)
    db = DeviceBatch(lib, b)
    out = db.prefill()
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle.paged_prefill_attn(b.q, ekc, evc, b.block_tables, b.cu_seqlens_q,
                                     b.cu_seqlens_k, b.scale)
    assert_close(out.double().cpu().numpy(), want, "mixed batch")
    # the decode rows agree with the decode kernel on the same cache
    rows = np.array([int(b.cu_seqlens_q[s]) for s in (0, 2, 4)])
    dec_seqs = [0, 2, 4]
    q_dec = db.q[torch.as_tensor(rows, device="cuda")].contiguous()
    bt = db.block_tables[torch.as_tensor(dec_seqs, device="cuda")].contiguous()
    cl = db.context_lens[torch.as_tensor(dec_seqs, device="cuda")].contiguous()
    mtb = sum(wl.blocks_for(int(b.context_lens[s])) for s in dec_seqs)
    ws = lib.decode_workspace(3, 16, 8, 128, mtb)
    dec = torch.empty_like(q_dec)
    lib.paged_decode_attn(dec, q_dec, db.k_cache, db.v_cache, bt, cl, b.scale, ws, mtb, db.status)
    assert db.status_value() == 0
    d = dec.double().cpu().numpy()
    assert np.all(np.abs(out.double().cpu().numpy()[rows] - d) <= 2 * (8e-3 + 1e-2 * np.abs(d)))


def test_mixed_workload_full_size_every_row(lib):
    # The benchmark's mixed step: 48 decode rows (contexts U[128, 2048]) and 8
    # prompt chunks (U[256, 1024] new after U[0, 2048] cached) in one launch.
    b = wl.mixed()
    db = DeviceBatch(lib, b)
    out = db.prefill()
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle_prefill_all_rows(b, ekc, evc)
    assert not np.isnan(want).any()
    assert_close(out.double().cpu().numpy(), want, "mixed step, every row")


def shared_prefix_batch(kind, seed, cached, new):
    """Sequences 1.. reuse sequence 0's first two physical blocks (a common
    512-token prefix): their block tables point at the same block ids."""
    b = wl.build_batch("shared", kind, seed, cached, new, 8, 2, 128, num_blocks=64)
    for s in range(1, b.num_seqs):
        b.block_tables[s, :2] = b.block_tables[0, :2]
    # slots of new tokens never fall in the shared blocks (all contexts > 512)
    assert all(int(c) >= 512 for c in b.cached_lens)
    return b


def test_decode_over_shared_prefix_blocks(lib):
    b = shared_prefix_batch("decode", 72, [600, 900, 1300], [1, 1, 1])
    b.slot_mapping[:] = [oracle.slot_of(b.block_tables[s], int(b.cached_lens[s]), 256)
                         for s in range(3)]
    db = DeviceBatch(lib, b)
    out = db.decode()
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle.paged_decode_attn(b.q, ekc, evc, b.block_tables, b.context_lens, b.scale)
    assert_close(out.double().cpu().numpy(), want, "decode, shared prefix")


def test_prefill_over_shared_prefix_blocks(lib):
    b = shared_prefix_batch("prefill", 73, [512, 512, 700], [100, 257, 64])
    t = 0
    for s in range(b.num_seqs):
        for i in range(int(b.new_lens[s])):
            b.slot_mapping[t] = oracle.slot_of(b.block_tables[s], int(b.cached_lens[s]) + i, 256)
            t += 1
    db = DeviceBatch(lib, b)
    out = db.prefill()
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle.paged_prefill_attn(b.q, ekc, evc, b.block_tables, b.cu_seqlens_q,
                                     b.cu_seqlens_k, b.scale)
    assert_close(out.double().cpu().numpy(), want, "prefill, shared prefix")


def _kv_of(tokens, positions, table):
    # K/V of a token as a fixed function of (token id, position): identical
    # prompt prefixes give identical K/V, as a model's would
    idx = (tokens.astype(np.int64) * 2654435761 + positions.astype(np.int64) * 40503) % len(table)
    return table[idx]


def test_block_manager_prefix_sharing_end_to_end(lib):
    Hq, Hkv, D, bs, NB = 8, 4, 128, 256, 24
    rng = np.random.default_rng(90)
    ktab = wl.normal_bf16(rng, (4099, Hkv, D))
    vtab = wl.normal_bf16(rng, (4099, Hkv, D))
    a = rng.integers(0, 50000, size=700).astype(np.int32)
    prompts = [a,
               np.concatenate([a[:512], rng.integers(0, 50000, 288)]).astype(np.int32),
               np.concatenate([a[:256], rng.integers(0, 50000, 44)]).astype(np.int32),
               rng.integers(0, 50000, size=70).astype(np.int32)]
    bm = lib.BlockManager(NB, bs)
    cached = [bm.allocate(i, p) for i, p in enumerate(prompts)]
    assert cached == [0, 512, 256, 0]
    new = [len(p) - c for p, c in zip(prompts, cached)]
    maxb = 4
    tables = np.stack([bm.block_table(i, maxb) for i in range(4)])
    # only the uncached tokens are stored
    slots = np.concatenate([bm.slots(i, c, n) for i, (c, n) in enumerate(zip(cached, new))])
    toks = np.concatenate([p[c:] for p, c in zip(prompts, cached)])
    pos = np.concatenate([np.arange(c, len(p)) for p, c in zip(prompts, cached)])
    k_new, v_new = _kv_of(toks, pos, ktab), _kv_of(toks, pos, vtab)
    stale = np.full((NB, bs, Hkv, D), wl.BF16_QNAN, dtype=np.uint16)
    q = wl.normal_bf16(rng, (sum(new), Hq, D))
    cu_q = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum([len(p) for p in prompts])]).astype(np.int32)
    scale = 1.0 / np.sqrt(D)

    kc, vc = bf16(stale), bf16(stale)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.kv_store(bf16(k_new), bf16(v_new), kc, vc, i32(slots), status)
    out = torch.empty((sum(new), Hq, D), dtype=torch.bfloat16, device="cuda")
    lib.paged_prefill_attn(out, bf16(q), kc, vc, i32(tables), i32(cu_q), i32(cu_k), max(new),
                           scale, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    ekc, evc = oracle.kv_store(stale, stale, k_new, v_new, slots)
    want = oracle.paged_prefill_attn(q, ekc, evc, tables, cu_q, cu_k, scale)
    # what prefix caching must preserve: the same result as attending over
    # each sequence's whole prompt, its K/V computed afresh
    for s, (p, c) in enumerate(zip(prompts, cached)):
        kf = oracle.bf16_bits_to_f64(_kv_of(p, np.arange(len(p)), ktab))
        vf = oracle.bf16_bits_to_f64(_kv_of(p, np.arange(len(p)), vtab))
        qf = oracle.bf16_bits_to_f64(q[cu_q[s]:cu_q[s + 1]])
        for i in (0, new[s] - 1):
            for h in (0, Hq - 1):
                j = oracle.kv_head_of(h, Hq, Hkv)
                ref = oracle.attend(qf[i, h], kf[: c + i + 1, j], vf[: c + i + 1, j], scale)
                assert np.allclose(want[cu_q[s] + i, h], ref, rtol=1e-12, atol=1e-12)
    assert_close(out.double().cpu().numpy(), want, "prefill over shared prefix blocks")

    # one decode step per sequence on top of the shared blocks
    nxt = rng.integers(0, 50000, size=4).astype(np.int32)
    for i, t in enumerate(nxt):
        bm.append(i, int(t))
    lens = np.array([bm.num_tokens(i) for i in range(4)], dtype=np.int32)
    tables = np.stack([bm.block_table(i, maxb) for i in range(4)])
    slots1 = np.concatenate([bm.slots(i, int(L) - 1, 1) for i, L in enumerate(lens)])
    k1, v1 = _kv_of(nxt, lens - 1, ktab), _kv_of(nxt, lens - 1, vtab)
    q1 = wl.normal_bf16(rng, (4, Hq, D))
    lib.kv_store(bf16(k1), bf16(v1), kc, vc, i32(slots1), status)
    ws = lib.decode_workspace(4, Hq, Hkv, D, 16)
    dec = torch.empty((4, Hq, D), dtype=torch.bfloat16, device="cuda")
    lib.paged_decode_attn(dec, bf16(q1), kc, vc, i32(tables), i32(lens), scale, ws, 16, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ekc, evc = oracle.kv_store(ekc, evc, k1, v1, slots1)
    want1 = oracle.paged_decode_attn(q1, ekc, evc, tables, lens, scale)
    assert_close(dec.double().cpu().numpy(), want1, "decode over shared prefix blocks")
