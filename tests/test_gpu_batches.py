"""Batch shapes an engine produces beyond plain decode or prefill batches:

* mixed batches: decode is the n = 1 case of prefill with a cached prefix, so
  one prefill launch serves decode rows and prompt chunks together (the
  chunked-prefill-with-decode scheduling the CSDN essay says nano-vllm lacks,
  Mountain 2);
* shared prefix blocks: reference-counted blocks (nano-vllm hub page, "core
  tech 4") let sequences point at the same physical blocks.
Both run on the unchanged kernels; results are checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import DeviceBatch, assert_close, bits, oracle_caches

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
