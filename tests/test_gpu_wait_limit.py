"""A bounded wait that runs out, on the GPU, without a fault or a hang.

Every wait inside the kernels gives up after a wall-clock limit, flags
PKV_DEV_TIMEOUT in the caller's status word and unwinds (the roles stop
together, copies in flight are waited for, tensor memory is freed).  Here the
decode producer is told to skip one tile, which nothing else will ever
deliver, with the limit cut to 2 ms: the call must come back with the flag set,
and the next call on the same stream must be correct."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import DeviceBatch, assert_close, oracle_caches

pytestmark = pytest.mark.gpu


def few_items(G):
    # fewer items than CTAs: items taken round-robin
    return wl.build_batch("limit", "decode", 90 + G, [4, 299, 700], [1, 1, 1], 2 * G, 2, 64,
                          num_blocks=12)


def many_items(G):
    # ~14K items: handed out by the workspace counter, which must be left at
    # zero even by a call whose waits ran out
    rng = np.random.default_rng(95 + G)
    L = rng.integers(3000, 4000, size=128, endpoint=True)
    return wl.build_batch("limit", "decode", 95 + G, L - 1, np.ones(128, np.int64), 2 * G, 2, 64,
                          block_size=64, rng=rng)


def two_block_items(G):
    # ~20K one-block items over 160 sequences and 4 kv heads: the kernel's
    # two-block form, items of two blocks handed out by the counter
    rng = np.random.default_rng(97 + G)
    L = rng.integers(1500, 2500, size=160, endpoint=True)
    return wl.build_batch("limit", "decode", 97 + G, L - 1, np.ones(160, np.int64), 4 * G, 4, 64,
                          block_size=64, rng=rng)


@pytest.mark.parametrize("make", [few_items, many_items, two_block_items])
@pytest.mark.parametrize("G", [2, 4])  # 4-stage ring (TMA + cp.async) and 3-stage ring (TMA)
def test_decode_wait_runs_out_then_next_call_is_correct(lib, G, make):
    b = make(G)
    db = DeviceBatch(lib, b)
    mtb = b.total_blocks_used
    ws = lib.decode_workspace(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim, mtb)
    out = torch.empty((b.num_seqs, b.num_q_heads, b.head_dim), dtype=torch.bfloat16, device="cuda")
    try:
        lib.test_decode_fault(2_000_000, 1)  # 2 ms limit; each CTA's second tile never loads
        lib.paged_decode_attn(out, db.q, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                              b.scale, ws, mtb, db.status)
        torch.cuda.synchronize()
    finally:
        lib.test_decode_fault(1_000_000_000, -1)
    assert db.status_value() & lib.DEV_TIMEOUT
    assert int(ws[:256].count_nonzero().item()) == 0  # the work counter is left at zero
    db.status.zero_()
    lib.paged_decode_attn(out, db.q, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                          b.scale, ws, mtb, db.status)
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle.paged_decode_attn(b.q, ekc, evc, b.block_tables, b.context_lens, b.scale)
    assert_close(out.double().cpu().numpy(), want, "decode after a timed-out call")
