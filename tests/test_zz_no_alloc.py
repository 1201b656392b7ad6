"""The allocation-free decode entry point, checked against the regular one.

pkv_paged_decode_attn_noalloc exists for callers that cannot give this library
a device workspace: code under a framework whose allocator owns all device
memory, plugins that may not allocate in their host process, or serving loops
that keep cudaMalloc/cudaFree (which synchronise the device) off their latency
path.  Its scratch is a fixed array inside the library, shared by every call,
so two calls in a row must both give the regular entry point's result (the
second one finds the first one's leftovers in the array).

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import workloads as wl
from gpu_util import DeviceBatch, assert_close

pytestmark = pytest.mark.gpu


def call_noalloc(c, out, db, max_total_blocks):
    b = db.b
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    return c.pkv_paged_decode_attn_noalloc(
        ptr(out), ptr(db.q), ptr(db.k_cache), ptr(db.v_cache), ptr(db.block_tables),
        ptr(db.context_lens), b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim,
        b.block_size, b.block_tables.shape[1], b.num_blocks, max_total_blocks, b.scale,
        ptr(db.status), torch.cuda.current_stream().cuda_stream)


def test_no_alloc_decode_matches_workspace_decode_twice(lib):
    lens = [1, 200, 256, 257, 1000, 2048, 3000, 513]
    b = wl.build_batch("noalloc", "decode", 77, [L - 1 for L in lens], [1] * len(lens), 16, 8,
                       128, max_blocks_pad=1)
    db = DeviceBatch(lib, b)
    ref = db.decode().double().cpu().numpy()  # regular entry point, torch workspace
    c = lib.load()
    for call in range(2):
        out = torch.full((b.num_seqs, b.num_q_heads, b.head_dim), float("nan"),
                         dtype=torch.bfloat16, device="cuda")
        assert call_noalloc(c, out, db, b.total_blocks_used) == lib.PKV_OK
        torch.cuda.synchronize()
        assert_close(out.double().cpu().numpy(), ref, f"no-alloc decode, call {call}")
    assert db.status_value() == 0


def test_no_alloc_rejects_sizes_beyond_its_scratch(lib):
    b = wl.build_batch("big", "decode", 78, [99], [1], 16, 8, 128)
    db = DeviceBatch(lib, b)
    c = lib.load()
    out = torch.empty((1, 16, 128), dtype=torch.bfloat16, device="cuda")
    # 16 MiB cannot hold the partials of 10,000 blocks x 16 heads x 128 dims
    assert call_noalloc(c, out, db, 10_000) == 3  # PKV_ERR_WORKSPACE, nothing launched
