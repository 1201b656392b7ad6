"""Paged varlen causal prefill on the GPU (tcgen05 path) against the fp64 oracle.

Tolerance: |gpu - oracle| <= 8e-3 + 1e-2 |oracle| elementwise."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import DeviceBatch, assert_close, bits, oracle_caches, oracle_prefill_all_rows

pytestmark = pytest.mark.gpu


def check_prefill(lib, b, rows=None):
    db = DeviceBatch(lib, b)
    out = db.prefill()
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle.paged_prefill_attn(b.q, ekc, evc, b.block_tables, b.cu_seqlens_q,
                                     b.cu_seqlens_k, b.scale, rows=rows)
    got = out.double().cpu().numpy()
    sel = slice(None) if rows is None else rows
    assert_close(got[sel], want[sel], f"prefill {b.name}")
    return db, out


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_prefill_varlen_with_prefix_small(lib, D, G):
    cached = [0, 256, 0, 512, 3, 0, 100]
    new = [1, 64, 127, 128, 129, 300, 200]
    b = wl.build_batch("small", "prefill", 50 + D + G, cached, new, 2 * G, 2, D,
                       max_blocks_pad=2)
    check_prefill(lib, b)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_prefill_single_row_units(lib, D, G):
    # Units with one query row (decode rows of a mixed batch; the one-row tail
    # of a 129- or 257-token prompt), contexts across the tile (64-key) and
    # block (256-key) boundaries, with stale NaN in every slot past a context:
    # one valid row in a 128-row MMA tile.
    cached = [0, 15, 16, 17, 63, 64, 65, 255, 256, 257, 1000, 2047, 0, 300]
    new = [1] * 12 + [129, 257]
    b = wl.build_batch("rows1", "prefill", 80 + D + G, cached, new, 2 * G, 2, D, stale="nan")
    db, out = check_prefill(lib, b)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [2, 4, 8])
def test_prefill_packed_tiles(lib, D, G):
    # A decode-heavy batch (mean new tokens per sequence <= 128) runs the
    # packing kernel: tiles with at most 64 valid rows hold both heads of a
    # pair, 64 rows each.  Tails of 1, 31, 32, 33, 63, 64 and 65 rows (the
    # packing limit and the warp boundaries), short prompts, decode rows and
    # full tiles in one launch, over cached prefixes, NaN in stale slots.
    new = [1] * 24 + [129, 159, 160, 161, 191, 192, 193, 64, 65, 33, 256]
    cached = [(37 * i) % 700 for i in range(len(new))]
    b = wl.build_batch("packed", "prefill", 110 + D + G, cached, new, 2 * G, 2, D, stale="nan")
    assert b.q.shape[0] <= 128 * b.num_seqs and max(new) <= 1024
    db, out = check_prefill(lib, b)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("scale", [0.0, -1.0 / np.sqrt(128.0)])
@pytest.mark.parametrize("form", ["short", "long", "packed"])
def test_prefill_zero_and_negative_scale(lib, scale, form):
    # softmax(q K^T * scale) is defined for any scale.  A negative scale makes
    # a row's largest scaled logit come from its smallest q.k (the kernel's
    # minimum path instead of the load-with-max); zero gives the mean of the
    # row's visible values.  Each batch selects one kernel form: short
    # prompts (one MMA issuer per head), long prompts (the S / P.V issuer
    # pair) and a decode-heavy batch (packed tiles); all cross the causal
    # diagonal over cached prefixes, with ragged tails and NaN in stale slots.
    cached, new = {"short": ([0, 256, 70], [300, 129, 64]),
                   "long": ([0, 300], [1100, 1300]),
                   "packed": ([5, 400, 0, 77, 1000, 256], [1, 1, 65, 1, 33, 129])}[form]
    b = wl.build_batch("scale", "prefill", 91, cached, new, 4, 2, 128, stale="nan")
    b = dataclasses.replace(b, scale=float(scale))
    db, out = check_prefill(lib, b)
    assert torch.isfinite(out.float()).all()


def test_prefill_single_row_of_context_one_returns_v_bits(lib):
    b = wl.build_batch("one1", "prefill", 79, [0, 0, 0], [1, 1, 1], 8, 4, 128)
    db = DeviceBatch(lib, b)
    out = bits(db.prefill())
    for s in range(3):
        for h in range(8):
            assert np.array_equal(out[s, h], b.v[s, h // 2])


def test_prefill_single_tile_prompts_d128(lib):
    # every prompt fits one 128-row query tile, some with long cached prefixes
    b = wl.build_batch("onetile", "prefill", 66, [0, 300, 1000, 0], [1, 77, 128, 128], 16, 8, 128)
    check_prefill(lib, b)


@pytest.mark.parametrize("new", [[129], [256], [257], [383, 40], [640, 1, 129]])
def test_prefill_tile_counts(lib, new):
    # query tile counts 2, 2, 3, (3, 1), (5, 1, 2): ragged last tiles, one- and
    # many-tile prompts in one launch, cached prefixes of 0, 256 and 512 keys
    cached = [256 * (i % 3) for i in range(len(new))]
    b = wl.build_batch("tiles", "prefill", 67 + sum(new), cached, new, 8, 4, 128)
    check_prefill(lib, b)


def test_prefill_single_long_prompt(lib):
    b = wl.build_batch("long", "prefill", 60, [0], [1500], 4, 2, 128)
    check_prefill(lib, b)


@pytest.mark.parametrize("bs", [64, 128, 512])
def test_prefill_other_block_sizes(lib, bs):
    b = wl.build_batch("bs", "prefill", 61 + bs, [0, bs, 2 * bs + 7], [200, 70, 129], 4, 2, 128,
                       block_size=bs)
    check_prefill(lib, b)


def test_prefill_never_reads_stale_slots(lib):
    b = wl.build_batch("nan", "prefill", 62, [0, 256, 5], [100, 37, 300], 4, 2, 128, stale="nan")
    db, out = check_prefill(lib, b)
    assert torch.isfinite(out.float()).all()


def test_prefill_first_row_returns_first_value(lib):
    b = wl.build_batch("first", "prefill", 63, [0, 0], [130, 7], 4, 2, 128)
    db = DeviceBatch(lib, b)
    out = bits(db.prefill())
    for s, row in enumerate(b.cu_seqlens_q[:-1]):
        for h in range(4):
            assert np.array_equal(out[row, h], b.v[row, h // 2])


def test_prefill_last_row_matches_decode(lib):
    b = wl.build_batch("pd", "prefill", 64, [0, 256, 40], [300, 90, 1], 8, 2, 128)
    db = DeviceBatch(lib, b)
    pre = db.prefill().double().cpu().numpy()
    last = b.cu_seqlens_q[1:] - 1
    q_last = db.q[torch.as_tensor(last, dtype=torch.long, device="cuda")].contiguous()
    ws = lib.decode_workspace(b.num_seqs, 8, 2, 128, b.total_blocks_used)
    dec = torch.empty_like(q_last)
    lib.paged_decode_attn(dec, q_last, db.k_cache, db.v_cache, db.block_tables, db.context_lens,
                          b.scale, ws, b.total_blocks_used, db.status)
    assert db.status_value() == 0
    # both are within tolerance of the same oracle value: within twice of each other
    d = dec.double().cpu().numpy()
    assert np.all(np.abs(pre[last] - d) <= 2 * (8e-3 + 1e-2 * np.abs(d)))


def check_every_row(lib, b):
    """Every query row and head of a full-size workload against the oracle."""
    db = DeviceBatch(lib, b)
    out = db.prefill()
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle_prefill_all_rows(b, ekc, evc)
    assert not np.isnan(want).any()
    assert_close(out.double().cpu().numpy(), want, f"prefill {b.name}, every row")


def test_prefill_full_size_every_row(lib):
    # 16 prompts, U[64, 4096] tokens (41K query rows), 16 q / 8 kv heads, D 128
    check_every_row(lib, wl.prefill())


def test_prefix_cached_full_size_every_row(lib):
    # 32 sequences, k*256 cached (k in {0,1,2,4}) + U[1, 512] new tokens
    check_every_row(lib, wl.prefix())


def test_prefill_flags_inconsistent_seqlens(lib):
    b = wl.build_batch("bad", "prefill", 65, [0, 0], [50, 60], 4, 2, 128)
    db = DeviceBatch(lib, b)
    db.cu_k[2] = db.cu_k[1] + 10  # second sequence: fewer keys than queries
    db.prefill()
    assert db.status_value() & lib.DEV_BAD_SEQLEN


def test_prefill_workspace_is_left_zeroed_and_reusable(lib):
    # the CTAs take units from a counter in the workspace; each call must leave
    # it zeroed so the next call (same workspace) starts from unit 0
    b = wl.build_batch("ws", "prefill", 68, [0, 256, 0], [700, 90, 3], 8, 4, 128)
    db = DeviceBatch(lib, b)
    ws = lib.prefill_workspace()
    ekc, evc = oracle_caches(b)
    want = oracle.paged_prefill_attn(b.q, ekc, evc, b.block_tables, b.cu_seqlens_q,
                                     b.cu_seqlens_k, b.scale)
    for _ in range(3):
        out = torch.full((b.q.shape[0], b.num_q_heads, b.head_dim), float("nan"),
                         dtype=torch.bfloat16, device="cuda")
        lib.paged_prefill_attn(out, db.q, db.k_cache, db.v_cache, db.block_tables, db.cu_q,
                               db.cu_k, int(b.new_lens.max()), b.scale, workspace=ws,
                               dev_status=db.status)
        torch.cuda.synchronize()
        assert int(ws.count_nonzero().item()) == 0
        assert_close(out.double().cpu().numpy(), want, "prefill, reused workspace")
    assert db.status_value() == 0


def test_prefill_output_only_16_byte_aligned(lib):
    # rows are written with 32-byte stores when `out` allows it; an `out` that
    # is 16- but not 32-byte aligned takes the 16-byte store path
    b = wl.build_batch("align", "prefill", 69, [0, 256], [300, 45], 8, 4, 128)
    db = DeviceBatch(lib, b)
    T, Hq, D = b.q.shape[0], b.num_q_heads, b.head_dim
    buf = torch.zeros(T * Hq * D + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(T, Hq, D)
    assert out.data_ptr() % 32 == 16
    lib.paged_prefill_attn(out, db.q, db.k_cache, db.v_cache, db.block_tables, db.cu_q, db.cu_k,
                           int(b.new_lens.max()), b.scale, dev_status=db.status)
    assert db.status_value() == 0
    ekc, evc = oracle_caches(b)
    want = oracle.paged_prefill_attn(b.q, ekc, evc, b.block_tables, b.cu_seqlens_q,
                                     b.cu_seqlens_k, b.scale)
    assert_close(out.double().cpu().numpy(), want, "prefill, 16-byte aligned out")
    assert torch.count_nonzero(buf[:8]) == 0


@pytest.mark.parametrize("num_seqs", [256, 257])
@pytest.mark.parametrize("D,G", [(128, 2), (64, 1)])
def test_prefill_many_sequences(lib, num_seqs, D, G):
    # Up to 256 sequences the kernel orders them longest context first (sorted
    # in shared memory); beyond that it keeps their given order.  Both paths,
    # with many equal lengths (ties keep their index order) and one-token
    # prompts, for two heads per CTA (D 128) and one (D 64).
    rng = np.random.default_rng(70 + num_seqs)
    new = [int(x) for x in rng.choice([1, 7, 40, 130], size=num_seqs)]
    cached = [int(x) for x in rng.choice([0, 0, 256, 300], size=num_seqs)]
    b = wl.build_batch("many", "prefill", 70 + num_seqs + D, cached, new, 2 * G, 2, D)
    check_prefill(lib, b)


def test_prefill_sequence_order_keeps_results(lib):
    # The same sequences given in another order give the same rows, bit for
    # bit: the processing order is a schedule, not part of the result.
    cached = [0, 1024, 256, 0, 512, 0]
    new = [300, 20, 129, 1, 64, 900]
    b = wl.build_batch("order", "prefill", 71, cached, new, 8, 4, 128)
    db, out = check_prefill(lib, b)
    perm = [5, 2, 0, 4, 1, 3]
    starts = b.cu_seqlens_q[:-1]
    rows = torch.as_tensor(np.concatenate([np.arange(starts[s], starts[s] + new[s]) for s in perm]),
                           device="cuda")
    q2 = db.q[rows].contiguous()
    bt2 = db.block_tables[torch.as_tensor(perm, device="cuda")].contiguous()
    cu_q2 = torch.as_tensor(np.concatenate([[0], np.cumsum([new[s] for s in perm])]),
                            dtype=torch.int32, device="cuda")
    cu_k2 = torch.as_tensor(np.concatenate([[0], np.cumsum([new[s] + cached[s] for s in perm])]),
                            dtype=torch.int32, device="cuda")
    out2 = torch.empty_like(out)
    lib.paged_prefill_attn(out2, q2, db.k_cache, db.v_cache, bt2, cu_q2, cu_k2, max(new), b.scale,
                           dev_status=db.status)
    torch.cuda.synchronize()
    assert db.status_value() == 0
    assert torch.equal(out2, out[rows])


def test_prefill_sequence_without_new_tokens_is_skipped(lib):
    # A sequence with cached context but no new tokens (empty query range)
    # has no units; it still sorts among the others by its context length.
    # The other sequences' rows equal those of the batch that includes it.
    cached = [0, 2048, 256, 0]
    new = [200, 64, 129, 40]
    b = wl.build_batch("empty", "prefill", 72, cached, new, 8, 4, 128)
    db, out = check_prefill(lib, b)
    keep = [0, 2, 3]
    starts = b.cu_seqlens_q[:-1]
    rows = torch.as_tensor(np.concatenate([np.arange(starts[s], starts[s] + new[s]) for s in keep]),
                           device="cuda")
    q2 = db.q[rows].contiguous()
    n2 = [new[0], 0, new[2], new[3]]  # sequence 1 keeps its cached keys, loses its queries
    k2 = [new[0], cached[1], cached[2] + new[2], new[3]]
    cu_q2 = torch.as_tensor(np.concatenate([[0], np.cumsum(n2)]), dtype=torch.int32, device="cuda")
    cu_k2 = torch.as_tensor(np.concatenate([[0], np.cumsum(k2)]), dtype=torch.int32, device="cuda")
    out2 = torch.empty((len(rows), b.num_q_heads, b.head_dim), dtype=torch.bfloat16, device="cuda")
    lib.paged_prefill_attn(out2, q2, db.k_cache, db.v_cache, db.block_tables, cu_q2, cu_k2,
                           max(n2), b.scale, dev_status=db.status)
    torch.cuda.synchronize()
    assert db.status_value() == 0
    assert torch.equal(out2, out[rows])
