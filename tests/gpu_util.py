"""Helpers for the GPU parity tests: move a workloads.PagedBatch to the device,
run the library's calls on it, and compare with the oracle."""
import os

import numpy as np
import torch

import oracle

ATOL = 8e-3  # |gpu - oracle| <= ATOL + RTOL * |oracle|, elementwise (bf16 in, fp32 accumulate)
RTOL = 1e-2


def bf16(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def i32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def assert_close(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want)
    bound = ATOL + RTOL * np.abs(want)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; "
                             f"worst at {i}: got {got[i]!r} want {want[i]!r}")


class DeviceBatch:
    """A PagedBatch on the GPU, with its cache already updated by kv_store."""

    def __init__(self, pkv, b, dev="cuda", store=True):
        self.pkv, self.b = pkv, b
        self.k_cache = bf16(b.k_cache, dev)
        self.v_cache = bf16(b.v_cache, dev)
        self.q = bf16(b.q, dev)
        self.k = bf16(b.k, dev)
        self.v = bf16(b.v, dev)
        self.slot_mapping = i32(b.slot_mapping, dev)
        self.block_tables = i32(b.block_tables, dev)
        self.context_lens = i32(b.context_lens, dev)
        self.cu_q = i32(b.cu_seqlens_q, dev)
        self.cu_k = i32(b.cu_seqlens_k, dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.dev = dev
        if store:
            pkv.kv_store(self.k, self.v, self.k_cache, self.v_cache, self.slot_mapping,
                         self.status)

    def decode(self, max_total_blocks=None):
        b = self.b
        mtb = b.total_blocks_used if max_total_blocks is None else max_total_blocks
        ws = self.pkv.decode_workspace(b.num_seqs, b.num_q_heads, b.num_kv_heads, b.head_dim,
                                       mtb, self.dev)
        out = torch.empty((b.num_seqs, b.num_q_heads, b.head_dim), dtype=torch.bfloat16,
                          device=self.dev)
        self.pkv.paged_decode_attn(out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                   self.context_lens, b.scale, ws, mtb, self.status)
        return out

    def prefill(self):
        b = self.b
        out = torch.empty((b.q.shape[0], b.num_q_heads, b.head_dim), dtype=torch.bfloat16,
                          device=self.dev)
        self.pkv.paged_prefill_attn(out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                    self.cu_q, self.cu_k, int(b.new_lens.max()), b.scale,
                                    dev_status=self.status)
        return out

    def status_value(self):
        torch.cuda.synchronize()
        return int(self.status.item())


def oracle_caches(b):
    return oracle.kv_store(b.k_cache, b.v_cache, b.k, b.v, b.slot_mapping)


# ------------------------------------------- oracle over whole workloads, in parallel
#
# The full-size parity tests compare every output row.  The oracle is a plain
# per-row loop, so its rows are computed in a pool of worker processes (spawn:
# a forked child of a process that already holds a CUDA context can hang).
# Each task is one sequence (or a slice of a long one's rows) passed to the
# unchanged oracle as a batch of that one sequence.

_POOL_STATE = {}


def _pool_init(k_cache, v_cache, scale):
    _POOL_STATE["kc"], _POOL_STATE["vc"], _POOL_STATE["scale"] = k_cache, v_cache, scale


def _prefill_task(args):
    q_seq, bt_row, n, len_k, r0, r1 = args
    out = oracle.paged_prefill_attn(q_seq, _POOL_STATE["kc"], _POOL_STATE["vc"], bt_row[None, :],
                                    np.array([0, n], np.int32), np.array([0, len_k], np.int32),
                                    _POOL_STATE["scale"], rows=np.arange(r0, r1))
    return out[r0:r1]


_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _workers():
    return max(1, min(16, os.cpu_count() or 1))


def oracle_prefill_all_rows(b, ekc, evc, chunk=256):
    """The oracle's output for every query row of prefill batch `b` (caches
    `ekc`/`evc` after the store), float64 [T_q, Hq, D]."""
    import multiprocessing as mp

    cu_q, cu_k = b.cu_seqlens_q, b.cu_seqlens_k
    tasks, where = [], []
    for s in range(b.num_seqs):
        q0, q1 = int(cu_q[s]), int(cu_q[s + 1])
        n, len_k = q1 - q0, int(cu_k[s + 1] - cu_k[s])
        for r0 in range(0, n, chunk):
            r1 = min(n, r0 + chunk)
            tasks.append((b.q[q0:q1], b.block_tables[s], n, len_k, r0, r1))
            where.append((q0 + r0, q0 + r1))
    out = np.full((b.q.shape[0], b.num_q_heads, b.head_dim), np.nan)
    # the longest tasks (latest rows of the longest keys) first
    order = sorted(range(len(tasks)), key=lambda i: -(tasks[i][3] - tasks[i][2] + tasks[i][5]))
    ctx = mp.get_context("spawn")
    # one BLAS thread per worker (the children read these when numpy loads)
    saved = {v: os.environ.get(v) for v in _BLAS_VARS}
    os.environ.update({v: "1" for v in _BLAS_VARS})
    try:
        with ctx.Pool(_workers(), initializer=_pool_init, initargs=(ekc, evc, b.scale)) as pool:
            res = pool.map(_prefill_task, [tasks[i] for i in order], chunksize=1)
    finally:
        for v, x in saved.items():
            if x is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = x
    for i, r in zip(order, res):
        a, z = where[i]
        out[a:z] = r
    return out
