"""Helpers for the GPU parity tests: move a workloads.PagedBatch to the device,
run the library's calls on it, and compare with the oracle."""
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
