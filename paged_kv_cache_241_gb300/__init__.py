"""Paged KV-cache attention for GB300 (sm_103a): Python binding of libpkv.

A thin ctypes layer over the C ABI declared in include/pkv.h.  It only
marshals arguments (torch tensors -> device pointers and sizes, the current
CUDA stream) and raises on a non-OK status; every step of the computation runs
in the library's CUDA kernels.  There is no CPU fallback: if the shared library
has not been built, `load()` raises.

    import paged_kv_cache_241_gb300 as pkv
    pkv.kv_store(k, v, k_cache, v_cache, slot_mapping)
    pkv.paged_decode_attn(out, q, k_cache, v_cache, block_tables, context_lens,
                          scale, workspace, max_total_blocks)
    pkv.paged_prefill_attn(out, q, k_cache, v_cache, block_tables, cu_q, cu_k,
                           max_seqlen_q, scale)   # workspace: one per stream, cached
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
                3: "PKV_ERR_WORKSPACE", 4: "PKV_ERR_CUDA", 5: "PKV_ERR_OUT_OF_BLOCKS"}
PKV_ERR_OUT_OF_BLOCKS = 5
DEV_BAD_SLOT = 0x1
DEV_BAD_BLOCK = 0x2
DEV_BAD_CONTEXT = 0x4
DEV_TIMEOUT = 0x8
DEV_WORKSPACE = 0x10
DEV_BAD_SEQLEN = 0x20

# Exported symbols and their ctypes signatures (must match include/pkv.h).
_c_int, _c_i64, _c_sz, _c_f, _p = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                   ctypes.c_float, ctypes.c_void_p)
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [_c_int]),
    "pkv_abi_version": (_c_int, []),
    "pkv_kv_store": (_c_int, [_p, _p, _p, _p, _p, _c_i64, _c_int, _c_int, _c_i64, _c_i64, _c_i64,
                              _c_int, _p, _p]),
    "pkv_decode_workspace_size": (_c_sz, [_c_int, _c_int, _c_int, _c_int, _c_i64]),
    "pkv_paged_decode_attn": (_c_int, [_p, _p, _p, _p, _p, _p, _c_int, _c_int, _c_int, _c_int,
                                       _c_int, _c_int, _c_i64, _c_i64, _c_f, _p, _c_sz, _p, _p]),
    "pkv_paged_decode_store_attn": (_c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _c_int, _c_int,
                                             _c_int, _c_int, _c_int, _c_int, _c_i64, _c_i64, _c_f,
                                             _p, _c_sz, _p, _p]),
    "pkv_paged_decode_attn_noalloc": (_c_int, [_p, _p, _p, _p, _p, _p, _c_int, _c_int, _c_int,
                                               _c_int, _c_int, _c_int, _c_i64, _c_i64, _c_f, _p,
                                               _p]),
    "pkv_paged_prefill_attn": (_c_int, [_p, _p, _p, _p, _p, _p, _p, _c_int, _c_i64, _c_int,
                                        _c_int, _c_int, _c_int, _c_int, _c_int, _c_i64, _c_f, _p,
                                        _c_sz, _p, _p]),
    "pkv_prefill_workspace_size": (_c_sz, []),
    "pkv_test_decode_fault": (_c_int, [_c_i64, _c_int]),
    "pkv_w4a16_dequant": (_c_int, [_p, _p, _p, _c_i64, _c_i64, _c_int, _p]),
    "pkv_bm_create": (_p, [_c_int, _c_int]),
    "pkv_bm_destroy": (None, [_p]),
    "pkv_bm_num_free_blocks": (_c_int, [_p]),
    "pkv_bm_allocate": (_c_int, [_p, _c_i64, _p, _c_int, ctypes.POINTER(_c_int)]),
    "pkv_bm_append": (_c_int, [_p, _c_i64, ctypes.c_int32]),
    "pkv_bm_free": (_c_int, [_p, _c_i64]),
    "pkv_bm_num_tokens": (_c_int, [_p, _c_i64]),
    "pkv_bm_block_table": (_c_int, [_p, _c_i64, _p, _c_int]),
    "pkv_bm_slots": (_c_int, [_p, _c_i64, _c_int, _c_int, _p]),
    "pkv_bm_ref_count": (_c_int, [_p, _c_int]),
}

_lib = None


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what} failed: {STATUS_NAMES.get(status, status)}")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libpkv.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m paged_kv_cache_241_gb300.build` "
            "(the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, what: str) -> None:
    if status != PKV_OK:
        raise PkvError(status, what)


def _stream(stream) -> int:
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return int(getattr(stream, "cuda_stream", stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, ndim=None):
    import torch

    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t


def kv_store(k, v, k_cache, v_cache, slot_mapping, dev_status=None, stream=None) -> None:
    """Write new K/V rows k/v [T, Hkv, D] (bf16; rows may be strided by a
    token stride) into k_cache/v_cache [NB, BS, Hkv, D] at slot_mapping [T]."""
    import torch

    lib = load()
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(slot_mapping, torch.int32, "slot_mapping", 1)
    NB, BS, Hkv, D = k_cache.shape
    for name, t in (("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 3:
            raise ValueError(f"{name}: expected a CUDA bf16 [T, Hkv, D] tensor")
        if t.stride(2) != 1 or t.stride(1) != D or tuple(t.shape[1:]) != (Hkv, D):
            raise ValueError(f"{name}: rows must be contiguous [Hkv, D] = {(Hkv, D)}")
    st = lib.pkv_kv_store(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                          k.shape[0], Hkv, D, k.stride(0), v.stride(0), NB, BS,
                          _ptr(dev_status), _stream(stream))
    _check(st, "pkv_kv_store")


def decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_total_blocks) -> int:
    return int(load().pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                max_total_blocks))


def decode_workspace(num_seqs, num_q_heads, num_kv_heads, head_dim, max_total_blocks,
                     device="cuda"):
    """Allocate a zero-filled decode workspace (uint8, 256-byte aligned by torch)."""
    import torch

    n = decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_total_blocks)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def paged_decode_attn(out, q, k_cache, v_cache, block_tables, context_lens, scale, workspace,
                      max_total_blocks, dev_status=None, stream=None) -> None:
    """out/q [S, Hq, D] bf16; block_tables [S, max_blocks] int32; context_lens [S] int32."""
    import torch

    lib = load()
    _need(out, torch.bfloat16, "out", 3)
    _need(q, torch.bfloat16, "q", 3)
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(context_lens, torch.int32, "context_lens", 1)
    S, Hq, D = q.shape
    NB, BS, Hkv, Dc = k_cache.shape
    if Dc != D or tuple(out.shape) != (S, Hq, D) or block_tables.shape[0] != S or \
            context_lens.shape[0] != S or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("paged_decode_attn: inconsistent shapes")
    st = lib.pkv_paged_decode_attn(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(context_lens), S, Hq, Hkv, D, BS, block_tables.shape[1], NB, int(max_total_blocks),
        float(scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream))
    _check(st, "pkv_paged_decode_attn")


def paged_decode_store_attn(out, q, k, v, slot_mapping, k_cache, v_cache, block_tables,
                            context_lens, scale, workspace, max_total_blocks, dev_status=None,
                            stream=None) -> None:
    """One decode step: store k/v [S, Hkv, D] (row s = the newest token of
    sequence s) at slot_mapping [S] and attend, fused (see include/pkv.h)."""
    import torch

    lib = load()
    for name, t, dt, nd in (("out", out, torch.bfloat16, 3), ("q", q, torch.bfloat16, 3),
                            ("k", k, torch.bfloat16, 3), ("v", v, torch.bfloat16, 3),
                            ("slot_mapping", slot_mapping, torch.int32, 1),
                            ("k_cache", k_cache, torch.bfloat16, 4),
                            ("v_cache", v_cache, torch.bfloat16, 4),
                            ("block_tables", block_tables, torch.int32, 2),
                            ("context_lens", context_lens, torch.int32, 1)):
        _need(t, dt, name, nd)
    S, Hq, D = q.shape
    NB, BS, Hkv, _ = k_cache.shape
    if tuple(k.shape) != (S, Hkv, D) or tuple(v.shape) != (S, Hkv, D) or \
            slot_mapping.shape[0] != S or tuple(out.shape) != (S, Hq, D):
        raise ValueError("paged_decode_store_attn: inconsistent shapes")
    st = lib.pkv_paged_decode_store_attn(
        _ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), _ptr(context_lens), S, Hq, Hkv, D, BS, block_tables.shape[1], NB,
        int(max_total_blocks), float(scale), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    _check(st, "pkv_paged_decode_store_attn")


def paged_decode_attn_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                              max_total_blocks, dev_status=None, stream=None) -> None:
    """paged_decode_attn for callers that cannot allocate a workspace: the
    scratch is a fixed 16 MiB array inside the library (see include/pkv.h).
    Calls that overlap on the GPU must not be issued: they share that array."""
    import torch

    lib = load()
    for name, t, dt, nd in (("out", out, torch.bfloat16, 3), ("q", q, torch.bfloat16, 3),
                            ("k_cache", k_cache, torch.bfloat16, 4),
                            ("v_cache", v_cache, torch.bfloat16, 4),
                            ("block_tables", block_tables, torch.int32, 2),
                            ("context_lens", context_lens, torch.int32, 1)):
        _need(t, dt, name, nd)
    S, Hq, D = q.shape
    NB, BS, Hkv, _ = k_cache.shape
    st = lib.pkv_paged_decode_attn_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        _ptr(context_lens), S, Hq, Hkv, D, BS, block_tables.shape[1], NB, int(max_total_blocks),
        float(scale), _ptr(dev_status), _stream(stream))
    _check(st, "pkv_paged_decode_attn_noalloc")


def test_decode_fault(wait_limit_ns: int, withhold_tile: int) -> None:
    """TEST ONLY: shorten the decode kernels' wait limit on the current device
    and make every decode CTA skip loading its tile number `withhold_tile`
    (-1: none), so that a decode call times out and reports PKV_DEV_TIMEOUT.
    Restore with test_decode_fault(10**9, -1)."""
    _check(load().pkv_test_decode_fault(int(wait_limit_ns), int(withhold_tile)),
           "test_decode_fault")


def prefill_workspace(device="cuda"):
    """A zero-filled prefill workspace (the work counter the kernel's CTAs
    share; every call leaves it zeroed).  Calls that may overlap on the GPU
    need workspaces of their own."""
    import torch

    n = int(load().pkv_prefill_workspace_size())
    return torch.zeros(n, dtype=torch.uint8, device=device)


_prefill_ws = {}


def _default_prefill_workspace(device, stream):
    # One workspace per (device, stream): calls on one stream are serialised.
    key = (device.index, _stream(stream))
    ws = _prefill_ws.get(key)
    if ws is None:
        ws = _prefill_ws[key] = prefill_workspace(device)
    return ws


def paged_prefill_attn(out, q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k,
                       max_seqlen_q, scale, workspace=None, dev_status=None, stream=None) -> None:
    """out/q [T, Hq, D] bf16 packed by cu_seqlens_q; keys from the paged cache.
    workspace: from prefill_workspace(); by default one cached per stream."""
    import torch

    lib = load()
    _need(out, torch.bfloat16, "out", 3)
    _need(q, torch.bfloat16, "q", 3)
    _need(k_cache, torch.bfloat16, "k_cache", 4)
    _need(v_cache, torch.bfloat16, "v_cache", 4)
    _need(block_tables, torch.int32, "block_tables", 2)
    _need(cu_seqlens_q, torch.int32, "cu_seqlens_q", 1)
    _need(cu_seqlens_k, torch.int32, "cu_seqlens_k", 1)
    T, Hq, D = q.shape
    NB, BS, Hkv, Dc = k_cache.shape
    S = cu_seqlens_q.shape[0] - 1
    if Dc != D or tuple(out.shape) != (T, Hq, D) or block_tables.shape[0] != S or \
            cu_seqlens_k.shape[0] != S + 1 or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("paged_prefill_attn: inconsistent shapes")
    if workspace is None:
        workspace = _default_prefill_workspace(q.device, stream)
    st = lib.pkv_paged_prefill_attn(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_k), S, T, int(max_seqlen_q), Hq, Hkv, D, BS, block_tables.shape[1], NB,
        float(scale), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream))
    _check(st, "pkv_paged_prefill_attn")


def w4a16_dequant(out, packed, scales, group_size=128, stream=None) -> None:
    """out [N, K] bf16 <- packed [N, K/8] int32 (eight 4-bit values per word,
    lowest nibble first, value = nibble - 8) times scales [N, K/128] bf16."""
    import torch

    lib = load()
    _need(out, torch.bfloat16, "out", 2)
    _need(packed, torch.int32, "packed", 2)
    _need(scales, torch.bfloat16, "scales", 2)
    N, K = out.shape
    if tuple(packed.shape) != (N, K // 8) or tuple(scales.shape) != (N, K // group_size):
        raise ValueError("w4a16_dequant: inconsistent shapes")
    st = lib.pkv_w4a16_dequant(_ptr(out), _ptr(packed), _ptr(scales), N, K, int(group_size),
                               _stream(stream))
    _check(st, "pkv_w4a16_dequant")


class BlockManager:
    """Host allocator of the cache's blocks with reference counts and
    hash-chained prefix sharing (the library's pkv_bm_* calls; no GPU work).

        bm = BlockManager(num_blocks, block_size=256)
        cached = bm.allocate(seq_id, prompt_tokens)   # leading tokens already in reused blocks
        slots = bm.slots(seq_id, cached, len(prompt_tokens) - cached)
        row = bm.block_table(seq_id, max_blocks)
        bm.append(seq_id, token); bm.free(seq_id)
    """

    def __init__(self, num_blocks: int, block_size: int = 256):
        self._lib = load()
        self._h = self._lib.pkv_bm_create(int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError("BlockManager: bad sizes or out of host memory")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_bm_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    @property
    def num_free_blocks(self) -> int:
        return int(self._lib.pkv_bm_num_free_blocks(self._h))

    def allocate(self, seq_id: int, tokens) -> int:
        import numpy as np

        t = np.ascontiguousarray(tokens, dtype=np.int32)
        cached = ctypes.c_int(0)
        _check(self._lib.pkv_bm_allocate(self._h, int(seq_id), t.ctypes.data, int(t.size),
                                         ctypes.byref(cached)), "pkv_bm_allocate")
        return int(cached.value)

    def append(self, seq_id: int, token: int) -> None:
        _check(self._lib.pkv_bm_append(self._h, int(seq_id), int(token)), "pkv_bm_append")

    def free(self, seq_id: int) -> None:
        _check(self._lib.pkv_bm_free(self._h, int(seq_id)), "pkv_bm_free")

    def num_tokens(self, seq_id: int) -> int:
        return int(self._lib.pkv_bm_num_tokens(self._h, int(seq_id)))

    def block_table(self, seq_id: int, max_blocks: int):
        import numpy as np

        out = np.empty(int(max_blocks), dtype=np.int32)
        n = self._lib.pkv_bm_block_table(self._h, int(seq_id), out.ctypes.data, int(max_blocks))
        if n < 0:
            raise KeyError(seq_id)
        return out

    def slots(self, seq_id: int, first: int, count: int):
        import numpy as np

        out = np.empty(int(count), dtype=np.int32)
        _check(self._lib.pkv_bm_slots(self._h, int(seq_id), int(first), int(count),
                                      out.ctypes.data), "pkv_bm_slots")
        return out

    def ref_count(self, block: int) -> int:
        return int(self._lib.pkv_bm_ref_count(self._h, int(block)))
