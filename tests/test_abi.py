"""CPU checks of the C-ABI library: it loads, exports every symbol the header
declares, and its host-side argument checks reject bad calls without launching
anything (these calls never reach the GPU)."""
import ctypes
import os
import re

import pytest

import paged_kv_cache_241_gb300 as pkv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pkv.LIB_PATH):
        from paged_kv_cache_241_gb300 import build

        build.build()
    return pkv.load()


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("pkv_kv_store", "pkv_paged_decode_attn", "pkv_paged_prefill_attn",
              "pkv_decode_workspace_size", "pkv_status_string", "pkv_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in pkv.h but not exported"
    # and the binding's signature table covers exactly the declared set
    assert sorted(pkv.SIGNATURES) == declared_functions()


def test_status_strings(lib):
    assert lib.pkv_status_string(0) == b"PKV_OK"
    assert lib.pkv_status_string(3) == b"PKV_ERR_WORKSPACE"
    assert lib.pkv_status_string(99) == b"PKV_ERR_UNKNOWN"
    assert lib.pkv_abi_version() == 3
    assert lib.pkv_status_string(5) == b"PKV_ERR_OUT_OF_BLOCKS"


def test_workspace_size_formula(lib):
    # work counter (256 bytes) + sequence prefix ((S+1) int32) + partial
    # max/sum (B*Hq*2 f32) + partial outputs (B*Hq*D f32), each rounded up to
    # 256 bytes
    up = lambda x: (x + 255) // 256 * 256
    S, Hq, Hkv, D, B = 64, 16, 8, 128, 300
    assert lib.pkv_decode_workspace_size(S, Hq, Hkv, D, B) == \
        256 + up((S + 1) * 4) + up(B * Hq * 2 * 4) + up(B * Hq * D * 4)
    assert lib.pkv_decode_workspace_size(0, Hq, Hkv, D, B) == 0
    # a block bound whose workspace would wrap a size_t has no workspace size
    assert lib.pkv_decode_workspace_size(S, Hq, Hkv, D, 1 << 62) == 0
    assert lib.pkv_decode_workspace_size(S, 1 << 20, Hkv, D, B) == 0


NULL = None


def test_kv_store_rejects_bad_arguments(lib):
    f = lib.pkv_kv_store
    # zero kv heads
    assert f(NULL, NULL, NULL, NULL, NULL, 4, 0, 128, 0, 0, 16, 256, NULL, NULL) == 1
    # row of Hkv*D not a multiple of 8 elements
    assert f(NULL, NULL, NULL, NULL, NULL, 4, 1, 12, 0, 0, 16, 256, NULL, NULL) == 2
    # null pointers with work to do
    assert f(NULL, NULL, NULL, NULL, NULL, 4, 8, 128, 0, 0, 16, 256, NULL, NULL) == 1
    # token stride shorter than a row
    assert f(NULL, NULL, NULL, NULL, NULL, 4, 8, 128, 512, 0, 16, 256, NULL, NULL) == 1
    # misaligned pointers
    p = ctypes.c_void_p(0x1002)
    assert f(p, p, p, p, p, 4, 8, 128, 0, 0, 16, 256, NULL, NULL) == 1
    # nothing to do is fine
    assert f(NULL, NULL, NULL, NULL, NULL, 0, 8, 128, 0, 0, 16, 256, NULL, NULL) == 0


def decode_call(lib, **kw):
    a = dict(out=NULL, q=NULL, kc=NULL, vc=NULL, bt=NULL, cl=NULL, S=4, Hq=16, Hkv=8, D=128,
             BS=256, maxb=8, NB=64, mtb=32, scale=0.1, ws=NULL, wsb=0, st=NULL, stream=NULL)
    a.update(kw)
    return lib.pkv_paged_decode_attn(*a.values())


def test_decode_rejects_bad_arguments(lib):
    assert decode_call(lib, Hq=12, Hkv=8) == 1            # Hq % Hkv != 0
    assert decode_call(lib, D=96) == 2                    # head_dim not built
    assert decode_call(lib, Hq=48, Hkv=3) == 2            # group size 16 not built
    assert decode_call(lib, BS=100) == 2                  # block size not built
    assert decode_call(lib, S=20000) == 2                 # too many sequences
    assert decode_call(lib, scale=float("nan")) == 1
    for bad in (float("nan"), float("inf"), -float("inf")):   # checked before the empty batch
        assert decode_call(lib, S=0, scale=bad) == 1
    assert decode_call(lib, S=0, scale=0.0) == 0 and decode_call(lib, S=0, scale=-2.0) == 0
    assert decode_call(lib) == 1                          # null pointers
    p = ctypes.c_void_p(0x10000)
    # workspace missing / too small / misaligned
    assert decode_call(lib, out=p, q=p, kc=p, vc=p, bt=p, cl=p) == 3
    assert decode_call(lib, out=p, q=p, kc=p, vc=p, bt=p, cl=p, ws=p, wsb=16) == 3
    need = lib.pkv_decode_workspace_size(4, 16, 8, 128, 32)
    assert decode_call(lib, out=p, q=p, kc=p, vc=p, bt=p, cl=p, ws=ctypes.c_void_p(0x10010),
                       wsb=need) == 3
    assert decode_call(lib, S=0) == 0                     # empty batch
    # a workspace bound too large to address: rejected before anything runs
    assert decode_call(lib, out=p, q=p, kc=p, vc=p, bt=p, cl=p, ws=p, wsb=1 << 40,
                       mtb=1 << 62) == 1
    # the shared-memory layout of the largest group and block size holds at
    # most 16093 sequences; other shapes reach the 16384-sequence limit first
    big = dict(out=p, q=p, kc=p, vc=p, bt=p, cl=p, Hq=64, Hkv=8, BS=512)
    assert decode_call(lib, **big, S=16094) == 2
    assert decode_call(lib, **big, S=16093) == 3          # fits: the (missing) workspace is next
    assert decode_call(lib, out=p, q=p, kc=p, vc=p, bt=p, cl=p, S=16384) == 3


def prefill_call(lib, **kw):
    a = dict(out=NULL, q=NULL, kc=NULL, vc=NULL, bt=NULL, cq=NULL, ck=NULL, S=2, T=100, mq=64,
             Hq=16, Hkv=8, D=128, BS=256, maxb=4, NB=16, scale=0.1, ws=NULL, wsb=0, st=NULL,
             stream=NULL)
    a.update(kw)
    return lib.pkv_paged_prefill_attn(*a.values())


def test_prefill_rejects_bad_arguments(lib):
    assert prefill_call(lib, Hq=10, Hkv=4) == 1
    assert prefill_call(lib, D=80) == 2
    assert prefill_call(lib, BS=32) == 2
    assert prefill_call(lib, Hq=32, Hkv=2) == 2           # group size 16 not built
    assert prefill_call(lib, T=-1) == 1
    assert prefill_call(lib) == 1                         # null pointers
    assert prefill_call(lib, T=0) == 0                    # nothing to do
    for bad in (float("nan"), float("inf"), -float("inf")):   # checked before the empty batch
        assert prefill_call(lib, T=0, scale=bad) == 1
    assert prefill_call(lib, T=0, scale=0.0) == 0 and prefill_call(lib, T=0, scale=-2.0) == 0
    # workspace missing / too small / misaligned
    p = ctypes.c_void_p(0x10000)
    ptrs = dict(out=p, q=p, kc=p, vc=p, bt=p, cq=p, ck=p)
    need = lib.pkv_prefill_workspace_size()
    assert need >= 8
    assert prefill_call(lib, **ptrs) == 3
    assert prefill_call(lib, **ptrs, ws=p, wsb=need - 1) == 3
    assert prefill_call(lib, **ptrs, ws=ctypes.c_void_p(0x10010), wsb=need) == 3


def test_decode_fault_hook_rejects_bad_arguments(lib):
    # checked before any device call
    assert lib.pkv_test_decode_fault(0, -1) == 1
    assert lib.pkv_test_decode_fault(1000, -2) == 1


def test_dequant_rejects_bad_arguments(lib):
    f = lib.pkv_w4a16_dequant
    p = ctypes.c_void_p(0x10000)
    assert f(p, p, p, 4, 256, 64, NULL) == 2          # only groups of 128
    assert f(p, p, p, 4, 200, 128, NULL) == 1         # k not a multiple of 128
    assert f(NULL, NULL, NULL, 4, 256, 128, NULL) == 1  # null pointers
    assert f(ctypes.c_void_p(0x10008), p, p, 4, 256, 128, NULL) == 1  # out misaligned
    assert f(p, p, ctypes.c_void_p(0x10001), 4, 256, 128, NULL) == 1  # scales misaligned
    assert f(NULL, NULL, NULL, 0, 256, 128, NULL) == 0  # nothing to do
