"""Pins for the CPU oracle: checks against facts the pages and mathematics fix.

None of these re-types the oracle's own formula.  They check it against
  * the allocation rule the pages print (golden fixture),
  * brute force on never-paged (logical) arrays, in pure Python,
  * an independent library routine (torch's scaled_dot_product_attention, fp64),
  * closed forms (context of one token, zero scale, equal keys, one-hot logits,
    the two-key logistic form),
  * invariances (physical block permutation) and the prefill/decode relation,
and each pin is shown to catch a planted mistake in the oracle.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oa
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ helpers

def page_logical(rng, logical_k, logical_v, num_blocks, bs):
    """Place logical per-sequence K/V [L, Hkv, D] into a shuffled paged pool
    (test-side construction; independent of the oracle's gather)."""
    Hkv, D = logical_k[0].shape[1:]
    kc = np.zeros((num_blocks, bs, Hkv, D), np.uint16)
    vc = np.zeros_like(kc)
    perm = rng.permutation(num_blocks)
    maxb = max(-(-len(k) // bs) for k in logical_k)
    bt = np.full((len(logical_k), maxb), -1, np.int32)
    off = 0
    for s, (K, V) in enumerate(zip(logical_k, logical_v)):
        nb = -(-len(K) // bs)
        bt[s, :nb] = perm[off:off + nb]
        off += nb
        for p in range(len(K)):
            kc[bt[s, p // bs], p % bs] = K[p]
            vc[bt[s, p // bs], p % bs] = V[p]
    return kc, vc, bt


def brute_attention(q_row, K, V, scale):
    """Pure-Python float64 softmax attention, one query (lists of floats)."""
    logits = [scale * math.fsum(a * b for a, b in zip(q_row, k)) for k in K]
    top = max(logits)
    e = [math.exp(x - top) for x in logits]
    z = math.fsum(e)
    return [math.fsum(e[p] * V[p][d] for p in range(len(K))) / z for d in range(len(V[0]))]


def sdpa_reference(q, K, V, scale, mask):
    """torch's fp64 CPU scaled_dot_product_attention for one head.
    q [n, D], K/V [L, D], mask [n, L] bool (True = may attend)."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    out = torch.nn.functional.scaled_dot_product_attention(
        t(q), t(K), t(V), attn_mask=torch.from_numpy(mask)[None, None], scale=scale)
    return out[0, 0].numpy()


# ------------------------------------------------------------ bf16 encoding

def test_bf16_widening_known_patterns():
    bits = np.array([0x0000, 0x3F80, 0xC000, 0x3F81, 0x4049, 0x8000], np.uint16)
    want = [0.0, 1.0, -2.0, 1.0 + 2.0 ** -7, 3.140625, -0.0]
    got = oracle.bf16_bits_to_f64(bits)
    assert got.tolist() == want
    assert math.copysign(1.0, got[-1]) == -1.0


def test_generator_rounds_to_nearest_even():
    one = 1.0
    cases = {
        one: 0x3F80,
        one + 2.0 ** -8: 0x3F80,                   # halfway, tie to even (down)
        one + 3 * 2.0 ** -8: 0x3F82,               # halfway, tie to even (up)
        one + 2.0 ** -8 + 2.0 ** -20: 0x3F81,      # just above halfway
        -2.0: 0xC000,
    }
    x = np.array(list(cases.keys()), np.float32)
    assert wl.f32_to_bf16_bits(x).tolist() == list(cases.values())
    rng = np.random.default_rng(0)
    r = rng.standard_normal(10000, dtype=np.float32)
    back = oracle.bf16_bits_to_f64(wl.f32_to_bf16_bits(r))
    assert np.all(np.abs(back - r) <= np.abs(r) * 2.0 ** -8 + 1e-45)


# --------------------------------------------------------- block bookkeeping

def read_golden_allocation():
    bs, points = None, []
    with open(os.path.join(GOLDEN, "allocation_rule.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if not line:
                continue
            if line[0] == "block_size":
                bs = int(line[1])
            elif line[0] == "new_block_at":
                points.append(int(line[1]))
    return bs, points


def test_allocation_rule_matches_pages():
    bs, printed = read_golden_allocation()
    assert bs == oracle.BLOCK_SIZE == wl.BLOCK_SIZE == 256
    pts = oracle.allocation_points(2048, bs)
    for p in printed:
        assert p in pts
        assert p - 1 not in pts and p + 1 not in pts
    assert pts == [1 + bs * k for k in range(8)]
    # the block count of a length changes exactly at those points
    changes = [L for L in range(1, 2049)
               if oracle.blocks_for_length(L, bs) != oracle.blocks_for_length(L - 1, bs)]
    assert changes == pts
    assert [oracle.blocks_for_length(L) for L in (1, 255, 256, 257, 511, 512, 513)] == \
        [1, 1, 1, 2, 2, 2, 3]


def test_generator_slots_follow_block_tables():
    for make in (wl.tiny, wl.prefix):
        b = make(fill_cache=False)
        t = 0
        for s in range(b.num_seqs):
            for i in range(int(b.new_lens[s])):
                pos = int(b.cached_lens[s]) + i
                assert b.slot_mapping[t] == oracle.slot_of(b.block_tables[s], pos, b.block_size)
                t += 1
        used = b.block_tables[b.block_tables >= 0]
        assert len(set(used.tolist())) == len(used)          # no block shared
        assert len(set(b.slot_mapping.tolist())) == len(b.slot_mapping)


def test_slot_of_hand_values():
    row = np.array([7, 2, 5], np.int32)
    assert oracle.slot_of(row, 0, 4) == 28
    assert oracle.slot_of(row, 3, 4) == 31
    assert oracle.slot_of(row, 4, 4) == 8
    assert oracle.slot_of(row, 9, 4) == 21


# ----------------------------------------------------------------- kv_store

def test_kv_store_hand_example():
    # pool of 2 blocks of 4 slots, 1 kv head, D=2; sentinel everywhere
    kc = np.full((2, 4, 1, 2), 0xAAAA, np.uint16)
    vc = np.full((2, 4, 1, 2), 0x5555, np.uint16)
    k = np.array([[[1, 2]], [[3, 4]], [[5, 6]]], np.uint16)
    v = k + 100
    slots = np.array([5, -1, 0], np.int32)
    nk, nv = oracle.kv_store(kc, vc, k, v, slots)
    want_k = kc.copy()
    want_k[1, 1, 0] = [1, 2]     # slot 5 -> block 1, offset 1
    want_k[0, 0, 0] = [5, 6]     # slot 0 -> block 0, offset 0
    want_v = vc.copy()
    want_v[1, 1, 0] = [101, 102]
    want_v[0, 0, 0] = [105, 106]
    assert np.array_equal(nk, want_k) and np.array_equal(nv, want_v)
    assert np.all(kc == 0xAAAA)  # input untouched


def test_kv_store_then_gather_sees_new_token():
    b = wl.tiny()
    kc, vc = oracle.kv_store(b.k_cache, b.v_cache, b.k, b.v, b.slot_mapping)
    for s in range(b.num_seqs):
        L = int(b.context_lens[s])
        g = oracle.gather_sequence(kc, b.block_tables[s], L)
        assert np.array_equal(g[L - 1], b.k[s])
        gv = oracle.gather_sequence(vc, b.block_tables[s], L)
        assert np.array_equal(gv[L - 1], b.v[s])


# -------------------------------------------------------- decode attention

def tiny_logical_case(seed=11, lens=(5, 300), Hq=4, Hkv=2, D=8, bs=256, nb=8):
    rng = np.random.default_rng(seed)
    lk = [wl.normal_bf16(rng, (L, Hkv, D)) for L in lens]
    lv = [wl.normal_bf16(rng, (L, Hkv, D)) for L in lens]
    q = wl.normal_bf16(rng, (len(lens), Hq, D))
    kc, vc, bt = page_logical(rng, lk, lv, nb, bs)
    return q, lk, lv, kc, vc, bt, np.array(lens, np.int32)


def test_decode_matches_bruteforce_on_logical_arrays():
    q, lk, lv, kc, vc, bt, lens = tiny_logical_case()
    scale = 1 / math.sqrt(8)
    out = oracle.paged_decode_attn(q, kc, vc, bt, lens, scale)
    Hq, Hkv = 4, 2
    for s in range(2):
        K = oracle.bf16_bits_to_f64(lk[s])
        V = oracle.bf16_bits_to_f64(lv[s])
        qs = oracle.bf16_bits_to_f64(q[s])
        for h in range(Hq):
            j = h // (Hq // Hkv)
            want = brute_attention(qs[h].tolist(), K[:, j].tolist(), V[:, j].tolist(), scale)
            assert np.allclose(out[s, h], want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_decode_matches_torch_sdpa(G):
    rng = np.random.default_rng(100 + G)
    Hkv, D = 2, 16
    Hq = G * Hkv
    lens = [1, 255, 256, 257, 513]
    b = wl.build_batch("t", "decode", 0, [L - 1 for L in lens], [1] * len(lens), Hq, Hkv, D,
                       num_blocks=12, rng=rng)
    kc, vc = oracle.kv_store(b.k_cache, b.v_cache, b.k, b.v, b.slot_mapping)
    out = oracle.paged_decode_attn(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    for s, L in enumerate(lens):
        K = oracle.bf16_bits_to_f64(oracle.gather_sequence(kc, b.block_tables[s], L))
        V = oracle.bf16_bits_to_f64(oracle.gather_sequence(vc, b.block_tables[s], L))
        for h in range(Hq):
            ref = sdpa_reference(oracle.bf16_bits_to_f64(b.q[s, h])[None], K[:, h // G],
                                 V[:, h // G], b.scale, np.ones((1, L), bool))
            assert np.allclose(out[s, h], ref[0], rtol=0, atol=1e-12)


def test_decode_block_permutation_invariance():
    q, lk, lv, kc, vc, bt, lens = tiny_logical_case(seed=3)
    out = oracle.paged_decode_attn(q, kc, vc, bt, lens, 0.3)
    rng = np.random.default_rng(9)
    perm = rng.permutation(kc.shape[0])          # new id of old block b is perm[b]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2 = oracle.paged_decode_attn(q, kc2, vc2, bt2, lens, 0.3)
    assert np.array_equal(out, out2)


def test_context_of_one_returns_v_exactly():
    b = wl.build_batch("t", "decode", 4, [0, 0, 0], [1, 1, 1], 4, 2, 64, num_blocks=5)
    kc, vc = oracle.kv_store(b.k_cache, b.v_cache, b.k, b.v, b.slot_mapping)
    out = oracle.paged_decode_attn(b.q, kc, vc, b.block_tables, b.context_lens, b.scale)
    for s in range(3):
        for h in range(4):
            assert np.array_equal(out[s, h], oracle.bf16_bits_to_f64(b.v[s, h // 2]))


def test_zero_scale_and_equal_keys_give_mean_of_values():
    q, lk, lv, kc, vc, bt, lens = tiny_logical_case(seed=5)
    out = oracle.paged_decode_attn(q, kc, vc, bt, lens, 0.0)
    for s in range(2):
        mean = oracle.bf16_bits_to_f64(lv[s]).mean(axis=0)      # [Hkv, D]
        for h in range(4):
            assert np.allclose(out[s, h], mean[h // 2], rtol=0, atol=1e-13)
    # all keys equal: logits equal for any scale
    kc_eq = np.broadcast_to(kc[:1, :1], kc.shape).copy()
    bt0 = bt.copy()
    out = oracle.paged_decode_attn(q, kc_eq, vc, bt0, lens, 0.7)
    for s in range(2):
        mean = oracle.bf16_bits_to_f64(lv[s]).mean(axis=0)
        for h in range(4):
            assert np.allclose(out[s, h], mean[h // 2], rtol=0, atol=1e-13)


def test_one_hot_logit_selects_one_value_row():
    # one key aligned with q, others orthogonal: weight of the rest is e^-(big)
    D, L, hot = 4, 40, 17
    K = np.zeros((L, 1, D), np.uint16)
    K[:, 0, 1] = wl.f32_to_bf16_bits(np.ones(L, np.float32))
    K[hot, 0, :] = wl.f32_to_bf16_bits(np.array([64, 0, 0, 0], np.float32))
    V = wl.normal_bf16(np.random.default_rng(2), (L, 1, D))
    q = wl.f32_to_bf16_bits(np.array([[[2, 0, 0, 0]]], np.float32))
    kc, vc, bt = page_logical(np.random.default_rng(1), [K], [V], 1, 64)
    out = oracle.paged_decode_attn(q, kc, vc, bt, np.array([L], np.int32), 1.0)
    assert np.allclose(out[0, 0], oracle.bf16_bits_to_f64(V[hot, 0]), rtol=0, atol=1e-40)


def test_two_keys_logistic_closed_form():
    rng = np.random.default_rng(8)
    D = 6
    K = wl.normal_bf16(rng, (2, 1, D))
    V = wl.normal_bf16(rng, (2, 1, D))
    q = wl.normal_bf16(rng, (1, 1, D))
    kc, vc, bt = page_logical(rng, [K], [V], 3, 4)
    scale = 0.37
    out = oracle.paged_decode_attn(q, kc, vc, bt, np.array([2], np.int32), scale)
    qf, Kf, Vf = (oracle.bf16_bits_to_f64(a) for a in (q[0, 0], K[:, 0], V[:, 0]))
    delta = scale * float(np.dot(qf, Kf[0] - Kf[1]))
    w0 = 1.0 / (1.0 + math.exp(-delta))
    assert np.allclose(out[0, 0], w0 * Vf[0] + (1 - w0) * Vf[1], rtol=0, atol=1e-14)


# ------------------------------------------------------- prefill attention

def prefill_case(seed, cached, new, Hq=4, Hkv=2, D=16, bs=256):
    b = wl.build_batch("t", "prefill", seed, cached, new, Hq, Hkv, D, block_size=bs)
    kc, vc = oracle.kv_store(b.k_cache, b.v_cache, b.k, b.v, b.slot_mapping)
    return b, kc, vc


@pytest.mark.parametrize("G", [1, 2])
def test_prefill_matches_torch_sdpa_with_cached_prefix(G):
    Hkv = 2
    b, kc, vc = prefill_case(21 + G, [0, 256, 300], [70, 33, 257], Hq=G * Hkv, Hkv=Hkv)
    out = oracle.paged_prefill_attn(b.q, kc, vc, b.block_tables, b.cu_seqlens_q,
                                    b.cu_seqlens_k, b.scale)
    cu_q, cu_k = b.cu_seqlens_q, b.cu_seqlens_k
    for s in range(b.num_seqs):
        n = int(cu_q[s + 1] - cu_q[s])
        Lk = int(cu_k[s + 1] - cu_k[s])
        c = Lk - n
        K = oracle.bf16_bits_to_f64(oracle.gather_sequence(kc, b.block_tables[s], Lk))
        V = oracle.bf16_bits_to_f64(oracle.gather_sequence(vc, b.block_tables[s], Lk))
        Q = oracle.bf16_bits_to_f64(b.q[cu_q[s]:cu_q[s + 1]])
        mask = np.arange(Lk)[None, :] <= (c + np.arange(n))[:, None]
        for h in range(b.num_q_heads):
            ref = sdpa_reference(Q[:, h], K[:, h // G], V[:, h // G], b.scale, mask)
            assert np.allclose(out[cu_q[s]:cu_q[s + 1], h], ref, rtol=0, atol=1e-12)


def test_prefill_without_prefix_is_torch_causal():
    b, kc, vc = prefill_case(31, [0], [45], Hq=2, Hkv=2)
    out = oracle.paged_prefill_attn(b.q, kc, vc, b.block_tables, b.cu_seqlens_q,
                                    b.cu_seqlens_k, b.scale)
    K = oracle.bf16_bits_to_f64(oracle.gather_sequence(kc, b.block_tables[0], 45))
    V = oracle.bf16_bits_to_f64(oracle.gather_sequence(vc, b.block_tables[0], 45))
    Q = oracle.bf16_bits_to_f64(b.q)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))[None, None]
    for h in range(2):
        ref = torch.nn.functional.scaled_dot_product_attention(
            t(Q[:, h]), t(K[:, h]), t(V[:, h]), is_causal=True, scale=b.scale)[0, 0].numpy()
        assert np.allclose(out[:, h], ref, rtol=0, atol=1e-12)


def test_prefill_first_row_returns_first_value_and_last_row_equals_decode():
    b, kc, vc = prefill_case(41, [0, 512], [300, 20])
    out = oracle.paged_prefill_attn(b.q, kc, vc, b.block_tables, b.cu_seqlens_q,
                                    b.cu_seqlens_k, b.scale)
    # sequence 0 has no prefix: its first query sees only key 0
    for h in range(4):
        assert np.array_equal(out[0, h], oracle.bf16_bits_to_f64(b.v[0, h // 2]))
    # the last query of each sequence sees the whole context, as decode does
    last = b.cu_seqlens_q[1:] - 1
    dec = oracle.paged_decode_attn(b.q[last], kc, vc, b.block_tables, b.context_lens, b.scale)
    assert np.allclose(out[last], dec, rtol=0, atol=1e-13)


def test_prefill_row_subset_matches_full():
    b, kc, vc = prefill_case(51, [256, 0], [40, 90])
    full = oracle.paged_prefill_attn(b.q, kc, vc, b.block_tables, b.cu_seqlens_q,
                                     b.cu_seqlens_k, b.scale)
    rows = np.array([0, 39, 40, 77, 129])
    part = oracle.paged_prefill_attn(b.q, kc, vc, b.block_tables, b.cu_seqlens_q,
                                     b.cu_seqlens_k, b.scale, rows=rows)
    assert np.array_equal(full[rows], part[rows])
    mask = np.ones(len(full), bool)
    mask[rows] = False
    assert np.all(np.isnan(part[mask]))


def test_stale_nan_slots_are_never_read():
    b = wl.build_batch("t", "prefill", 61, [3, 256], [10, 5], 4, 2, 16, stale="nan")
    kc, vc = oracle.kv_store(b.k_cache, b.v_cache, b.k, b.v, b.slot_mapping)
    out = oracle.paged_prefill_attn(b.q, kc, vc, b.block_tables, b.cu_seqlens_q,
                                    b.cu_seqlens_k, b.scale)
    assert np.all(np.isfinite(out))
    dec = oracle.paged_decode_attn(b.q[b.cu_seqlens_q[1:] - 1], kc, vc, b.block_tables,
                                   b.context_lens, b.scale)
    assert np.all(np.isfinite(dec))


# --------------------------------------------- planted mistakes get caught

def test_pins_catch_a_wrong_gqa_mapping(monkeypatch):
    monkeypatch.setattr(oa, "kv_head_of", lambda h, Hq, Hkv: h % Hkv)
    with pytest.raises(AssertionError):
        test_decode_matches_torch_sdpa(2)


def test_pins_catch_a_wrong_causal_offset(monkeypatch):
    real = oa.paged_prefill_attn

    def top_left_aligned(q, kc, vc, bt, cu_q, cu_k, scale, rows=None):
        # plant: ignore the cached prefix when aligning the causal mask
        return real(q, kc, vc, bt, cu_q, cu_q, scale, rows)

    monkeypatch.setattr(oracle, "paged_prefill_attn", top_left_aligned)
    with pytest.raises(AssertionError):
        test_prefill_matches_torch_sdpa_with_cached_prefix(1)


def test_pins_catch_a_dropped_scale(monkeypatch):
    real = oa.attend
    monkeypatch.setattr(oa, "attend", lambda q, K, V, scale: real(q, K, V, 1.0))
    with pytest.raises(AssertionError):
        test_two_keys_logistic_closed_form()


def test_pins_catch_an_off_by_one_block_walk(monkeypatch):
    def shifted_gather(cache, row, length):
        bs = cache.shape[1]
        out = np.empty((length,) + cache.shape[2:], dtype=cache.dtype)
        for p in range(length):
            out[p] = cache[int(row[p // bs]), (p + 1) % bs]
        return out

    monkeypatch.setattr(oa, "gather_sequence", shifted_gather)
    with pytest.raises(AssertionError):
        test_decode_matches_bruteforce_on_logical_arrays()
