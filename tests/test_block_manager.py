"""The host block manager (pkv_bm_*): reference-counted 256-token blocks with
hash-chained prefix sharing.  CPU only.

Pinned to the pages through the allocation rule of the golden fixture (a new
block when the length reaches 257, 513, ...) and to the oracle's slot
definition; the sharing rules are checked against a plain Python model of
which leading full blocks two prompts have in common."""
import os

import numpy as np
import pytest

import oracle
import paged_kv_cache_241_gb300 as pkv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "allocation_rule.txt")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pkv.LIB_PATH):
        from paged_kv_cache_241_gb300 import build

        build.build()
    return pkv.load()


def golden_rule():
    bs, points = None, []
    for line in open(GOLDEN):
        line = line.split("#")[0].split()
        if line and line[0] == "block_size":
            bs = int(line[1])
        elif line and line[0] == "new_block_at":
            points.append(int(line[1]))
    return bs, points


def test_growth_follows_the_allocation_rule(lib):
    bs, points = golden_rule()
    bm = pkv.BlockManager(8, bs)
    bm.allocate(0, [7])
    seen, held = [], bm.num_blocks - bm.num_free_blocks
    for length in range(2, max(points) + 2):
        bm.append(0, length)
        now = bm.num_blocks - bm.num_free_blocks
        if now > held:
            seen.append(length)
        held = now
    assert seen[: len(points)] == points
    assert oracle.allocation_points(max(points) + 1, bs)[: len(points) + 1] == [1] + points


def test_slots_match_the_oracle_definition(lib):
    bm = pkv.BlockManager(16, 256)
    rng = np.random.default_rng(1)
    bm.allocate(5, rng.integers(0, 1000, size=700))
    row = bm.block_table(5, 6)
    slots = bm.slots(5, 0, 700)
    assert [int(s) for s in slots] == [oracle.slot_of(row, p) for p in range(700)]


def prompt(rng, n, prefix=None):
    t = rng.integers(0, 50000, size=n).astype(np.int32)
    if prefix is not None:
        t[: len(prefix)] = prefix
    return t


def test_shared_full_prefix_blocks(lib):
    rng = np.random.default_rng(2)
    bm = pkv.BlockManager(32, 256)
    a = prompt(rng, 700)
    assert bm.allocate(0, a) == 0
    assert bm.allocate(1, prompt(rng, 600, a[:512])) == 512   # two full blocks in common
    assert bm.allocate(2, prompt(rng, 300, a[:256])) == 256   # one
    assert bm.allocate(3, prompt(rng, 300, a[:255])) == 0     # no full block in common
    ra, r1, r2 = bm.block_table(0, 3), bm.block_table(1, 3), bm.block_table(2, 2)
    assert list(r1[:2]) == list(ra[:2]) and r1[2] != ra[2]
    assert r2[0] == ra[0] and r2[1] not in ra
    assert bm.ref_count(int(ra[0])) == 3 and bm.ref_count(int(ra[1])) == 2
    assert bm.ref_count(int(ra[2])) == 1


def test_same_block_after_a_different_prefix_is_not_shared(lib):
    rng = np.random.default_rng(3)
    bm = pkv.BlockManager(16, 256)
    a = prompt(rng, 512)
    b = prompt(rng, 512)
    b[256:] = a[256:]  # same second block, different first block
    bm.allocate(0, a)
    assert bm.allocate(1, b) == 0
    assert set(bm.block_table(0, 2)).isdisjoint(set(bm.block_table(1, 2)))


def test_partial_block_never_shared_and_last_token_recomputed(lib):
    rng = np.random.default_rng(4)
    bm = pkv.BlockManager(16, 256)
    a = prompt(rng, 300)
    bm.allocate(0, a)
    assert bm.allocate(1, a.copy()) == 256          # the 44-token tail is not shared
    assert bm.block_table(0, 2)[1] != bm.block_table(1, 2)[1]
    full = prompt(rng, 512)
    bm.allocate(2, full)
    assert bm.allocate(3, full.copy()) == 511       # every block shared, last token recomputed
    assert list(bm.block_table(2, 2)) == list(bm.block_table(3, 2))


def test_free_keeps_content_until_reused(lib):
    rng = np.random.default_rng(5)
    bm = pkv.BlockManager(4, 256)
    a = prompt(rng, 512)
    bm.allocate(0, a)
    blocks = list(bm.block_table(0, 2))
    bm.free(0)
    assert bm.num_free_blocks == 4 and all(bm.ref_count(b) == 0 for b in blocks)
    assert bm.allocate(1, prompt(rng, 600, a)) == 512  # freed blocks found again
    assert list(bm.block_table(1, 2)) == blocks
    bm.free(1)
    bm.allocate(2, prompt(rng, 1024))                  # the pool turns over
    bm.free(2)
    assert bm.allocate(3, prompt(rng, 600, a)) == 0    # content is gone


def test_generated_blocks_become_shareable(lib):
    rng = np.random.default_rng(6)
    bm = pkv.BlockManager(8, 256)
    a = prompt(rng, 200)
    bm.allocate(0, a)
    gen = rng.integers(0, 50000, size=56)
    for t in gen:
        bm.append(0, int(t))
    full = np.concatenate([a, gen]).astype(np.int32)
    assert bm.allocate(1, prompt(rng, 400, full)) == 256


def test_out_of_blocks_changes_nothing(lib):
    rng = np.random.default_rng(7)
    bm = pkv.BlockManager(3, 256)
    bm.allocate(0, prompt(rng, 300))
    with pytest.raises(pkv.PkvError) as e:
        bm.allocate(1, prompt(rng, 600))
    assert e.value.status == pkv.PKV_ERR_OUT_OF_BLOCKS
    assert bm.num_free_blocks == 1 and bm.num_tokens(1) == -1
    bm.allocate(1, prompt(rng, 200))       # the last free block
    for _ in range(56):
        bm.append(1, 1)                    # fills it
    with pytest.raises(pkv.PkvError):
        bm.append(1, 1)                    # token 257 needs a block
    assert bm.num_tokens(1) == 256


def test_bad_calls(lib):
    bm = pkv.BlockManager(4, 256)
    with pytest.raises(pkv.PkvError):
        bm.free(9)
    with pytest.raises(pkv.PkvError):
        bm.append(9, 1)
    with pytest.raises(pkv.PkvError):
        bm.allocate(1, [])
    bm.allocate(1, [1, 2, 3])
    with pytest.raises(pkv.PkvError):
        bm.allocate(1, [4])          # already present
    with pytest.raises(pkv.PkvError):
        bm.slots(1, 2, 5)            # past the sequence
    assert lib.pkv_bm_create(0, 256) is None


def common_full_blocks(a, b, bs):
    n = 0
    while (n + 1) * bs <= min(len(a), len(b)) and np.array_equal(a[: (n + 1) * bs], b[: (n + 1) * bs]):
        n += 1
    return n


def test_random_operations_keep_the_invariants(lib):
    # A plain model: each live sequence's tokens; a block is shared by two
    # sequences only where they hold the same leading full blocks, and the
    # reference counts equal the number of live sequences holding a block.
    rng = np.random.default_rng(8)
    bs, nb = 16, 64
    bm = pkv.BlockManager(nb, bs)
    live, roots, next_id = {}, [prompt(rng, 64) for _ in range(4)], 0
    for step in range(3000):
        op = rng.integers(0, 3)
        if op == 0 or not live:
            root = roots[rng.integers(0, len(roots))]
            n = int(rng.integers(1, 80))
            keep = int(rng.integers(0, 65))
            t = prompt(rng, n, root[: min(keep, n)])
            try:
                bm.allocate(next_id, t)
                live[next_id] = list(t)
            except pkv.PkvError as e:
                assert e.status == pkv.PKV_ERR_OUT_OF_BLOCKS
            next_id += 1
        elif op == 1:
            s = list(live)[rng.integers(0, len(live))]
            tok = int(rng.integers(0, 50000))
            try:
                bm.append(s, tok)
                live[s].append(tok)
            except pkv.PkvError as e:
                assert e.status == pkv.PKV_ERR_OUT_OF_BLOCKS
        else:
            s = list(live)[rng.integers(0, len(live))]
            bm.free(s)
            del live[s]
        if step % 50 == 0 or step == 2999:
            tables = {s: list(bm.block_table(s, (len(t) + bs - 1) // bs)) for s, t in live.items()}
            refs = np.zeros(nb, dtype=int)
            for s, t in live.items():
                assert bm.num_tokens(s) == len(t)
                assert len(tables[s]) == (len(t) + bs - 1) // bs
                for b in tables[s]:
                    refs[b] += 1
            assert [bm.ref_count(b) for b in range(nb)] == list(refs)
            assert bm.num_free_blocks == int((refs == 0).sum())
            ids = list(live)
            for i in range(len(ids)):
                for j in range(i + 1, len(ids)):
                    a, b = np.array(live[ids[i]]), np.array(live[ids[j]])
                    shared = [k for k in range(min(len(tables[ids[i]]), len(tables[ids[j]])))
                              if tables[ids[i]][k] == tables[ids[j]][k]]
                    # blocks are only ever shared at equal logical positions,
                    # and only within the common full prefix
                    assert set(tables[ids[i]]) & set(tables[ids[j]]) == {tables[ids[i]][k] for k in shared}
                    assert all(k < common_full_blocks(a, b, bs) for k in shared)
