"""The host block pool (pkv_pool_*, C++ in libpkv.so) against the plain Python model in
oracle/blocks.py, and the model against what the pages and the hash's definition fix.

No GPU: the pool is host code. The model is pinned by FNV-1a's published test vectors, by
invariants (reference counts equal the tables that hold a block; every block is exactly one of
free, held or warm) and by the copy-on-write outcome the prefix-sharing fixture encodes; the
library's pool must then make exactly the model's choices (tables, reuse counts, copy pairs,
free-list order) over long random operation sequences.
"""
import numpy as np
import pytest

from oracle import blocks
from paged_kv_cache_147_gb300 import pkv


# ------------------------------------------------------------------------------ model pins
def test_fnv1a_matches_published_test_vectors():
    # FNV-1a 64-bit of "", "a" and "foobar" (one byte per step: token ids below 256)
    assert blocks.fnv1a([]) == 0xCBF29CE484222325
    assert blocks.fnv1a([0x61]) == 0xAF63DC4C8601EC8C
    assert blocks.fnv1a([ord(c) for c in "foobar"]) == 0x85944171F73967E8
    # chaining: hashing in two calls equals one call over the concatenation
    assert blocks.fnv1a([5, 6], blocks.fnv1a([1, 2, 3])) == blocks.fnv1a([1, 2, 3, 5, 6])


def _check_invariants(p, live):
    held = np.zeros(p.nb, int)
    for t in live.values():
        for b in t:
            held[b] += 1
    assert list(held) == p.ref
    free = set(p.free)
    assert len(free) == len(p.free)
    for b in range(p.nb):
        warm = p.ref[b] == 0 and p.key[b] is not None
        assert (b in free) + (p.ref[b] > 0) + warm == 1, b


def test_model_prefix_sharing_and_release():
    p = blocks.BlockPool(32, 4)
    sys_prompt = list(range(100, 112))                    # three full blocks
    a, ra = p.allocate(sys_prompt + [1, 2])
    b, rb = p.allocate(sys_prompt + [7, 8, 9, 10, 11])
    assert ra == 0 and rb == 3 and a[:3] == b[:3] and a[3] != b[3]
    c, rc = p.allocate([100, 101, 102, 999] + sys_prompt[4:])   # differs in block 0
    assert rc == 0 and not set(c) & set(a)
    d, rd = p.allocate(sys_prompt[:4] + [0] * 4 + sys_prompt[8:])  # same block 2 tokens, other parent
    assert rd == 1 and d[2] != a[2]
    live = {"a": a, "b": b, "c": c, "d": d}
    _check_invariants(p, live)
    p.release(a)
    del live["a"]
    _check_invariants(p, live)
    assert p.ref[b[0]] == 2                                 # still held by b and d
    for k in list(live):
        p.release(live.pop(k))
    _check_invariants(p, live)
    assert p.stats()["free"] == 32 and not p.index


def test_model_collision_needs_token_match():
    # with a 2-bit key almost every block collides; sharing must still follow the tokens
    p = blocks.BlockPool(64, 2, hash_bits=2)
    rng = np.random.default_rng(0)
    tables = []
    for _ in range(12):
        toks = list(rng.integers(0, 4, 6))
        t, r = p.allocate(toks)
        for q, (tq, prev) in enumerate(tables):
            shared = 0
            while shared < 3 and prev[2 * shared:2 * shared + 2] == toks[2 * shared:2 * shared + 2]:
                shared += 1
            assert list(t[:shared]) == list(tq[:shared])
        assert r == max([0] + [
            next((k for k in range(3) if prev[2 * k:2 * k + 2] != toks[2 * k:2 * k + 2]), 3)
            for _, prev in tables])
        tables.append((t, toks))


def test_model_fork_then_append_copies_until_one_holder_is_left():
    # the prefix fixture's reading: four children of a parent whose last block is partly
    # filled append one token each; the first three copy the block, the last writes in place
    p = blocks.BlockPool(16, 4)
    parent, _ = p.allocate(list(range(10)))               # blocks 0-1 full, block 2 holds 2
    kids = [p.fork(parent) for _ in range(4)]
    p.release(parent)
    copies = []
    for i, k in enumerate(kids):
        t, c = p.append(k, 10, 1)
        copies.append(c)
        kids[i] = t
    assert [len(c) for c in copies] == [1, 1, 1, 0]
    assert all(c[0][0] == parent[2] for c in copies[:3])
    assert kids[3][2] == parent[2] and len({k[2] for k in kids}) == 4
    assert all(k[:2] == parent[:2] for k in kids) and p.ref[parent[0]] == 4


def test_model_warm_blocks_are_reused_then_reclaimed_oldest_first():
    p = blocks.BlockPool(6, 2)
    p.warm([1, 2, 3, 4])                                  # two warm blocks
    p.warm([9, 9])                                        # one more, newer
    assert p.stats() == {"total": 6, "used": 0, "shared": 0, "free": 3, "warm": 3}
    t, r = p.allocate([1, 2, 3, 4, 5])                    # reuses both, takes one
    assert r == 2 and p.stats()["warm"] == 1
    u, _ = p.allocate(list(range(20, 24)))                # 2 blocks: free list has 2
    v, _ = p.allocate([7, 7])                             # reclaims the warm [9, 9] block
    assert p.stats()["warm"] == 0
    with pytest.raises(blocks.OutOfBlocks):
        p.allocate([8, 8])


def test_model_evicting_a_parent_drops_its_children_from_the_index():
    # Two warm blocks [1,2] -> [3,4]; a new prompt evicts the parent [1,2] and its id is
    # re-indexed for [5,6]. The child [3,4] followed [1,2], not [5,6], so a prompt [5,6,3,4]
    # may reuse only its first block. (With a 1-bit key every block collides: only the
    # parent and token checks stand between the prompt and the stale child.)
    for make in (lambda: blocks.BlockPool(2, 2, hash_bits=1),
                 lambda: pkv.BlockPool(2, 2, 1)):
        p = make()
        p.warm([1, 2, 3, 4])
        t1, r1 = p.allocate([5, 6])
        assert r1 == 0 and list(t1) == [0]
        t2, r2 = p.allocate([5, 6, 3, 4])
        assert r2 == 1 and list(t2) == [0, 1]
        if hasattr(p, "close"):
            p.close()


class _Shadow:
    """What each physical block really holds: the token prefix, from position 0, that was
    current when its last row was written (copies carry it over). A reused block is correct
    only if its prefix equals the new prompt's."""

    def __init__(self, nb, bs):
        self.bs = bs
        self.held = [()] * nb

    def allocated(self, table, reused, toks):
        for j in range(reused):
            assert self.held[table[j]] == tuple(toks[:(j + 1) * self.bs]), (j, table[j])
        for j in range(reused, len(table)):
            end = min((j + 1) * self.bs, len(toks))
            self.held[table[j]] = tuple(toks[:end]) if j * self.bs < len(toks) else ()

    def appended(self, table, copies, length, n, toks):
        for src, dst in copies:
            self.held[dst] = self.held[src]
        for j in range(length // self.bs, (length + n - 1) // self.bs + 1):
            self.held[table[j]] = tuple(toks[:min((j + 1) * self.bs, length + n)])


# ------------------------------------------------------------------------------ library == model
def _random_ops(seed, nb=48, bs=4, steps=400, hash_bits=64):
    rng = np.random.default_rng(seed)
    lib = pkv.BlockPool(nb, bs, hash_bits)
    ref = blocks.BlockPool(nb, bs, hash_bits)
    shadow = _Shadow(nb, bs)
    prompts = [list(rng.integers(0, 50, rng.integers(0, 14))) for _ in range(5)]
    live = {}     # name -> (table, length, tokens)
    nid = 0
    for step in range(steps):
        op = rng.choice(["alloc", "alloc", "append", "append", "fork", "release", "warm"])
        if op == "alloc" or not live:
            base = prompts[rng.integers(len(prompts))]
            toks = base + list(rng.integers(0, 50, rng.integers(0, 6)))
            mt = len(toks) + int(rng.integers(0, 6))
            try:
                tr, rr = ref.allocate(toks, mt)
            except blocks.OutOfBlocks:
                with pytest.raises(pkv.PkvError) as e:
                    lib.allocate(toks, mt)
                assert e.value.status == pkv.ENOSPC
                continue
            tl, rl = lib.allocate(toks, mt)
            assert list(tl) == tr and rl == rr, step
            shadow.allocated(tr, rr, toks)
            live[nid] = (tr, len(toks), toks)
            nid += 1
        elif op == "append":
            k = list(live)[rng.integers(len(live))]
            t, L, toks = live[k]
            n = int(rng.integers(1, 6))
            toks2 = toks + list(rng.integers(0, 50, n))
            try:
                tr, cr = ref.append(t, L, n, all_tokens=toks2)
            except blocks.OutOfBlocks:
                with pytest.raises(pkv.PkvError):
                    lib.append(np.asarray(t, np.int32), L, n, all_tokens=toks2)
                continue
            tl, cl = lib.append(np.asarray(t, np.int32), L, n, all_tokens=toks2)
            assert list(tl) == tr and [tuple(x) for x in cl.tolist()] == cr, step
            shadow.appended(tr, cr, L, n, toks2)
            live[k] = (tr, L + n, toks2)
        elif op == "fork":
            k = list(live)[rng.integers(len(live))]
            t, L, toks = live[k]
            ref.fork(t)
            lib.fork(np.asarray(t, np.int32))
            live[nid] = (list(t), L, list(toks))
            nid += 1
        elif op == "release":
            k = list(live)[rng.integers(len(live))]
            t, _, _ = live.pop(k)
            ref.release(t)
            lib.release(np.asarray(t, np.int32))
        else:
            toks = prompts[rng.integers(len(prompts))]
            try:
                tw, rw = ref.warm(toks)
            except blocks.OutOfBlocks:
                with pytest.raises(pkv.PkvError):
                    lib.warm(toks)
                continue
            lib.warm(toks)
            shadow.allocated(tw, rw, toks[:(len(toks) // bs) * bs])
        assert lib.stats() == ref.stats(), (step, op)
        assert [lib.refcount(b) for b in range(nb)] == ref.ref, (step, op)
    _check_invariants(ref, {k: v[0] for k, v in live.items()})
    lib.close()


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_library_pool_equals_model(seed):
    _random_ops(seed)


def test_library_pool_equals_model_under_collisions_and_pressure():
    _random_ops(7, nb=20, bs=2, steps=600, hash_bits=3)


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_reused_blocks_hold_the_prompt_prefix_under_eviction(seed):
    # tiny pools, one-bit keys and few distinct tokens: parents are evicted and their ids
    # reused all the time; every reused block must still hold exactly the prompt's prefix
    _random_ops(seed, nb=10, bs=2, steps=800, hash_bits=1)


def test_library_pool_rejects_bad_arguments_without_change():
    lib = pkv.BlockPool(8, 4)
    t, _ = lib.allocate(list(range(9)))
    before = lib.stats()
    with pytest.raises(pkv.PkvError) as e:
        lib.release(np.array([t[0], 99], np.int32))       # not a block
    assert e.value.status == pkv.EINVAL
    with pytest.raises(pkv.PkvError) as e:
        lib.allocate(list(range(100)))                    # more than the pool holds
    assert e.value.status == pkv.ENOSPC
    assert lib.stats() == before
    lib.release(t)
    with pytest.raises(pkv.PkvError):
        lib.release(t)                                    # no longer held
    assert lib.stats()["free"] == 8


def test_model_reuse_equals_longest_common_block_prefix():
    # with nothing released, a new prompt reuses exactly as many leading full blocks as the
    # longest full-block prefix it shares with any earlier prompt (brute force over pairs)
    rng = np.random.default_rng(5)
    bs = 3
    p = blocks.BlockPool(2000, bs)
    lib = pkv.BlockPool(2000, bs)
    stems = [list(rng.integers(0, 3, 12)) for _ in range(4)]
    seen = []
    for _ in range(120):
        s = stems[rng.integers(len(stems))]
        cut = int(rng.integers(0, 13))
        toks = s[:cut] + list(rng.integers(0, 3, rng.integers(0, 7)))
        want = 0
        for prev in seen:
            k = 0
            while (k + 1) * bs <= min(len(prev), len(toks)) and \
                    prev[k * bs:(k + 1) * bs] == toks[k * bs:(k + 1) * bs]:
                k += 1
            want = max(want, k)
        _, r = p.allocate(toks)
        _, rl = lib.allocate(toks)
        assert r == want == rl
        seen.append(toks)
