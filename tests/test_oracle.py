"""Pins for the fp64 CPU oracle (no GPU).

Each test checks the oracle against something other than itself: the pages' printed byte
figures, the IEEE binary16 decoding that numpy implements, a brute-force enumeration of a
sequence's slots, torch's float64 scaled-dot-product attention on contiguous K/V, closed-form
special cases, invariants (block permutation, shared = private), a literal replay of the
sink + ring buffer, and the algebra of rotations.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_147_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------------------ ledger
def test_ledger_matches_printed_figures():
    data = json.load(open(os.path.join(GOLDEN, "kv_ledger.json"), encoding="utf-8"))
    assert len(data["entries"]) >= 8
    for e in data["entries"]:
        got = oracle.kv_bytes(*e["args"])
        assert got == e["exact_bytes"], e["what"]
        printed = e["printed_value"]
        decimals = len(str(printed).split(".")[1]) if "." in str(printed) else 0
        tol = e.get("tol", 0.5 * 10 ** (-decimals) + 1e-12)
        assert abs(got / e["printed_unit_bytes"] - printed) <= tol, e["what"]


def test_ledger_is_linear_in_every_factor():
    base = oracle.kv_bytes(3, 5, 7, 11, 2, 13)
    assert base == 2 * 3 * 5 * 7 * 11 * 2 * 13
    for i in range(6):
        args = [3, 5, 7, 11, 2, 13]
        args[i] *= 2
        assert oracle.kv_bytes(*args) == 2 * base


# ------------------------------------------------------------------------------ fp16
def test_f16_decoder_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # signed zero keeps its sign
    assert math.copysign(1.0, ours[0x8000]) == -1.0


# ------------------------------------------------------------------------------ slots
def _enumerated_slots(table_row, n_blocks, bs):
    """All slots of one sequence in logical order: its blocks in table order, each block's
    offsets 0..bs-1 (an enumeration, not the div/mod formula)."""
    out = []
    for j in range(n_blocks):
        for o in range(bs):
            out.append(int(table_row[j]) * bs + o)
    return out


@pytest.mark.parametrize("bs", [16, 64, 5])
def test_slot_mapping_equals_enumeration(bs):
    rng = np.random.default_rng(bs)
    B, maxb = 5, 9
    nb = B * maxb + 3
    tables = rng.permutation(nb)[: B * maxb].reshape(B, maxb).astype(np.int32)
    seq, pos = [], []
    for b in range(B):
        for p in range(maxb * bs):
            seq.append(b)
            pos.append(p)
    got = oracle.slot_mapping(seq, pos, tables, bs)
    exp = []
    for b in range(B):
        exp.extend(_enumerated_slots(tables[b], maxb, bs))
    assert np.array_equal(got, np.array(exp, dtype=np.int64))
    # a negative position is padding
    assert oracle.slot_mapping([0], [-1], tables, bs)[0] == -1


# ------------------------------------------------------------------------------ ring
@pytest.mark.parametrize("S,W", [(4, 1020), (4, 20), (0, 7), (3, 1)])
def test_ring_slot_properties(S, W):
    cap = S + W
    for p in range(3 * cap + 5):
        r = oracle.ring_slot(p, S, W)
        if p < S:
            assert r == p                     # sinks are fixed
        else:
            assert S <= r < cap               # window slots
            assert oracle.ring_slot(p + W, S, W) == r   # period W
    # any W consecutive window positions cover the window slots exactly once
    for start in (S, S + 1, S + W - 1, 5 * W + S + 2):
        got = sorted(oracle.ring_slot(p, S, W) for p in range(start, start + W))
        assert got == list(range(S, cap))


class _LiteralRing:
    """Replays writes into a literal ring of S + W cells, cell index by the page's
    piecewise Slot definition, and reports what survives (independent of the oracle's
    closed-form valid set)."""

    def __init__(self, S, W):
        self.S, self.W = S, W
        self.cell = {}
        self.L = 0

    def slot(self, p):
        return p if p < self.S else self.S + (p - self.S) % self.W

    def append(self, n=1):
        for _ in range(n):
            self.cell[self.slot(self.L)] = self.L
            self.L += 1

    def rollback(self, n):
        if self.L >= n:
            self.L -= n

    def visible(self):
        return sorted(p for p in self.cell.values() if p < self.L)


def _hw(ring):
    return max(ring.cell.values()) + 1 if ring.cell else 0


@pytest.mark.parametrize("S,W", [(4, 20), (4, 1020), (2, 5)])
def test_ring_valid_set_matches_literal_replay(S, W):
    rng = np.random.default_rng(S * 100 + W)
    ring = _LiteralRing(S, W)
    for step in range(400):
        ring.append(int(rng.integers(1, 6)))
        if rng.random() < 0.4:
            n = int(rng.integers(0, 4))
            # precondition of the valid-set rule: a rollback never reaches below hw - W
            if ring.L - n >= _hw(ring) - W:
                ring.rollback(n)
        hw = _hw(ring)
        got = oracle.ring_valid(ring.L, hw, S, W)
        assert list(got) == ring.visible(), (step, ring.L, hw)
        if hw == ring.L:
            assert len(got) == min(ring.L, S + W)
        slots = [oracle.ring_slot(int(p), S, W) for p in got]
        assert len(set(slots)) == len(slots)


def test_ring_valid_without_rollback_is_sinks_plus_last_window():
    S, W = 4, 1020
    for L in (1, 3, 4, 5, 1023, 1024, 1025, 5000):
        got = list(oracle.ring_valid(L, L, S, W))
        if L <= S + W:
            assert got == list(range(L))
        else:
            assert got == list(range(S)) + list(range(L - W, L))


def test_ring_causal_drafts():
    S, W, P = 4, 20, 100
    # 4 drafts at P..P+3 appended (hw = L = P + 4); draft i sees up to P + i
    for i in range(4):
        got = list(oracle.ring_valid(P + 4, P + 4, S, W, q_len=4, qi=i))
        assert got == list(range(S)) + list(range(P + 4 - W, P + i + 1))


# ------------------------------------------------------------------------------ RoPE
def test_rope_identity_norm_and_relative_invariance():
    rng = np.random.default_rng(7)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    assert np.array_equal(oracle.rope(q, 0.0), q)
    for a in (1.0, 17.0, 1019.0):
        assert np.linalg.norm(oracle.rope(q, a)) == pytest.approx(np.linalg.norm(q), rel=1e-13)
    for a, b in ((3, 10), (100, 40), (0, 1023)):
        ref = oracle.rope(q, a) @ oracle.rope(k, b)
        for c in (1, 57, 900):
            assert oracle.rope(q, a + c) @ oracle.rope(k, b + c) == pytest.approx(ref, rel=1e-9, abs=1e-9)


def test_rope_matches_complex_rotation():
    """Rotate-half RoPE == multiplying the complex numbers x_i + i x_{i+D/2} by
    exp(i * index * base^(-2i/D))."""
    rng = np.random.default_rng(8)
    D = 128
    x = rng.standard_normal(D)
    for idx in (1.0, 5.0, 1000.0):
        z = x[: D // 2] + 1j * x[D // 2:]
        theta = 10000.0 ** (-2.0 * np.arange(D // 2) / D)
        z = z * np.exp(1j * idx * theta)
        ref = np.concatenate([z.real, z.imag])
        assert np.allclose(oracle.rope(x, idx), ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------------------------ attention
def _gather_contiguous(w, k_pool, v_pool, b, ctx):
    """Contiguous K/V [ctx, Hkv, D] of sequence b via the slot enumeration."""
    slots = _enumerated_slots(w.block_tables[b], (ctx + w.block_size - 1) // w.block_size,
                              w.block_size)[:ctx]
    blk = np.array(slots) // w.block_size
    off = np.array(slots) % w.block_size
    K = k_pool[blk, :, off, :].astype(np.float64)
    V = v_pool[blk, :, off, :].astype(np.float64)
    return K, V


def _sdpa_reference(w, q, k_pool, v_pool, context_lens):
    """torch float64 scaled_dot_product_attention over contiguous, enumerated K/V."""
    B, q_len, Hq, D = q.shape
    G = Hq // w.num_kv_heads
    out = np.zeros((B, q_len, Hq, D))
    for b in range(B):
        ctx = int(context_lens[b])
        K, V = _gather_contiguous(w, k_pool, v_pool, b, ctx)
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0)   # [Hq, ctx, D]
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0)
        Qt = torch.from_numpy(q[b].astype(np.float64)).permute(1, 0, 2)        # [Hq, q_len, D]
        mask = torch.ones(q_len, ctx, dtype=torch.bool)
        for i in range(q_len):
            mask[i, ctx - q_len + i + 1:] = False
        o = torch.nn.functional.scaled_dot_product_attention(
            Qt, Kt, Vt, attn_mask=mask, scale=w.scale)
        out[b] = o.permute(1, 0, 2).numpy()
    return out


def _tiny_inputs(poison=True):
    w = workloads.tiny()
    k, v = w.pools(poison=poison)
    k, v = k[0].numpy(), v[0].numpy()
    q = w.query(0).numpy()
    return w, q, k, v


def _fill_appended(w, k, v):
    """Replace the NaN-poisoned slots that the step appends with data (via the oracle)."""
    seq, pos = w.new_token_positions()
    slots = oracle.slot_mapping(seq, pos, w.block_tables, w.block_size)
    kn, vn = w.new_kv(0)
    oracle.kv_append(kn.numpy(), vn.numpy(), slots, k, v, w.block_size)
    return slots


def test_paged_attention_matches_torch_sdpa_tiny():
    w, q, k, v = _tiny_inputs()
    _fill_appended(w, k, v)
    got = oracle.paged_attention(q, k, v, w.block_tables, w.context_lens, w.block_size, w.scale)
    ref = _sdpa_reference(w, q, k, v, w.context_lens)
    assert np.isfinite(got).all()
    assert np.max(np.abs(got - ref)) < 1e-12


def test_paged_attention_causal_multi_query_matches_sdpa():
    rng = np.random.default_rng(11)
    w = workloads.tiny()
    k = rng.standard_normal((64, 2, 16, 128)).astype(np.float16)
    v = rng.standard_normal((64, 2, 16, 128)).astype(np.float16)
    q = rng.standard_normal((2, 4, 12, 128)).astype(np.float16)
    got = oracle.paged_attention(q, k, v, w.block_tables, w.context_lens, 16, w.scale)
    ref = _sdpa_reference(w, q, k, v, w.context_lens)
    assert np.max(np.abs(got - ref)) < 1e-12


@pytest.mark.parametrize("q_len,hq,bs", [(37, 16, 16), (64, 12, 16), (101, 16, 64)])
def test_paged_attention_prefill_chunk_matches_sdpa(q_len, hq, bs):
    """A chunk of q_len new queries over a paged cache (the chunked-prefill shape): query i sees
    positions [0, ctx - q_len + i]; a query with no visible position (q_len > ctx) gives 0."""
    rng = np.random.default_rng(q_len)
    lens = np.array([38, 101, 20], dtype=np.int32)
    nblk = [(int(n) + bs - 1) // bs for n in lens]
    perm = rng.permutation(sum(nblk) + 3).astype(np.int32)
    tables = np.full((3, max(nblk)), -1, np.int32)
    cur = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[cur:cur + n]
        cur += n
    nb = len(perm)
    k = rng.standard_normal((nb, 2, bs, 128)).astype(np.float16)
    v = rng.standard_normal((nb, 2, bs, 128)).astype(np.float16)
    q = rng.standard_normal((3, q_len, hq, 128)).astype(np.float16)
    scale = 0.0883
    got = oracle.paged_attention(q, k, v, tables, lens, bs, scale)
    G = hq // 2
    for b in range(3):
        ctx = int(lens[b])
        slots = _enumerated_slots(tables[b], nblk[b], bs)[:ctx]
        K = k[np.array(slots) // bs, :, np.array(slots) % bs, :].astype(np.float64)
        V = v[np.array(slots) // bs, :, np.array(slots) % bs, :].astype(np.float64)
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, dim=0)
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, dim=0)
        for i in range(q_len):
            vis = ctx - q_len + i + 1
            if vis <= 0:
                assert np.all(got[b, i] == 0.0)
                continue
            Qt = torch.from_numpy(q[b, i].astype(np.float64))[:, None, :]        # [Hq, 1, D]
            o = torch.nn.functional.scaled_dot_product_attention(
                Qt, Kt[:, :vis], Vt[:, :vis], scale=scale)
            assert np.max(np.abs(got[b, i] - o[:, 0].numpy())) < 1e-12, (b, i)


def test_single_token_context_returns_v():
    w, q, k, v = _tiny_inputs(poison=False)
    lens = np.array([1, 1], dtype=np.int32)
    got = oracle.paged_attention(q, k, v, w.block_tables, lens, 16, w.scale)
    for b in range(2):
        blk = w.block_tables[b, 0]
        for h in range(12):
            assert np.array_equal(got[b, 0, h], v[blk, h // 6, 0].astype(np.float64))


def test_constant_keys_or_zero_query_give_mean_v():
    w, q, k, v = _tiny_inputs(poison=False)
    k_const = np.ones_like(k)
    got = oracle.paged_attention(q, k_const, v, w.block_tables, w.context_lens, 16, w.scale)
    got0 = oracle.paged_attention(np.zeros_like(q), k, v, w.block_tables, w.context_lens, 16,
                                  w.scale)
    for b in range(2):
        _, V = _gather_contiguous(w, k, v, b, int(w.context_lens[b]))
        mean = V.mean(axis=0)                                    # [Hkv, D]
        for h in range(12):
            assert np.allclose(got[b, 0, h], mean[h // 6], rtol=0, atol=1e-12)
            assert np.allclose(got0[b, 0, h], mean[h // 6], rtol=0, atol=1e-12)


def test_huge_scale_selects_argmax_value():
    w, q, k, v = _tiny_inputs(poison=False)
    got = oracle.paged_attention(q, k, v, w.block_tables, w.context_lens, 16, 1e6)
    for b in range(2):
        K, V = _gather_contiguous(w, k, v, b, int(w.context_lens[b]))
        for h in range(12):
            s = K[:, h // 6, :] @ q[b, 0, h].astype(np.float64)
            assert np.array_equal(got[b, 0, h], V[int(np.argmax(s)), h // 6])


def test_block_permutation_invariance_is_exact():
    w, q, k, v = _tiny_inputs()
    _fill_appended(w, k, v)
    base = oracle.paged_attention(q, k, v, w.block_tables, w.context_lens, 16, w.scale)
    perm = np.random.default_rng(5).permutation(64)
    inv = np.argsort(perm)
    k2, v2 = k[inv], v[inv]          # block j moves to position perm[j]
    tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1)
    got = oracle.paged_attention(q, k2, v2, tables, w.context_lens, 16, w.scale)
    assert np.array_equal(got, base)


def test_shared_prefix_equals_private_copies():
    rng = np.random.default_rng(3)
    k = rng.standard_normal((20, 2, 16, 128)).astype(np.float16)
    v = rng.standard_normal((20, 2, 16, 128)).astype(np.float16)
    q = rng.standard_normal((3, 1, 12, 128)).astype(np.float16)
    shared = np.array([[0, 1, 2, 3], [0, 1, 4, 5], [0, 1, 6, 7]], dtype=np.int32)
    # private copies of blocks 0, 1 for sequences 1 and 2
    k[8:10], v[8:10] = k[0:2], v[0:2]
    k[10:12], v[10:12] = k[0:2], v[0:2]
    private = np.array([[0, 1, 2, 3], [8, 9, 4, 5], [10, 11, 6, 7]], dtype=np.int32)
    lens = np.array([60, 50, 64], dtype=np.int32)
    a = oracle.paged_attention(q, k, v, shared, lens, 16, 0.1)
    b = oracle.paged_attention(q, k, v, private, lens, 16, 0.1)
    assert np.array_equal(a, b)


def test_seq_mask_and_threads_do_not_change_results():
    w, q, k, v = _tiny_inputs()
    _fill_appended(w, k, v)
    a, nt = oracle.paged_attention(q, k, v, w.block_tables, w.context_lens, 16, w.scale,
                                   num_threads=1, return_threads=True)
    assert nt == 1
    b = oracle.paged_attention(q, k, v, w.block_tables, w.context_lens, 16, w.scale,
                               num_threads=3)
    assert np.array_equal(a, b)
    m = oracle.paged_attention(q, k, v, w.block_tables, w.context_lens, 16, w.scale,
                               seq_mask=np.array([0, 1]))
    assert np.array_equal(m[1], a[1]) and not m[0].any()


# ------------------------------------------------------------------------------ append / copy
def test_kv_append_round_trip_and_untouched_bytes():
    w, q, k, v = _tiny_inputs()
    k0, v0 = k.copy(), v.copy()
    seq, pos = w.new_token_positions()
    slots = oracle.slot_mapping(seq, pos, w.block_tables, w.block_size)
    kn, vn = (t.numpy() for t in w.new_kv(0))
    slots_pad = np.concatenate([slots, [-1]])
    kn_pad = np.concatenate([kn, np.full_like(kn[:1], 7.0)])
    vn_pad = np.concatenate([vn, np.full_like(vn[:1], 7.0)])
    oracle.kv_append(kn_pad, vn_pad, slots_pad, k, v, w.block_size)
    touched = np.zeros(k.shape[0] * k.shape[2], dtype=bool)
    for t, s in enumerate(slots):
        blk, off = divmod(int(s), w.block_size)
        assert k[blk, :, off].tobytes() == kn[t].tobytes()
        assert v[blk, :, off].tobytes() == vn[t].tobytes()
        touched[blk * w.block_size + off] = True
    kt = k.transpose(0, 2, 1, 3).reshape(-1, 2 * 128)
    k0t = k0.transpose(0, 2, 1, 3).reshape(-1, 2 * 128)
    assert kt[~touched].tobytes() == k0t[~touched].tobytes()
    assert not np.any(k == 7.0)      # the padded row went nowhere


def test_copy_blocks_all_layers():
    rng = np.random.default_rng(9)
    L, NB = 3, 10
    k = rng.standard_normal((L, NB, 2, 16, 128)).astype(np.float16)
    v = rng.standard_normal((L, NB, 2, 16, 128)).astype(np.float16)
    k0, v0 = k.copy(), v.copy()
    src, dst = [1, 1, 4], [7, 8, 9]
    oracle.copy_blocks(k, v, src, dst, L, NB * 2 * 16 * 128, 2 * 16 * 128)
    for l in range(L):
        for s, d in zip(src, dst):
            assert k[l, d].tobytes() == k0[l, s].tobytes()
            assert v[l, d].tobytes() == v0[l, s].tobytes()
        for j in range(NB):
            if j not in dst:
                assert k[l, j].tobytes() == k0[l, j].tobytes()


# ------------------------------------------------------------------------------ ring attention
def _ring_reference(q, k, v, table, L, hw, S, W, scale, bs=16):
    """Literal ring replay + complex-number RoPE + torch SDPA, one sequence, one kv head group."""
    q_len, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    ring = _LiteralRing(S, W)
    for p in range(hw):                 # positions 0..hw-1 written in order: each cell keeps
        ring.cell[ring.slot(p)] = p     # the last position written into it
    lo = max(S, hw - W)
    out = np.zeros((q_len, Hq, D))
    theta = 10000.0 ** (-2.0 * np.arange(D // 2) / D)

    def rot(x, idx):
        z = (x[..., : D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * idx * theta)
        return np.concatenate([z.real, z.imag], axis=-1)

    def cidx(p):
        return p if p < S else S + (p - lo)

    for i in range(q_len):
        vis = L - q_len + i + 1
        pos = sorted(p for p in ring.cell.values() if p < vis)
        rows = [ring.slot(p) for p in pos]
        blk = np.array([table[r // bs] for r in rows])
        off = np.array([r % bs for r in rows])
        K = k[blk, :, off, :].astype(np.float64)
        V = v[blk, :, off, :].astype(np.float64)
        K = np.stack([rot(K[t], cidx(p)) for t, p in enumerate(pos)])
        qv = rot(q[i].astype(np.float64), cidx(L - q_len + i))
        Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)
        Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
        Qt = torch.from_numpy(qv)[:, None, :]
        out[i] = torch.nn.functional.scaled_dot_product_attention(Qt, Kt, Vt, scale=scale)[:, 0].numpy()
    return out


@pytest.mark.parametrize("S,W,L,hw,q_len", [(4, 1020, 5000, 5004, 4), (4, 1020, 5002, 5004, 1),
                                             (4, 1020, 700, 700, 1), (4, 60, 130, 133, 2)])
def test_ring_attention_matches_literal_replay(S, W, L, hw, q_len):
    rng = np.random.default_rng(L + hw)
    bs = 16
    nblk = (S + W + bs - 1) // bs
    NB = nblk + 5
    k = rng.standard_normal((NB, 2, bs, 128)).astype(np.float16)
    v = rng.standard_normal((NB, 2, bs, 128)).astype(np.float16)
    table = rng.permutation(NB)[:nblk].astype(np.int32)
    q = rng.standard_normal((1, q_len, 12, 128)).astype(np.float16)
    got = oracle.ring_attention(q, k, v, table[None], [L], [hw], bs, S, W, 1 / math.sqrt(128))
    ref = _ring_reference(q[0], k, v, table, L, hw, S, W, 1 / math.sqrt(128), bs)
    assert np.max(np.abs(got[0] - ref)) < 1e-11


def test_ring_without_rope_and_wrap_is_paged_attention():
    """Before the ring wraps and with rotation off, ring attention is plain paged attention."""
    rng = np.random.default_rng(21)
    k = rng.standard_normal((70, 2, 16, 128)).astype(np.float16)
    v = rng.standard_normal((70, 2, 16, 128)).astype(np.float16)
    q = rng.standard_normal((2, 3, 12, 128)).astype(np.float16)
    tables = rng.permutation(70)[:64].reshape(2, 32).astype(np.int32)
    L = np.array([300, 511])
    a = oracle.ring_attention(q, k, v, tables, L, L, 16, 4, 508, 0.09, rope_mode=oracle.ROPE_NONE)
    b = oracle.paged_attention(q, k, v, tables, L.astype(np.int32), 16, 0.09)
    assert np.max(np.abs(a - b)) < 1e-13


# ------------------------------------------------------------------------------ FP8 (E4M3) cache
def _torch_e4m3_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decoder_matches_torch_for_every_code():
    ours = oracle.e4m3_to_f64(np.arange(256))
    ref = _torch_e4m3_decode_all()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # the format's landmarks: largest finite, smallest normal and subnormal, NaN codes
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF]) and nan.sum() == 2


def test_e4m3_encoder_matches_torch_rounding_in_range():
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(20000) * 4.0,
        rng.standard_normal(5000) * 2.0 ** -7,          # subnormal range
        rng.uniform(-447.0, 447.0, 5000),
        # exact ties between neighbouring codes: midpoints of every finite pair
        (lambda v: 0.5 * (v[:-1] + v[1:]))(np.sort(_torch_e4m3_decode_all()[:0x7F])),
    ]).astype(np.float32)
    ours = oracle.f64_to_e4m3(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encoder_nearest_ties_even_and_saturates():
    values = oracle.e4m3_to_f64(np.arange(0x7F))            # 0 .. 448, increasing
    assert np.all(np.diff(values) > 0)
    rng = np.random.default_rng(12)
    for x in rng.uniform(0.0, 448.0, 300):
        c = int(oracle.f64_to_e4m3(x))
        assert abs(values[c] - x) == np.min(np.abs(values - x))
    # ties go to the even code: 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39)
    assert oracle.f64_to_e4m3(1.0625) == 0x38 and oracle.f64_to_e4m3(1.1875) == 0x3A
    # finite values past the largest normal saturate; the sign is kept, zero too
    assert oracle.f64_to_e4m3(1000.0) == 0x7E and oracle.f64_to_e4m3(-1e6) == 0xFE
    assert oracle.f64_to_e4m3(-1e-9) == 0x80 and oracle.f64_to_e4m3(0.0) == 0x00
    # decode(encode(v)) == v for every finite code
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.f64_to_e4m3(oracle.e4m3_to_f64(c)) == c


def test_kv_append_fp8_quantises_in_binary32_and_touches_only_its_slots():
    rng = np.random.default_rng(13)
    nb, hkv, bs, d, T = 6, 2, 16, 128, 5
    k = rng.standard_normal((T, hkv, d)).astype(np.float16)
    v = rng.standard_normal((T, hkv, d)).astype(np.float16)
    ks = np.array([0.05, 0.37], np.float32)
    vs = np.array([0.11, 0.023], np.float32)
    slots = np.array([3, 17, -1, 95, 40], np.int64)
    kc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    vc = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    kc0, vc0 = kc.copy(), vc.copy()
    oracle.kv_append_fp8(k, v, slots, kc, vc, bs, ks, vs)
    ek, ev = kc0.copy(), vc0.copy()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        for h in range(hkv):
            xk = torch.from_numpy(k[t, h].astype(np.float32) / ks[h])
            xv = torch.from_numpy(v[t, h].astype(np.float32) / vs[h])
            ek[s // bs, h, s % bs] = xk.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            ev[s // bs, h, s % bs] = xv.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(kc, ek) and np.array_equal(vc, ev)


def test_fp8_attention_equals_fp16_attention_on_the_dequantised_cache():
    # with power-of-two scales every dequantised value is exact in fp16, so the FP8 oracle
    # must give exactly the fp16 oracle's result on that fp16 cache
    rng = np.random.default_rng(14)
    nb, hkv, hq, bs, d = 24, 2, 12, 16, 128
    lens = np.array([37, 100, 1, 64], np.int32)
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(lens), 8), -1, np.int32)
    o = 0
    for b, L in enumerate(lens):
        n = -(-int(L) // bs)
        bt[b, :n] = perm[o:o + n]
        o += n
    kc8 = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    vc8 = rng.integers(0, 256, (nb, hkv, bs, d), dtype=np.uint8)
    kc8[(kc8 & 0x7F) == 0x7F] = 0x11                    # no NaN codes in the cache
    vc8[(vc8 & 0x7F) == 0x7F] = 0x22
    ks = np.array([2.0 ** -3, 2.0 ** -6], np.float32)
    vs = np.array([2.0 ** -4, 1.0], np.float32)
    q = rng.standard_normal((len(lens), 1, hq, d)).astype(np.float16)
    got = oracle.paged_attention_fp8(q, kc8, vc8, ks, vs, bt, lens, bs, 1 / math.sqrt(d))
    kf = (oracle.e4m3_to_f64(kc8) * ks[None, :, None, None]).astype(np.float16)
    vf = (oracle.e4m3_to_f64(vc8) * vs[None, :, None, None]).astype(np.float16)
    assert np.array_equal(kf.astype(np.float64), oracle.e4m3_to_f64(kc8) * ks[None, :, None, None])
    want = oracle.paged_attention(q, kf, vf, bt, lens, bs, 1 / math.sqrt(d))
    assert np.array_equal(got, want)


# ------------------------------------------------------------------------------ speculative verify
def _softmax64(x):
    x = np.asarray(x, np.float64)
    e = np.exp(x - x.max(-1, keepdims=True))
    return e / e.sum(-1, keepdims=True)


def test_spec_verify_identical_models_accept_every_draft():
    rng = np.random.default_rng(31)
    B, K, V = 6, 4, 40
    t = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    d = t[:, :K].copy()
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    ua = rng.random((B, K)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    n, nxt = oracle.spec_verify(t, d, x, ua, us)
    assert np.all(n == K)
    # the bonus token: inverse CDF of the target's last position (first v with cdf > u)
    cdf = np.cumsum(_softmax64(t[:, K]), axis=-1)
    want = [int(np.searchsorted(cdf[b], float(us[b]) * cdf[b, -1], side="right"))
            for b in range(B)]
    assert list(nxt) == want


def test_spec_verify_two_token_closed_form():
    # draft P = (1/2, 1/2), target P = (1/4, 3/4): token 0 survives iff u < 1/2 and a rejection
    # always yields token 1 (the only positive residual); token 1 (ratio 3/2) always survives
    t = np.array([[[0.0, math.log(3.0)], [0.0, 0.0]]], np.float32)
    d = np.array([[[0.0, 0.0]]], np.float32)
    for u, acc in ((0.49, 1), (0.51, 0)):
        n, nxt = oracle.spec_verify(t, d, np.array([[0]]), np.array([[u]]), np.array([0.3]))
        assert n[0] == acc
        if not acc:
            assert nxt[0] == 1
    n, _ = oracle.spec_verify(t, d, np.array([[1]]), np.array([[0.999]]), np.array([0.3]))
    assert n[0] == 1


def test_spec_verify_first_token_follows_the_target_distribution():
    # speculative sampling's defining property: the first emitted token (the draft if accepted,
    # else the residual draw) is distributed as the target, whatever the draft distribution
    rng = np.random.default_rng(32)
    V, N = 6, 40000
    t = rng.standard_normal((1, 2, V)).astype(np.float32)
    d = (rng.standard_normal((1, 1, V)) * 1.5).astype(np.float32)
    pd = _softmax64(d[0, 0])
    x = rng.choice(V, size=N, p=pd).astype(np.int32)[:, None]
    ua = rng.random((N, 1)).astype(np.float32)
    us = rng.random(N).astype(np.float32)
    tt = np.repeat(t, N, axis=0)
    dd = np.repeat(d, N, axis=0)
    n, nxt = oracle.spec_verify(tt, dd, x, ua, us)
    first = np.where(n >= 1, x[:, 0], nxt)
    freq = np.bincount(first, minlength=V) / N
    assert np.max(np.abs(freq - _softmax64(t[0, 0]))) < 0.012
