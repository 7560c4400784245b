"""GPU parity: the CUDA library (through its C ABI) against the fp64 CPU oracle.

Addressing, appended cache contents and copy-on-write copies must be bit-exact (every pool
byte, NaN poison included); attention must be within the parity bar in tests/_util.py.
Inputs come from the seeded generators in paged_kv_cache_147_gb300.workloads; the oracle
always works on its own host copies, never on a result of the CUDA path.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_147_gb300 import pkv, workloads

from _util import assert_attn_close, f16_host, u16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(a, dtype):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=dtype, device=DEV)


def _run_decode_layer(w, k_l, v_l, bt_d, cl_d, slots_d, q, kn, vn, ws, fused=False):
    out = torch.empty_like(q)
    if fused:
        pkv.paged_attn_decode_append(out, q, kn, vn, k_l, v_l, bt_d, cl_d, w.scale, ws)
    else:
        pkv.kv_append(kn, vn, slots_d, k_l, v_l)
        pkv.paged_attn_decode(out, q, k_l, v_l, bt_d, cl_d, w.scale, ws)
    return out


def _check_layer(w, layer, k_all, v_all, bt_d, cl_d, slots_d, orc_slots, ws, seq_mask=None,
                 fused=False):
    """Append + decode one layer on the GPU (separate calls, or the fused entry point); the
    oracle redoes the append on a host copy of the pre-append pool and attends over its own
    copy."""
    k_host = f16_host(k_all[layer]).copy()
    v_host = f16_host(v_all[layer]).copy()
    q = w.query(layer, DEV)
    kn, vn = w.new_kv(layer, DEV)
    out = _run_decode_layer(w, k_all[layer], v_all[layer], bt_d, cl_d, slots_d, q, kn, vn, ws,
                            fused)
    torch.cuda.synchronize()
    oracle.kv_append(f16_host(kn), f16_host(vn), orc_slots, k_host, v_host, w.block_size)
    assert np.array_equal(u16(k_all[layer]), k_host.view(np.uint16)), f"K pool layer {layer}"
    assert np.array_equal(u16(v_all[layer]), v_host.view(np.uint16)), f"V pool layer {layer}"
    ref = oracle.paged_attention(f16_host(q), k_host, v_host, w.block_tables, w.context_lens,
                                 w.block_size, w.scale, seq_mask=seq_mask)
    if seq_mask is not None:
        sel = np.asarray(seq_mask, bool)
        return assert_attn_close(out[torch.as_tensor(sel, device=DEV)], ref[sel],
                                 f"{w.name} layer {layer}")
    return assert_attn_close(out, ref, f"{w.name} layer {layer}")


def _setup(w, poison=True):
    k_all, v_all = w.pools(DEV, poison=poison)
    bt_d = _dev(w.block_tables, torch.int32)
    cl_d = _dev(w.context_lens, torch.int32)
    seq, pos = w.new_token_positions()
    slots_d = pkv.slot_mapping(_dev(seq, torch.int32), _dev(pos, torch.int64), bt_d, w.block_size)
    orc_slots = oracle.slot_mapping(seq, pos, w.block_tables, w.block_size)
    torch.cuda.synchronize()
    assert np.array_equal(slots_d.cpu().numpy(), orc_slots), "slot mapping"
    ws = pkv.make_workspace(w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads)
    return k_all, v_all, bt_d, cl_d, slots_d, orc_slots, ws


@pytest.fixture(autouse=True)
def _clean_device_error():
    pkv.device_error(clear=True)
    yield
    assert pkv.device_error(clear=True) == 0, "a kernel bounds guard fired"


# ------------------------------------------------------------------------------ workloads
def test_tiny_append_decode():
    w = workloads.tiny()
    state = _setup(w)
    _check_layer(w, 0, *state)


def test_edge_1p1b_all_layers():
    w = workloads.edge_1p1b()
    state = _setup(w)
    worst = 0.0
    for layer in range(w.num_layers):
        worst = max(worst, _check_layer(w, layer, *state)[0])
    assert worst <= 2e-3


@pytest.mark.parametrize("make", [workloads.llama70b_b16, workloads.llama70b_mixed])
def test_llama70b_sampled_layers(make):
    w = make()
    state = _setup(w)
    for layer in (0, 1, 40, 79):
        _check_layer(w, layer, *state)


@pytest.mark.parametrize("make,layers", [(workloads.tiny, (0,)),
                                         (workloads.edge_1p1b, tuple(range(24))),
                                         (workloads.llama70b_b16, (0, 1, 40, 79)),
                                         (workloads.llama70b_mixed, (0, 79))])
def test_fused_append_decode(make, layers):
    w = make()
    state = _setup(w)
    for layer in layers:
        _check_layer(w, layer, *state, fused=True)


@pytest.mark.parametrize("q_len,lens", [(2, [33, 16, 2, 100]), (4, [64, 5, 31, 4]), (3, [1000, 47])])
def test_fused_append_multi_token(q_len, lens):
    """Several new tokens per sequence, straddling chunk and block boundaries."""
    rng = np.random.default_rng(q_len)
    lens = np.asarray(lens, dtype=np.int32)
    bs, hkv, hq = 16, 2, 8
    nblk = [(int(x) + bs - 1) // bs for x in lens]
    nb = sum(nblk) + 2
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(lens), max(nblk)), -1, np.int32)
    cur = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[cur:cur + n]
        cur += n
    k = rng.standard_normal((nb, hkv, bs, 128)).astype(np.float16)
    v = rng.standard_normal((nb, hkv, bs, 128)).astype(np.float16)
    q = rng.standard_normal((len(lens), q_len, hq, 128)).astype(np.float16)
    kn = rng.standard_normal((len(lens) * q_len, hkv, 128)).astype(np.float16)
    vn = rng.standard_normal((len(lens) * q_len, hkv, 128)).astype(np.float16)
    kd, vd = torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV)
    out = torch.empty((len(lens), q_len, hq, 128), dtype=torch.float16, device=DEV)
    ws = pkv.make_workspace(len(lens), q_len, hq, hkv)
    pkv.paged_attn_decode_append(out, torch.from_numpy(q).to(DEV), torch.from_numpy(kn).to(DEV),
                                 torch.from_numpy(vn).to(DEV), kd, vd, _dev(tables, torch.int32),
                                 _dev(lens, torch.int32), 0.09, ws)
    torch.cuda.synchronize()
    seq = np.repeat(np.arange(len(lens), dtype=np.int32), q_len)
    pos = (lens[:, None] - q_len + np.arange(q_len)[None, :]).reshape(-1).astype(np.int64)
    slots = oracle.slot_mapping(seq, pos, tables, bs)
    oracle.kv_append(kn, vn, slots, k, v, bs)
    assert np.array_equal(u16(kd), k.view(np.uint16)) and np.array_equal(u16(vd), v.view(np.uint16))
    ref = oracle.paged_attention(q, k, v, tables, lens, bs, 0.09)
    assert_attn_close(out, ref, f"fused q_len={q_len}")


def test_prefix_fork_copy_on_write():
    w = workloads.prefix()
    k_all, v_all = w.pools(DEV, poison=True)
    tables = w.block_tables.copy()
    ref = w.refcount.copy()
    free = list(w.free_blocks)
    # children 60..63 share the parent's partly filled last block X; a writer that finds X
    # shared (refcount > 1) copies it to a fresh block first, the last child writes in place
    last = (int(w.context_lens[60]) - 1) // w.block_size
    X = int(tables[60, last])
    assert ref[X] == 4 and w.block_fill[X] not in (0, w.block_size)
    src, dst = [], []
    for child in (60, 61, 62, 63):
        if ref[X] > 1:
            new = free.pop(0)
            src.append(X)
            dst.append(new)
            tables[child, last] = new
            ref[X] -= 1
            ref[new] = 1
    assert len(src) == 3 and ref[X] == 1
    k_host, v_host = f16_host(k_all).copy(), f16_host(v_all).copy()
    pkv.copy_blocks(k_all, v_all, _dev(src, torch.int32), _dev(dst, torch.int32))
    oracle.copy_blocks(k_host, v_host, src, dst, 1, k_host[0].size, k_host[0, 0].size)
    torch.cuda.synchronize()
    assert np.array_equal(u16(k_all), k_host.view(np.uint16))
    assert np.array_equal(u16(v_all), v_host.view(np.uint16))
    w.block_tables = tables
    bt_d = _dev(tables, torch.int32)
    cl_d = _dev(w.context_lens, torch.int32)
    seq, pos = w.new_token_positions()
    slots_d = pkv.slot_mapping(_dev(seq, torch.int32), _dev(pos, torch.int64), bt_d, w.block_size)
    orc_slots = oracle.slot_mapping(seq, pos, tables, w.block_size)
    torch.cuda.synchronize()
    assert np.array_equal(slots_d.cpu().numpy(), orc_slots)
    assert len(set(orc_slots.tolist())) == len(orc_slots)     # no child writes a shared slot
    ws = pkv.make_workspace(w.num_seqs, 1, w.num_q_heads, w.num_kv_heads)
    _check_layer(w, 0, k_all, v_all, bt_d, cl_d, slots_d, orc_slots, ws)


def _ring_step(w, k_l, v_l, bt_d, rope_d, ws, k_host, v_host, L, hw, q_len, kn, vn, q,
               fused=False):
    """Append the step's rows at their ring slots and decode: ring slot mapping + kv_append +
    ring_attn_decode, or the one fused call; the oracle replays the append on its host copy."""
    seq = np.repeat(np.arange(w.num_seqs, dtype=np.int32), q_len)
    pos = (L[:, None] - q_len + np.arange(q_len)[None, :]).reshape(-1).astype(np.int64)
    orc_slots = oracle.ring_slot_mapping(seq, pos, w.block_tables, w.sink, w.window, w.block_size)
    out = torch.empty_like(q)
    if fused:
        pkv.ring_attn_decode_append(out, q, kn, vn, k_l, v_l, bt_d, _dev(L, torch.int64),
                                    _dev(hw, torch.int64), w.sink, w.window, rope_d, w.scale, ws)
        torch.cuda.synchronize()
    else:
        slots_d = pkv.ring_slot_mapping(_dev(seq, torch.int32), _dev(pos, torch.int64), bt_d,
                                        w.sink, w.window, w.block_size)
        pkv.kv_append(kn, vn, slots_d, k_l, v_l)
        pkv.ring_attn_decode(out, q, k_l, v_l, bt_d, _dev(L, torch.int64), _dev(hw, torch.int64),
                             w.sink, w.window, rope_d, w.scale, ws)
        torch.cuda.synchronize()
        assert np.array_equal(slots_d.cpu().numpy(), orc_slots)
    oracle.kv_append(f16_host(kn), f16_host(vn), orc_slots, k_host, v_host, w.block_size)
    assert np.array_equal(u16(k_l), k_host.view(np.uint16))
    assert np.array_equal(u16(v_l), v_host.view(np.uint16))
    ref = oracle.ring_attention(f16_host(q), k_host, v_host, w.block_tables, L, hw,
                                w.block_size, w.sink, w.window, w.scale)
    return out, ref


@pytest.mark.parametrize("fused", [False, True])
def test_ring_drafts_rollback_append(fused):
    w = workloads.ring()
    k_all, v_all = w.pools(DEV)
    k_l, v_l = k_all[0], v_all[0]
    k_host, v_host = f16_host(k_l).copy(), f16_host(v_l).copy()
    bt_d = _dev(w.block_tables, torch.int32)
    rope_d = pkv.rope_table(w.sink + w.window).to(DEV)
    ws = pkv.make_workspace(w.num_seqs, 4, w.num_q_heads, w.num_kv_heads)
    L0 = w.ring_len0.astype(np.int64)
    # 4 drafts appended at L0..L0+3, decoded causally
    kn, vn = w.new_kv(0, DEV)
    q = w.query(0, DEV)
    L = L0 + 4
    hw = L.copy()
    out, ref = _ring_step(w, k_l, v_l, bt_d, rope_d, ws, k_host, v_host, L, hw, 4, kn, vn, q,
                          fused)
    assert_attn_close(out, ref, "ring drafts")
    # roll back 2 (high-water mark stays), append one token at L0 + 2, decode it
    L = L0 + 3
    kn1 = w.draw((w.num_seqs, 2, 128), 0, 100, DEV)
    vn1 = w.draw((w.num_seqs, 2, 128), 0, 101, DEV)
    q1 = w.draw((w.num_seqs, 1, 12, 128), 0, 102, DEV)
    out, ref = _ring_step(w, k_l, v_l, bt_d, rope_d, ws, k_host, v_host, L, hw, 1, kn1, vn1, q1,
                          fused)
    assert_attn_close(out, ref, "ring after rollback")


@pytest.mark.parametrize("fused", [False, True])
def test_ring_drafts_across_the_wrap_and_in_the_sinks(fused):
    """Drafts whose ring slots wrap from the window's end to its start, drafts that begin
    inside the sinks of a young sequence, and one ending right at the first wrap."""
    w = workloads.ring()
    S, W = w.sink, w.window
    L0 = w.ring_len0.astype(np.int64).copy()
    L0[:4] = [S + 10 * W + W - 2, 3, S + W - 1, 1021]
    k_all, v_all = w.pools(DEV)
    k_l, v_l = k_all[0], v_all[0]
    k_host, v_host = f16_host(k_l).copy(), f16_host(v_l).copy()
    bt_d = _dev(w.block_tables, torch.int32)
    rope_d = pkv.rope_table(S + W).to(DEV)
    ws = pkv.make_workspace(w.num_seqs, 4, w.num_q_heads, w.num_kv_heads)
    kn, vn = w.new_kv(0, DEV)
    q = w.query(0, DEV)
    out, ref = _ring_step(w, k_l, v_l, bt_d, rope_d, ws, k_host, v_host, L0 + 4, L0 + 4, 4,
                          kn, vn, q, fused)
    assert_attn_close(out, ref, "ring drafts across the wrap")


@pytest.mark.parametrize("fused", [False, True])
def test_ring_multi_layer_pool_at_layer_stride(fused):
    """The streaming step on layers 1 and 2 of a 3-layer pool (each layer's base pointer at the
    layer stride): every layer's bytes, the untouched layer 0 included, and every output."""
    w = workloads.ring(num_layers=3)
    k_all, v_all = w.pools(DEV)
    hosts = [(f16_host(k_all[l]).copy(), f16_host(v_all[l]).copy()) for l in range(3)]
    bt_d = _dev(w.block_tables, torch.int32)
    rope_d = pkv.rope_table(w.sink + w.window).to(DEV)
    ws = pkv.make_workspace(w.num_seqs, 4, w.num_q_heads, w.num_kv_heads)
    L0 = w.ring_len0.astype(np.int64)
    for layer in (1, 2):
        k_host, v_host = hosts[layer]
        kn, vn = w.new_kv(layer, DEV)
        q = w.query(layer, DEV)
        hw = L0 + 4
        out, ref = _ring_step(w, k_all[layer], v_all[layer], bt_d, rope_d, ws, k_host, v_host,
                              L0 + 4, hw, 4, kn, vn, q, fused)
        assert_attn_close(out, ref, f"ring drafts, layer {layer}")
        kn1 = w.draw((w.num_seqs, 2, 128), layer, 100, DEV)
        vn1 = w.draw((w.num_seqs, 2, 128), layer, 101, DEV)
        q1 = w.draw((w.num_seqs, 1, 12, 128), layer, 102, DEV)
        out, ref = _ring_step(w, k_all[layer], v_all[layer], bt_d, rope_d, ws, k_host, v_host,
                              L0 + 3, hw, 1, kn1, vn1, q1, fused)
        assert_attn_close(out, ref, f"ring after rollback, layer {layer}")
    for layer in range(3):
        assert np.array_equal(u16(k_all[layer]), hosts[layer][0].view(np.uint16)), layer
        assert np.array_equal(u16(v_all[layer]), hosts[layer][1].view(np.uint16)), layer


def test_ring_every_layer_of_the_benchmark_pool():
    """The benchmark's ring step through the fused calls on all 24 layers of its pool: per
    layer the 4 drafts appended and decoded, a rollback of 2, one more token appended and
    decoded; every layer's bytes and every output against the oracle."""
    w = workloads.ring(num_layers=24)
    k_all, v_all = w.pools(DEV)
    bt_d = _dev(w.block_tables, torch.int32)
    rope_d = pkv.rope_table(w.sink + w.window).to(DEV)
    ws = pkv.make_workspace(w.num_seqs, 4, w.num_q_heads, w.num_kv_heads)
    L0 = w.ring_len0.astype(np.int64)
    hw = L0 + 4
    for layer in range(w.num_layers):
        k_host, v_host = f16_host(k_all[layer]).copy(), f16_host(v_all[layer]).copy()
        kn, vn = w.new_kv(layer, DEV)
        q = w.query(layer, DEV)
        out, ref = _ring_step(w, k_all[layer], v_all[layer], bt_d, rope_d, ws, k_host, v_host,
                              L0 + 4, hw, 4, kn, vn, q, fused=True)
        assert_attn_close(out, ref, f"ring drafts, layer {layer}")
        kn1 = w.draw((w.num_seqs, 2, 128), layer, 100, DEV)
        vn1 = w.draw((w.num_seqs, 2, 128), layer, 101, DEV)
        q1 = w.draw((w.num_seqs, 1, 12, 128), layer, 102, DEV)
        out, ref = _ring_step(w, k_all[layer], v_all[layer], bt_d, rope_d, ws, k_host, v_host,
                              L0 + 3, hw, 1, kn1, vn1, q1, fused=True)
        assert_attn_close(out, ref, f"ring after rollback, layer {layer}")


# ------------------------------------------------------------------------------ invariants
def _small(lens, bs=16, hq=12, hkv=2, q_len=1, seed=0, extra_blocks=3, poison=True):
    """A hand-sized paged workload: returns (pools, tables, lens, q) as numpy + device."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    nblk = [(int(l) + bs - 1) // bs for l in lens]
    nb = sum(nblk) + extra_blocks
    maxb = max(max(nblk), 1)
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(lens), maxb), -1, dtype=np.int32)
    cur = 0
    k = rng.standard_normal((nb, hkv, bs, 128)).astype(np.float16)
    v = rng.standard_normal((nb, hkv, bs, 128)).astype(np.float16)
    used = np.zeros((nb, bs), bool)
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[cur:cur + n]
        for j in range(n):
            used[perm[cur + j], : max(0, min(bs, int(lens[b]) - j * bs))] = True
        cur += n
    if poison:
        k[~used[:, None, :, None].repeat(hkv, 1).repeat(128, 3)] = np.nan
        v[~used[:, None, :, None].repeat(hkv, 1).repeat(128, 3)] = np.nan
    q = rng.standard_normal((len(lens), q_len, hq, 128)).astype(np.float16)
    return k, v, tables, lens, q


def _gpu_decode(k, v, tables, lens, q, scale, bs=16):
    kd, vd = torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV)
    qd = torch.from_numpy(q).to(DEV)
    out = torch.empty_like(qd)
    ws = pkv.make_workspace(q.shape[0], q.shape[1], q.shape[2], k.shape[1])
    pkv.paged_attn_decode(out, qd, kd, vd, _dev(tables, torch.int32), _dev(lens, torch.int32),
                          scale, ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("lens,bs,hq,hkv,q_len", [
    ([1, 2, 15, 16, 17, 31, 33], 16, 12, 2, 1),          # ragged tails, single token
    ([1000, 3, 517], 64, 32, 32, 1),                       # MHA, 64-token blocks
    ([300, 47], 16, 64, 8, 1),                             # GQA 8
    ([77, 200, 5], 16, 12, 2, 3),                          # causal multi-query (R = 18)
    ([77, 200, 5], 16, 8, 4, 4),                           # causal, transposed tile (R = 8)
    ([33, 1, 60], 16, 4, 4, 3),                            # MHA drafts (R = 3)
    ([500, 70], 64, 16, 2, 1),                             # GQA 8, 64-token blocks
    ([129, 64], 32, 64, 8, 4),                             # R = 32, 32-token blocks
    ([20000], 16, 12, 2, 1),                               # one long sequence over many CTAs
    ([5] * 700, 16, 12, 2, 1),                             # many short sequences
    ([2, 40, 0, 9], 16, 12, 2, 1),                         # an empty sequence -> zeros
])
def test_edge_shapes(lens, bs, hq, hkv, q_len):
    k, v, tables, lens, q = _small(lens, bs, hq, hkv, q_len, seed=len(lens) + bs)
    scale = 1 / math.sqrt(128)
    out = _gpu_decode(k, v, tables, lens, q, scale, bs)
    ref = oracle.paged_attention(q, k, v, tables, lens, bs, scale)
    assert_attn_close(out, ref, f"lens={lens[:4]} bs={bs} G={hq // hkv} q_len={q_len}")


def test_block_permutation_and_sharing_are_bit_identical():
    k, v, tables, lens, q = _small([400, 1000, 33, 777], seed=5, poison=False)
    scale = 0.1
    base = _gpu_decode(k, v, tables, lens, q, scale)
    # relabel every physical block
    perm = np.random.default_rng(1).permutation(k.shape[0])
    inv = np.argsort(perm)
    t2 = np.where(tables >= 0, perm[np.maximum(tables, 0)], -1).astype(np.int32)
    out2 = _gpu_decode(k[inv], v[inv], t2, lens, q, scale)
    assert torch.equal(base, out2)
    # sequence 1 reads sequence 0's first 10 blocks as a shared prefix vs private copies
    t_sh = tables.copy()
    t_sh[1, :10] = tables[0, :10]
    k_pr, v_pr = k.copy(), v.copy()
    k_pr[tables[1, :10]] = k[tables[0, :10]]
    v_pr[tables[1, :10]] = v[tables[0, :10]]
    shared = _gpu_decode(k, v, t_sh, lens, q, scale)
    private = _gpu_decode(k_pr, v_pr, tables, lens, q, scale)
    assert torch.equal(shared, private)
    # repeated calls are deterministic
    assert torch.equal(base, _gpu_decode(k, v, tables, lens, q, scale))


def test_launch_sizes_can_shrink_and_grow_again():
    """A decode with a smaller shared-memory footprint (fewer sequences) between two larger
    ones must not break the larger launch (the kernel attribute is per kernel, not per call)."""
    scale = 0.1
    big = _small([100] * 600, seed=31, poison=False)
    small = _small([100, 7], seed=32, poison=False)
    for k, v, tables, lens, q in (big, small, big):
        out = _gpu_decode(k, v, tables, lens, q, scale)
        ref = oracle.paged_attention(q, k, v, tables, lens, 16, scale)
        assert_attn_close(out, ref, f"B={len(lens)}")


def test_single_token_context_is_v_exactly():
    k, v, tables, lens, q = _small([1, 1, 1], poison=True)
    out = _gpu_decode(k, v, tables, lens, q, 0.3)
    for b in range(3):
        vrow = torch.from_numpy(v[tables[b, 0], :, 0]).to(DEV)         # [Hkv, D]
        assert torch.equal(out[b, 0], vrow.repeat_interleave(6, 0))


# ------------------------------------------------------------------------------ guards
def test_bad_block_id_sets_error_bit_without_fault():
    k, v, tables, lens, q = _small([40, 40], poison=False)
    tables = tables.copy()
    tables[1, 1] = k.shape[0] + 5                  # out of range
    assert pkv.check_tables(torch.from_numpy(tables), torch.from_numpy(lens), 16, k.shape[0]) == 1
    _gpu_decode(k, v, tables, lens, q, 0.1)
    assert pkv.device_error(clear=True) & pkv.DEVERR_BLOCK_ID


def test_context_past_table_sets_error_bit():
    k, v, tables, lens, q = _small([40, 40], poison=False)
    lens = lens.copy()
    lens[0] = tables.shape[1] * 16 + 7
    _gpu_decode(k, v, tables, lens, q, 0.1)
    assert pkv.device_error(clear=True) & pkv.DEVERR_CONTEXT


def test_argument_errors_are_reported_before_launch():
    k, v, tables, lens, q = _small([40])
    kd, vd, qd = (torch.from_numpy(x).to(DEV) for x in (k, v, q))
    out = torch.empty_like(qd)
    small = torch.zeros(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attn_decode(out, qd, kd, vd, _dev(tables, torch.int32), _dev(lens, torch.int32),
                              0.1, small)
    assert e.value.status == pkv.ENOSPC
    ws = pkv.make_workspace(1, 1, 12, 2)
    with pytest.raises(pkv.PkvError) as e:           # head_dim 64 is not supported
        pkv.paged_attn_decode(out[..., :64], qd[..., :64], kd[..., :64], vd[..., :64],
                              _dev(tables, torch.int32), _dev(lens, torch.int32), 0.1, ws)
    assert e.value.status == pkv.EINVAL


def test_append_skips_negative_and_flags_out_of_range_slots():
    k = torch.zeros((4, 2, 16, 128), dtype=torch.float16, device=DEV)
    v = torch.zeros_like(k)
    kn = torch.ones((3, 2, 128), dtype=torch.float16, device=DEV)
    slots = torch.tensor([-1, 5, 4 * 16 + 3], dtype=torch.int64, device=DEV)
    pkv.kv_append(kn, kn, slots, k, v)
    torch.cuda.synchronize()
    assert k.sum().item() == 2 * 128 and k[0, :, 5].eq(1).all()
    assert pkv.device_error(clear=True) & pkv.DEVERR_SLOT
