"""GPU: a prefix-sharing batch whose block tables, forks and copy-on-write pairs come from the
library's host block pool, run through the CUDA entry points and checked against the oracle.

64 MHA sequences (32 heads, 64-token blocks) begin with the same 256-token system prompt, so
the pool hands all of them the same four blocks. Four children of a parent whose last block is
partly filled then append one token each: the pool returns a copy pair for each child that
still shares that block (three of them), pkv_copy_blocks copies them, and the fused append +
decode writes and attends. The oracle replays the copies and the append on host pools.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_147_gb300 import pkv

from _util import assert_attn_close, f16_host, u16

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(a, dtype):
    return torch.as_tensor(np.ascontiguousarray(a), dtype=dtype, device=DEV)


def test_pool_driven_prefix_batch_with_fork_and_copy_on_write():
    rng = np.random.default_rng(21)
    bs, hq, hkv, n_seq = 64, 32, 32, 64
    system = list(rng.integers(0, 32000, 256))
    pool = pkv.BlockPool(1200, bs)
    tables, lens, reused = [], [], []
    for b in range(60):
        prompt = system + list(rng.integers(0, 32000, rng.integers(32, 1025)))
        t, r = pool.allocate(prompt, len(prompt) + 1)      # room for this step's token
        tables.append(t)
        lens.append(len(prompt))
        reused.append(r)
    assert reused[0] == 0 and all(r == 4 for r in reused[1:])
    parent_prompt = system + list(rng.integers(0, 32000, 301))   # last block partly filled
    parent, _ = pool.allocate(parent_prompt)
    kids = [pool.fork(parent) for _ in range(4)]
    pool.release(parent)
    assert pool.refcount(parent[0]) == 64 and pool.refcount(parent[-1]) == 4
    copies = []
    for i, k in enumerate(kids):
        t, c = pool.append(k, len(parent_prompt), 1)
        kids[i] = t
        copies.extend(map(tuple, c.tolist()))
    assert len(copies) == 3 and all(s == parent[-1] for s, _ in copies)
    tables += kids
    lens += [len(parent_prompt)] * 4
    lens = np.asarray(lens, np.int32) + 1                # context after this step's token
    maxb = max(len(t) for t in tables)
    bt = np.full((n_seq, maxb), -1, np.int32)
    for b, t in enumerate(tables):
        bt[b, :len(t)] = t
    # every sequence's new slot is its own: no shared block is written
    slots = oracle.slot_mapping(np.arange(n_seq, dtype=np.int32), lens.astype(np.int64) - 1,
                                bt, bs)
    assert len(set(slots.tolist())) == n_seq and all(pool.refcount(int(s) // bs) == 1
                                                     for s in slots)

    nb = pool.num_blocks
    k = torch.randn((nb, hkv, bs, 128), device=DEV).half()
    v = torch.randn((nb, hkv, bs, 128), device=DEV).half()
    k_host, v_host = f16_host(k).copy(), f16_host(v).copy()
    src = np.array([s for s, _ in copies], np.int32)
    dst = np.array([d for _, d in copies], np.int32)
    pkv.copy_blocks(k, v, _dev(src, torch.int32), _dev(dst, torch.int32))
    oracle.copy_blocks(k_host, v_host, src, dst, 1, k_host.size, k_host[0].size)

    q = torch.randn((n_seq, 1, hq, 128), device=DEV).half()
    kn = torch.randn((n_seq, hkv, 128), device=DEV).half()
    vn = torch.randn((n_seq, hkv, 128), device=DEV).half()
    out = torch.empty_like(q)
    ws = pkv.make_workspace(n_seq, 1, hq, hkv)
    scale = 1 / math.sqrt(128)
    pkv.paged_attn_decode_append(out, q, kn, vn, k, v, _dev(bt, torch.int32),
                                 _dev(lens, torch.int32), scale, ws)
    torch.cuda.synchronize()
    assert pkv.device_error(clear=True) == 0
    oracle.kv_append(f16_host(kn), f16_host(vn), slots, k_host, v_host, bs)
    assert np.array_equal(u16(k), k_host.view(np.uint16))
    assert np.array_equal(u16(v), v_host.view(np.uint16))
    ref = oracle.paged_attention(f16_host(q), k_host, v_host, bt, lens, bs, scale)
    assert_attn_close(out, ref, "pool-driven prefix batch")
    pool.close()
