"""GPU parity of chunked-prefill attention (pkv_paged_prefill, tcgen05) against the fp64 oracle.

Each case appends the chunk's K/V rows to a NaN-poisoned paged pool (pkv_kv_append, checked
byte for byte), runs the prefill through the C ABI and holds every output to the oracle's
causal paged attention within the parity bar. Lengths are ragged so that chunks start and end
inside blocks and inside the kernel's 64-key tiles; one sequence is shorter than its chunk.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_147_gb300 import pkv, workloads

from _util import assert_attn_close, f16_host, u16

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_device_error():
    pkv.device_error(clear=True)
    yield
    assert pkv.device_error(clear=True) == 0, "a kernel bounds guard fired"


def _append_chunk(w, k, v):
    """The chunk's rows into the pools (GPU) and into host copies (oracle); returns the host
    pools after the append and the chunk's queries."""
    k_host, v_host = f16_host(k[0]).copy(), f16_host(v[0]).copy()
    bt = torch.as_tensor(w.block_tables, device=DEV)
    seq, pos = w.new_token_positions()
    slots = pkv.slot_mapping(torch.as_tensor(seq, device=DEV), torch.as_tensor(pos, device=DEV),
                             bt, w.block_size)
    kn, vn = w.new_kv(0, DEV)
    pkv.kv_append(kn, vn, slots, k[0], v[0])
    orc_slots = oracle.slot_mapping(seq, pos, w.block_tables, w.block_size)
    oracle.kv_append(f16_host(kn), f16_host(vn), orc_slots, k_host, v_host, w.block_size)
    torch.cuda.synchronize()
    assert np.array_equal(slots.cpu().numpy(), orc_slots)
    assert np.array_equal(u16(k[0]), k_host.view(np.uint16))
    assert np.array_equal(u16(v[0]), v_host.view(np.uint16))
    return k_host, v_host, bt


def _prefill(w, k, v, bt, q):
    out = torch.full_like(q, float("nan"))
    cl = torch.as_tensor(w.context_lens, device=DEV)
    pkv.paged_prefill(out, q, k[0], v[0], bt, cl, w.scale)
    torch.cuda.synchronize()
    return out


CASES = [
    # (seed, lens after the chunk, q_len, Hq, Hkv, block size)
    (1, [100, 37, 16, 5], 16, 12, 2, 16),          # G 6, q_len 16, one context below q_len
    (2, [300, 129, 1000, 200], 128, 16, 2, 16),    # G 8, q_len 128
    (3, [1500, 513, 777], 512, 12, 2, 64),         # G 6, q_len 512, 64-token blocks
    (4, [4096, 700], 512, 16, 2, 16),              # G 8, q_len 512, long context
    (5, [333, 130], 128, 64, 8, 16),               # 70B head shape, 8 kv heads
    (6, [250, 71], 200, 4, 4, 32),                 # MHA (G 1), 128-token query tiles
    (7, [95, 64], 40, 32, 2, 16),                  # G 16: 8 tokens per tile
]


@pytest.mark.parametrize("seed,lens,q_len,hq,hkv,bs", CASES)
def test_prefill_matches_oracle(seed, lens, q_len, hq, hkv, bs):
    w = workloads.prefill(seed, lens, q_len, hq, hkv, bs)
    k, v = w.pools(DEV, poison=True)
    k_host, v_host, bt = _append_chunk(w, k, v)
    q = w.query(0, DEV)
    out = _prefill(w, k, v, bt, q)
    ref = oracle.paged_attention(f16_host(q), k_host, v_host, w.block_tables, w.context_lens,
                                 w.block_size, w.scale)
    assert_attn_close(out, ref, f"prefill q_len={q_len} G={hq // hkv} bs={bs}")


def test_prefill_is_deterministic_and_independent_of_block_placement():
    w = workloads.prefill(8, [700, 300, 129], 128, 16, 2, 16)
    k, v = w.pools(DEV, poison=True)
    _, _, bt = _append_chunk(w, k, v)
    q = w.query(0, DEV)
    a = _prefill(w, k, v, bt, q)
    b = _prefill(w, k, v, bt, q)
    assert torch.equal(a, b)
    # move every block to another physical id (a permutation of the pool) and relabel the
    # tables: the same logical cache, so the same bits
    perm = np.random.default_rng(9).permutation(w.num_blocks)
    k2, v2 = torch.empty_like(k), torch.empty_like(v)
    idx = torch.as_tensor(perm, device=DEV)
    k2[0, idx] = k[0]
    v2[0, idx] = v[0]
    tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    w.block_tables = tables
    c = _prefill(w, k2, v2, torch.as_tensor(tables, device=DEV), q)
    assert torch.equal(a, c)


def test_prefill_single_token_chunk_equals_decode():
    # a chunk of one token is a decode step: the tensor-core path and the decode kernel agree
    # within the parity bar of each against the oracle
    w = workloads.prefill(10, [517, 1, 64], 1, 12, 2, 16)
    k, v = w.pools(DEV, poison=True)
    k_host, v_host, bt = _append_chunk(w, k, v)
    q = w.query(0, DEV)
    out = _prefill(w, k, v, bt, q)
    ref = oracle.paged_attention(f16_host(q), k_host, v_host, w.block_tables, w.context_lens,
                                 w.block_size, w.scale)
    assert_attn_close(out, ref, "prefill q_len=1")


def test_prefill_bad_block_id_sets_the_error_bit_without_fault():
    # a table entry past the pool: that block reads as zeros (an out-of-range box), the
    # block-id bit is set, and the other sequence's outputs are unaffected
    w = workloads.prefill(11, [300, 129], 128, 16, 2, 16)
    k, v = w.pools(DEV, poison=True)
    k_host, v_host, _ = _append_chunk(w, k, v)
    tables = w.block_tables.copy()
    tables[1, 2] = w.num_blocks + 7
    q = w.query(0, DEV)
    out = torch.full_like(q, float("nan"))
    pkv.paged_prefill(out, q, k[0], v[0], torch.as_tensor(tables, device=DEV),
                      torch.as_tensor(w.context_lens, device=DEV), w.scale)
    torch.cuda.synchronize()
    assert pkv.device_error(clear=True) & pkv.DEVERR_BLOCK_ID
    assert torch.isfinite(out[1]).all()
    ref = oracle.paged_attention(f16_host(q), k_host, v_host, w.block_tables, w.context_lens,
                                 w.block_size, w.scale)
    assert_attn_close(out[:1], ref[:1], "prefill beside a sequence with a bad block id")


def test_prefill_context_past_the_table_is_clamped_and_flagged():
    w = workloads.prefill(12, [100, 60], 32, 12, 2, 16)
    k, v = w.pools(DEV, poison=True)
    k_host, v_host, bt = _append_chunk(w, k, v)
    lens = w.context_lens.copy()
    lens[1] = w.block_tables.shape[1] * w.block_size + 50      # past the end of its table
    q = w.query(0, DEV)
    out = torch.full_like(q, float("nan"))
    pkv.paged_prefill(out, q, k[0], v[0], bt, torch.as_tensor(lens, device=DEV), w.scale)
    torch.cuda.synchronize()
    assert pkv.device_error(clear=True) & pkv.DEVERR_CONTEXT
    ref = oracle.paged_attention(f16_host(q), k_host, v_host, w.block_tables, w.context_lens,
                                 w.block_size, w.scale)
    assert_attn_close(out[:1], ref[:1], "prefill beside a sequence whose context is clamped")
