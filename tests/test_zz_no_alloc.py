"""Decode for callers that cannot allocate device memory.

pkv_paged_attn_decode_noalloc takes its scratch from a fixed array inside the library instead
of a caller workspace, for code that runs where it may not allocate (under a framework that
owns all device memory, in a fixed-budget embedded runtime). These tests call it through the
C ABI and check it against the workspace entry point on the same inputs, twice in a row (the
array keeps the previous call's contents, so the second call also checks that the library
clears what must start at zero). Both entry points run the same kernel on the same grid with
the same merge order, so their outputs must be equal bit for bit; one call is also held to the
oracle. This file is collected last on purpose.
"""
import pytest
import torch

import oracle
from paged_kv_cache_147_gb300 import pkv, workloads

from _util import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
FIXED_BYTES = 8 << 20


def _inputs():
    w = workloads.edge_1p1b(num_layers=1)
    k, v = w.pools(DEV)
    bt = torch.as_tensor(w.block_tables, device=DEV)
    cl = torch.as_tensor(w.context_lens, device=DEV)
    return w, k[0], v[0], bt, cl


def _fits(R, num_seqs, hkv, sms):
    """The fixed array's size rule as the header states it."""
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    return up(4 * num_seqs * hkv) + up(8 * sms * R * 16) + up(8 * sms * R * 512) <= FIXED_BYTES


def _both(w, k, v, bt, cl, hq, tag):
    q = w.draw((w.num_seqs, 1, hq, w.head_dim), 0, tag, DEV)
    ws = pkv.make_workspace(w.num_seqs, 1, hq, w.num_kv_heads, DEV)
    ref = torch.empty_like(q)
    pkv.paged_attn_decode(ref, q, k, v, bt, cl, w.scale, ws)
    out = torch.full_like(q, float("nan"))
    pkv.paged_attn_decode_noalloc(out, q, k, v, bt, cl, w.scale)
    torch.cuda.synchronize()
    return q, out, ref


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    w, k, v, bt, cl = _inputs()
    for call in range(2):
        q, out, ref = _both(w, k, v, bt, cl, w.num_q_heads, 200 + call)
        assert torch.equal(out, ref), f"call {call}: noalloc output differs from the workspace one"
        if call == 0:
            want = oracle.paged_attention(q.cpu(), k.cpu(), v.cpu(), w.block_tables,
                                          w.context_lens, w.block_size, w.scale)
            assert_attn_close(out, want, "noalloc vs oracle")
    assert pkv.device_error(clear=True) == 0


def test_noalloc_size_limit_is_the_documented_one():
    w, k, v, bt, cl = _inputs()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # rows per unit R = query heads per kv head here (one query token)
    r_max = max(R for R in range(1, 33) if _fits(R, w.num_seqs, w.num_kv_heads, sms))
    q, out, ref = _both(w, k, v, bt, cl, r_max * w.num_kv_heads, 300)
    assert torch.equal(out, ref), f"R={r_max}: noalloc output differs"
    if r_max < 32:
        hq = (r_max + 1) * w.num_kv_heads
        q = torch.zeros((w.num_seqs, 1, hq, 128), dtype=torch.float16, device=DEV)
        with pytest.raises(pkv.PkvError) as e:
            pkv.paged_attn_decode_noalloc(torch.empty_like(q), q, k, v, bt, cl, w.scale)
        assert e.value.status == pkv.ENOSPC
    assert pkv.device_error(clear=True) == 0


def test_noalloc_rejects_bad_shapes_even_for_an_empty_batch():
    lib = pkv.load()
    # num_seqs 0 with head_dim 64: the same EINVAL as the workspace entry point
    st = lib.pkv_paged_attn_decode_noalloc(None, None, None, None, 1, None, 1, None, 0, 1, 8, 2,
                                           64, 16, 1.0, None)
    assert st == pkv.EINVAL
    st = lib.pkv_paged_attn_decode_noalloc(None, None, None, None, 1, None, 1, None, 0, 1, 8, 2,
                                           128, 16, 1.0, None)
    assert st == pkv.OK
