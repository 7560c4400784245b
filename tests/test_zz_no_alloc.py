"""Decode for callers that cannot allocate device memory.

pkv_paged_attn_decode_noalloc takes its scratch from a fixed array inside the library instead
of a caller workspace, for code that runs where it may not allocate (under a framework that
owns all device memory, in a fixed-budget embedded runtime). These tests call it through the
C ABI and check it against the workspace entry point on the same inputs, twice in a row (the
array keeps the previous call's contents, so the second call also checks that the library
clears what must start at zero). This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_147_gb300 import pkv, workloads

from _util import ATOL, assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs():
    w = workloads.edge_1p1b(num_layers=1)
    k, v = w.pools(DEV)
    bt = torch.as_tensor(w.block_tables, device=DEV)
    cl = torch.as_tensor(w.context_lens, device=DEV)
    return w, k[0], v[0], bt, cl


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    w, k, v, bt, cl = _inputs()
    for call in range(2):
        q = w.draw((w.num_seqs, 1, w.num_q_heads, w.head_dim), 0, 200 + call, DEV)
        ws = pkv.make_workspace(w.num_seqs, 1, w.num_q_heads, w.num_kv_heads, DEV)
        ref = torch.empty_like(q)
        pkv.paged_attn_decode(ref, q, k, v, bt, cl, w.scale, ws)
        out = torch.full_like(q, float("nan"))
        pkv.paged_attn_decode_noalloc(out, q, k, v, bt, cl, w.scale)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all(), f"call {call}: non-finite output"
        diff = (out.float() - ref.float()).abs().max().item()
        assert diff <= ATOL, f"call {call}: max |noalloc - workspace| = {diff}"
    assert pkv.device_error(clear=True) == 0


def test_noalloc_rejects_requests_beyond_its_fixed_array():
    w, k, v, bt, cl = _inputs()
    # 64 query heads over 2 kv heads with 1 token: 32 rows per unit needs more than 8 MiB
    q = torch.zeros((w.num_seqs, 1, 64, 128), dtype=torch.float16, device=DEV)
    out = torch.empty_like(q)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attn_decode_noalloc(out, q, k, v, bt, cl, w.scale)
    assert e.value.status == pkv.ENOSPC
