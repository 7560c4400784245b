"""Both ways a split unit can be merged give the same bits.

A unit cut by slice boundaries is normally merged by the CTA holding its first chunk, which
waits (for a bounded time) until the unit's other partials are in. When the wait runs out,
that CTA announces its own partial like the others and the last CTA to arrive merges
instead. A build of the library with no wait budget takes the second way whenever the other
partials are not already in, so comparing it with the default build checks that the two
paths produce bit-identical outputs (the partials and their order are the same).
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from paged_kv_cache_147_gb300 import build, pkv, workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def nowait_lib():
    out = os.path.join(os.path.dirname(build.LIB), "_variants", "libpkv_nowait.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    build.build(defines=["PKV_MERGE_WAIT_NS=0"], out=out)
    return pkv.load_variant(out)


def _decode(lib, out, q, k, v, bt, cl, scale, ws):
    B, q_len, hq, d = q.shape
    nb, hkv, bs, _ = k.shape
    status = lib.pkv_paged_attn_decode(
        pkv._p(out), pkv._p(q), pkv._p(k), pkv._p(v), nb, pkv._p(bt), bt.shape[1], pkv._p(cl),
        B, q_len, hq, hkv, d, bs, float(scale), pkv._p(ws), ws.numel() * ws.element_size(),
        pkv._stream())
    assert status == pkv.OK


def _device_error(lib) -> int:
    word = ctypes.c_uint(0)
    assert lib.pkv_device_error(ctypes.byref(word), 1, pkv._stream()) == pkv.OK
    return word.value


@pytest.mark.parametrize("name", ["edge_1p1b", "llama70b_mixed"])
def test_merge_without_wait_matches_default_bitwise(nowait_lib, name):
    w = workloads.WORKLOADS[name](num_layers=3)
    k, v = w.pools(DEV)
    bt = torch.as_tensor(w.block_tables, device=DEV)
    cl = torch.as_tensor(w.context_lens, device=DEV)
    ws_a = pkv.make_workspace(w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads, DEV)
    ws_b = pkv.make_workspace(w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads, DEV)
    default = pkv.load()
    for layer in range(w.num_layers):
        q = w.query(layer, DEV)
        ref = torch.empty_like(q)
        _decode(default, ref, q, k[layer], v[layer], bt, cl, w.scale, ws_a)
        for rep in range(3):
            out = torch.full_like(q, float("nan"))
            _decode(nowait_lib, out, q, k[layer], v[layer], bt, cl, w.scale, ws_b)
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), \
                f"{name} layer {layer} call {rep}: outputs differ"
    assert _device_error(default) == 0
    assert _device_error(nowait_lib) == 0
