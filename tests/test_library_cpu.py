"""CPU checks of the C-ABI library: it builds, loads, and exports every symbol the header
declares; its host-only entry points (validation, RoPE table) behave as documented. No
entry point that launches work on a GPU is called here."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from paged_kv_cache_147_gb300 import build, pkv, workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pkv.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_0-9]+)\s*\(", text)))


def test_header_symbols_are_exported(lib):
    declared = _declared()
    assert len(declared) >= 13
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(pkv.SYMBOLS) == declared


def test_version(lib):
    assert pkv.version() >= 100


def test_check_tables(lib):
    tables = torch.tensor([[3, 1, -1], [0, 2, 4]], dtype=torch.int32)
    assert pkv.check_tables(tables, torch.tensor([20, 48]), 16, 5) is None
    assert pkv.check_tables(tables, torch.tensor([40, 48]), 16, 5) == 0     # reads entry -1
    assert pkv.check_tables(tables, torch.tensor([20, 49]), 16, 5) == 1     # past the table
    assert pkv.check_tables(tables, torch.tensor([20, 48]), 16, 4) == 1     # id 4 >= 4 blocks
    assert pkv.check_tables(tables, torch.tensor([-1, 0]), 16, 5) == 0


def test_check_slots(lib):
    assert pkv.check_slots(torch.tensor([-1, 0, 5, -1, 79]), 5, 16) is None
    assert pkv.check_slots(torch.tensor([0, 5, 5]), 5, 16) == 2             # duplicate
    assert pkv.check_slots(torch.tensor([0, 80]), 5, 16) == 1               # past the pool


def test_rope_table_matches_fp64_angles(lib):
    t = pkv.rope_table(1024, 128, 10000.0).numpy()
    j = np.arange(1024, dtype=np.float64)[:, None]
    theta = 10000.0 ** (-2.0 * np.arange(64) / 128)
    assert np.array_equal(t[..., 0], np.cos(j * theta).astype(np.float32))
    assert np.array_equal(t[..., 1], np.sin(j * theta).astype(np.float32))


def test_invalid_host_arguments(lib):
    bad = ctypes.c_int(0)
    assert lib.pkv_check_tables(None, None, -1, 1, 16, 1, ctypes.byref(bad)) == pkv.EINVAL
    assert lib.pkv_rope_table(None, 4, 128, 10000.0) == pkv.EINVAL
    assert lib.pkv_decode_workspace_bytes(4, 1, 12, 5, 128) == 0            # 12 % 5 != 0


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_workload_structure(name):
    w = workloads.WORKLOADS[name]()
    nb = w.num_blocks
    used = w.block_tables[w.block_tables >= 0]
    assert used.max() < nb and used.min() >= 0
    assert (w.context_lens >= 1).all()
    if name in ("tiny", "edge_1p1b", "llama70b_b16", "llama70b_mixed"):
        assert len(np.unique(used)) == len(used)              # private blocks only
        for b in range(w.num_seqs):
            n = int(np.count_nonzero(w.block_tables[b] >= 0))
            assert n == (int(w.context_lens[b]) + w.block_size - 1) // w.block_size
            assert w.block_fill[w.block_tables[b, :n]].sum() == w.context_lens[b] - w.q_len
    if name == "prefix":
        assert (w.block_tables[:, :4] == w.block_tables[0, :4]).all()
        assert (w.refcount[w.block_tables[0, :4]] == 64).all()
    if name == "ring":
        assert w.block_tables.shape[1] * w.block_size == w.sink + w.window
        assert (w.ring_len0 >= 2000).all() and (w.ring_len0 <= 100000).all()


def test_new_entry_points_reject_bad_arguments_before_any_launch(lib):
    # argument checks run on the host before any CUDA call, so they are testable here
    n, t = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.pkv_spec_verify(None, None, None, None, None, -1, 4, 100, None, None,
                               None) == pkv.EINVAL
    assert lib.pkv_spec_verify(None, None, None, None, None, 4, 4, 0, None, None,
                               None) == pkv.EINVAL
    assert lib.pkv_spec_verify(None, None, None, None, None, 0, 4, 100, None, None,
                               None) == pkv.OK                      # nothing to do
    assert lib.pkv_kv_append_fp8(None, None, None, 4, None, None, 8, 2, 128, 16, None, None,
                                 None) == pkv.EINVAL                # no pointers, no scales
    assert lib.pkv_kv_append_fp8(None, None, None, 1, None, None, 8, 2, 128, 24, None, None,
                                 None) == pkv.EINVAL                # block size 24
    assert lib.pkv_paged_attn_decode_fp8(None, None, None, None, None, None, 8, None, 4, None,
                                         2, 1, 12, 2, 128, 16, 0.1, None, 0,
                                         None) == pkv.EINVAL        # scales missing
    assert lib.pkv_paged_attn_decode_append_fp8(None, None, None, None, None, None, None, None,
                                                8, None, 4, None, 2, 1, 12, 2, 128, 16, 0.1,
                                                None, 0, None) == pkv.EINVAL
    assert lib.pkv_pool_create(0, 16, 64, None) == pkv.EINVAL
    assert lib.pkv_pool_stats(None, None, None, None, None, None) == pkv.EINVAL
