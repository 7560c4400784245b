"""The fused append + decode after a kernel that writes its inputs.

By default pkv_paged_attn_decode_append may start while the kernel ahead of it finishes and
reads the pools, block tables and context lengths early. A serving loop that advances the
context lengths with its own device op, or that copies a shared block (copy-on-write) right
before the fused call, must switch that overlap off (pkv_set_early_start(0)); these tests run
exactly those orderings with the overlap off and hold the results to the oracle.
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


@pytest.fixture()
def no_early_start():
    prev = pkv.set_early_start(False)
    assert pkv.set_early_start(False) is False        # the call returns the previous setting
    yield
    pkv.set_early_start(prev)
    assert pkv.device_error(clear=True) == 0


def test_context_lengths_advanced_on_device_right_before_the_fused_call(no_early_start):
    w = workloads.edge_1p1b(num_layers=1)
    k, v = w.pools(DEV, poison=True)
    k_host, v_host = f16_host(k[0]).copy(), f16_host(v[0]).copy()
    bt = torch.as_tensor(w.block_tables, device=DEV)
    # the lengths before the step, advanced by a torch kernel on the same stream, then the
    # fused call with no other launch in between
    cl = torch.as_tensor(w.context_lens - 1, device=DEV)
    q = w.query(0, DEV)
    kn, vn = w.new_kv(0, DEV)
    ws = pkv.make_workspace(w.num_seqs, 1, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(q)
    torch.cuda.synchronize()
    cl.add_(1)
    pkv.paged_attn_decode_append(out, q, kn, vn, k[0], v[0], bt, cl, w.scale, ws)
    torch.cuda.synchronize()
    seq, pos = w.new_token_positions()
    slots = oracle.slot_mapping(seq, pos, w.block_tables, w.block_size)
    oracle.kv_append(f16_host(kn), f16_host(vn), slots, k_host, v_host, w.block_size)
    assert np.array_equal(u16(k[0]), k_host.view(np.uint16))
    assert np.array_equal(u16(v[0]), v_host.view(np.uint16))
    ref = oracle.paged_attention(f16_host(q), k_host, v_host, w.block_tables, w.context_lens,
                                 w.block_size, w.scale)
    assert_attn_close(out, ref, "lengths advanced on the device")


def test_copy_on_write_right_before_the_fused_call(no_early_start):
    w = workloads.prefix()
    k, v = w.pools(DEV, poison=True)
    tables = w.block_tables.copy()
    last = (int(w.context_lens[60]) - 1) // w.block_size
    shared = int(tables[60, last])
    src, dst = [], []
    for child, spare in zip((60, 61, 62), w.free_blocks[:3]):
        tables[child, last] = int(spare)
        src.append(shared)
        dst.append(int(spare))
    k_host, v_host = f16_host(k[0]).copy(), f16_host(v[0]).copy()
    q = w.query(0, DEV)
    kn, vn = w.new_kv(0, DEV)
    bt = torch.as_tensor(tables, device=DEV)
    cl = torch.as_tensor(w.context_lens, device=DEV)
    ws = pkv.make_workspace(w.num_seqs, 1, w.num_q_heads, w.num_kv_heads)
    out = torch.empty_like(q)
    src_d = torch.tensor(src, dtype=torch.int32, device=DEV)
    dst_d = torch.tensor(dst, dtype=torch.int32, device=DEV)
    torch.cuda.synchronize()
    pkv.copy_blocks(k, v, src_d, dst_d)
    pkv.paged_attn_decode_append(out, q, kn, vn, k[0], v[0], bt, cl, w.scale, ws)
    torch.cuda.synchronize()
    oracle.copy_blocks(k_host[None], v_host[None], src, dst, 1, k_host.size, k_host[0].size)
    seq, pos = w.new_token_positions()
    slots = oracle.slot_mapping(seq, pos, tables, w.block_size)
    oracle.kv_append(f16_host(kn), f16_host(vn), slots, k_host, v_host, w.block_size)
    assert np.array_equal(u16(k[0]), k_host.view(np.uint16))
    assert np.array_equal(u16(v[0]), v_host.view(np.uint16))
    ref = oracle.paged_attention(f16_host(q), k_host, v_host, tables, w.context_lens,
                                 w.block_size, w.scale)
    assert_attn_close(out, ref, "copy-on-write then fused append + decode")


def test_fp8_fused_call_after_lengths_advanced_on_device(no_early_start):
    """The E4M3 fused append + decode right after a torch kernel advances the lengths."""
    rng = np.random.default_rng(21)
    lens = np.array([37, 100, 16, 1, 250], np.int32)         # after this step's append
    bs, hq, hkv = 16, 12, 2
    nblk = [(int(L) + bs - 1) // bs for L in lens]
    nb = sum(nblk) + 2
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(lens), max(nblk)), -1, np.int32)
    cur = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[cur:cur + n]
        cur += n
    kf = rng.standard_normal((nb, hkv, bs, 128)).astype(np.float32)
    vf = rng.standard_normal((nb, hkv, bs, 128)).astype(np.float32)
    ks = (np.abs(kf).max(axis=(0, 2, 3)) / 448.0).astype(np.float32)
    vs = (np.abs(vf).max(axis=(0, 2, 3)) / 448.0).astype(np.float32)
    k8 = torch.from_numpy(kf / ks[None, :, None, None]).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    v8 = torch.from_numpy(vf / vs[None, :, None, None]).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    q = rng.standard_normal((len(lens), 1, hq, 128)).astype(np.float16)
    kn = rng.standard_normal((len(lens), hkv, 128)).astype(np.float16)
    vn = rng.standard_normal((len(lens), hkv, 128)).astype(np.float16)
    k8_d, v8_d = torch.from_numpy(k8).to(DEV), torch.from_numpy(v8).to(DEV)
    qd, knd, vnd = (torch.from_numpy(x).to(DEV) for x in (q, kn, vn))
    ks_d, vs_d = torch.from_numpy(ks).to(DEV), torch.from_numpy(vs).to(DEV)
    bt = torch.from_numpy(tables).to(DEV)
    cl = torch.from_numpy(lens - 1).to(DEV)
    ws = pkv.make_workspace(len(lens), 1, hq, hkv)
    out = torch.empty_like(qd)
    scale = 1 / math.sqrt(128)
    torch.cuda.synchronize()
    cl.add_(1)
    pkv.paged_attn_decode_append_fp8(out, qd, knd, vnd, k8_d, v8_d, ks_d, vs_d, bt, cl, scale, ws)
    torch.cuda.synchronize()
    seq = np.arange(len(lens), dtype=np.int32)
    slots = oracle.slot_mapping(seq, (lens - 1).astype(np.int64), tables, bs)
    oracle.kv_append_fp8(kn, vn, slots, k8, v8, bs, ks, vs)
    assert np.array_equal(k8_d.cpu().numpy(), k8) and np.array_equal(v8_d.cpu().numpy(), v8)
    ref = oracle.paged_attention_fp8(q, k8, v8, ks, vs, tables, lens, bs, scale)
    assert_attn_close(out, ref, "fp8 fused after lengths advanced on the device")
