"""GPU parity of the FP8 (E4M3) KV cache through the C ABI.

The append's pool bytes must equal the oracle's E4M3 rounding of x / scale (every byte, the
untouched ones included); decode attention over an E4M3 cache must be within the attention
bar of tests/_util.py of the fp64 oracle over the dequantised cache. Caches are built on the
host (torch's CPU float8 conversion of seeded normal data), never by the CUDA path.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_147_gb300 import pkv, workloads

from _util import assert_attn_close, f16_host

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(a, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(a))
    return t.to(DEV) if dtype is None else t.to(device=DEV, dtype=dtype)


def _quantise(x, scale):
    """fp32 data [NB, Hkv, bs, D] -> E4M3 codes with per-kv-head scales (host, torch CPU)."""
    y = torch.from_numpy(x / scale[None, :, None, None]).clamp(-448.0, 448.0)
    return y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _fp8_case(lens, bs=16, hq=12, hkv=2, q_len=1, seed=0, extra_blocks=3):
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    nblk = [(int(l) + bs - 1) // bs for l in lens]
    nb = sum(nblk) + extra_blocks
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(lens), max(max(nblk), 1)), -1, dtype=np.int32)
    used = np.zeros((nb, bs), bool)
    cur = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[cur:cur + n]
        for j in range(n):
            used[perm[cur + j], : max(0, min(bs, int(lens[b]) - j * bs))] = True
        cur += n
    kf = rng.standard_normal((nb, hkv, bs, 128)).astype(np.float32)
    vf = rng.standard_normal((nb, hkv, bs, 128)).astype(np.float32)
    ks = (np.abs(kf).max(axis=(0, 2, 3)) / 448.0 * rng.uniform(1.0, 3.0, hkv)).astype(np.float32)
    vs = (np.abs(vf).max(axis=(0, 2, 3)) / 448.0 * rng.uniform(1.0, 3.0, hkv)).astype(np.float32)
    k8, v8 = _quantise(kf, ks), _quantise(vf, vs)
    # slots no sequence may read hold NaN codes: any read of them shows in the output
    mask = ~used[:, None, :, None].repeat(hkv, 1).repeat(128, 3)
    k8[mask] = 0x7F
    v8[mask] = 0xFF
    q = rng.standard_normal((len(lens), q_len, hq, 128)).astype(np.float16)
    return k8, v8, ks, vs, tables, lens, q


def _gpu_decode_fp8(k8, v8, ks, vs, tables, lens, q, scale):
    qd = _dev(q)
    out = torch.empty_like(qd)
    ws = pkv.make_workspace(q.shape[0], q.shape[1], q.shape[2], k8.shape[1])
    pkv.paged_attn_decode_fp8(out, qd, _dev(k8), _dev(v8), _dev(ks), _dev(vs),
                              _dev(tables, torch.int32), _dev(lens, torch.int32), scale, ws)
    torch.cuda.synchronize()
    assert pkv.device_error(clear=True) == 0
    return out


@pytest.mark.parametrize("hkv,T", [(2, 40), (8, 33)])
def test_kv_append_fp8_bytes_equal_the_oracle(hkv, T):
    rng = np.random.default_rng(hkv * 100 + T)
    nb, bs = 9, 16
    k = (rng.standard_normal((T, hkv, 128)) * 2).astype(np.float16)
    v = (rng.standard_normal((T, hkv, 128)) * 2).astype(np.float16)
    # exact ties of the rounding, values that saturate, signed zeros and subnormals
    k[0, 0, :6] = np.array([1.0625, 1.1875, -1.0625, 1000.0, -1000.0, -0.0], np.float16)
    v[0, 0, :4] = np.array([2.0 ** -10, -(2.0 ** -10), 1.5 * 2.0 ** -10, 3.0 * 2.0 ** -11],
                           np.float16)
    ks = rng.uniform(0.01, 0.6, hkv).astype(np.float32)
    vs = rng.uniform(0.01, 0.6, hkv).astype(np.float32)
    ks[0] = vs[0] = 1.0
    slots = rng.choice(nb * bs, size=T, replace=False).astype(np.int64)
    slots[3] = -1
    kc = rng.integers(0, 256, (nb, hkv, bs, 128), dtype=np.uint8)
    vc = rng.integers(0, 256, (nb, hkv, bs, 128), dtype=np.uint8)
    kc_d, vc_d = _dev(kc), _dev(vc)
    pkv.kv_append_fp8(_dev(k), _dev(v), _dev(slots), kc_d, vc_d, _dev(ks), _dev(vs))
    torch.cuda.synchronize()
    oracle.kv_append_fp8(k, v, slots, kc, vc, bs, ks, vs)
    assert np.array_equal(kc_d.cpu().numpy(), kc)
    assert np.array_equal(vc_d.cpu().numpy(), vc)


@pytest.mark.parametrize("lens,bs,hq,hkv,q_len", [
    ([38, 101], 16, 12, 2, 1),                           # the tiny batch
    ([1, 2, 15, 16, 17, 31, 33], 16, 12, 2, 1),          # ragged tails
    ([300, 47], 16, 64, 8, 1),                           # GQA 8
    ([77, 200, 5], 16, 8, 4, 2),                         # causal pair of queries (R = 4)
    ([500, 70], 64, 16, 2, 1),                           # 64-token blocks
    ([33, 1, 60], 16, 4, 4, 3),                          # MHA drafts (R = 3)
    ([20000], 16, 12, 2, 1),                             # one long sequence over many CTAs
    ([5] * 700, 16, 12, 2, 1),                           # many short sequences
    ([2, 40, 0, 9], 16, 12, 2, 1),                       # an empty sequence -> zeros
])
def test_decode_fp8_matches_oracle(lens, bs, hq, hkv, q_len):
    k8, v8, ks, vs, tables, lens, q = _fp8_case(lens, bs, hq, hkv, q_len, seed=len(lens) + bs)
    scale = 1 / math.sqrt(128)
    out = _gpu_decode_fp8(k8, v8, ks, vs, tables, lens, q, scale)
    ref = oracle.paged_attention_fp8(q, k8, v8, ks, vs, tables, lens, bs, scale)
    assert_attn_close(out, ref, f"fp8 lens={list(lens[:4])} bs={bs} G={hq // hkv} q_len={q_len}")


@pytest.mark.parametrize("make", [workloads.edge_1p1b, workloads.llama70b_b16])
def test_decode_fp8_on_benchmark_shapes(make):
    w = make()
    rng = np.random.default_rng(7)
    kf = rng.standard_normal((w.num_blocks, w.num_kv_heads, w.block_size, 128), np.float32)
    vf = rng.standard_normal((w.num_blocks, w.num_kv_heads, w.block_size, 128), np.float32)
    ks = (np.abs(kf).max(axis=(0, 2, 3)) / 448.0).astype(np.float32)
    vs = (np.abs(vf).max(axis=(0, 2, 3)) / 448.0).astype(np.float32)
    k8, v8 = _quantise(kf, ks), _quantise(vf, vs)
    q = f16_host(w.query(0, DEV))
    out = _gpu_decode_fp8(k8, v8, ks, vs, w.block_tables, w.context_lens, q, w.scale)
    ref = oracle.paged_attention_fp8(q, k8, v8, ks, vs, w.block_tables, w.context_lens,
                                     w.block_size, w.scale)
    assert_attn_close(out, ref, f"fp8 {w.name}")


def test_decode_fp8_is_deterministic_and_rejects_wide_groups():
    k8, v8, ks, vs, tables, lens, q = _fp8_case([900, 33, 1500], seed=3)
    a = _gpu_decode_fp8(k8, v8, ks, vs, tables, lens, q, 0.1)
    b = _gpu_decode_fp8(k8, v8, ks, vs, tables, lens, q, 0.1)
    assert torch.equal(a, b)
    # 12 rows per kv head (G = 6, two query tokens) is past the E4M3 kernel's 8
    k8, v8, ks, vs, tables, lens, q = _fp8_case([40, 50], q_len=2, seed=4)
    with pytest.raises(pkv.PkvError) as e:
        _gpu_decode_fp8(k8, v8, ks, vs, tables, lens, q, 0.1)
    assert e.value.status == pkv.EINVAL


def _new_slots(tables, lens, q_len, bs):
    slots = []
    for b, L in enumerate(lens):
        for i in range(q_len):
            pos = int(L) - q_len + i
            slots.append(-1 if pos < 0 else int(tables[b, pos // bs]) * bs + pos % bs)
    return np.asarray(slots, np.int64)


@pytest.mark.parametrize("lens,bs,hq,hkv,q_len", [
    ([38, 101], 16, 12, 2, 1),                           # the tiny batch
    ([33, 16, 2, 100], 16, 8, 4, 2),                     # causal pairs, new rows across blocks
    ([64, 5, 31, 4], 16, 4, 4, 4),                       # MHA drafts (R = 4)
    ([500, 70, 1], 64, 16, 2, 1),                        # 64-token blocks
    ([18, 50, 97, 16], 16, 8, 4, 4),                     # drafts across both chunks of a stage
])
def test_fused_append_decode_fp8_matches_oracle(lens, bs, hq, hkv, q_len):
    k8, v8, ks, vs, tables, lens, q = _fp8_case(lens, bs, hq, hkv, q_len, seed=len(lens) * 7 + q_len)
    rng = np.random.default_rng(99)
    kn = rng.standard_normal((len(lens) * q_len, hkv, 128)).astype(np.float16)
    vn = rng.standard_normal((len(lens) * q_len, hkv, 128)).astype(np.float16)
    k8_d, v8_d = _dev(k8), _dev(v8)
    qd = _dev(q)
    out = torch.empty_like(qd)
    ws = pkv.make_workspace(q.shape[0], q_len, hq, hkv)
    scale = 1 / math.sqrt(128)
    pkv.paged_attn_decode_append_fp8(out, qd, _dev(kn), _dev(vn), k8_d, v8_d, _dev(ks), _dev(vs),
                                     _dev(tables, torch.int32), _dev(lens, torch.int32), scale, ws)
    torch.cuda.synchronize()
    assert pkv.device_error(clear=True) == 0
    oracle.kv_append_fp8(kn, vn, _new_slots(tables, lens, q_len, bs), k8, v8, bs, ks, vs)
    assert np.array_equal(k8_d.cpu().numpy(), k8) and np.array_equal(v8_d.cpu().numpy(), v8)
    ref = oracle.paged_attention_fp8(q, k8, v8, ks, vs, tables, lens, bs, scale)
    assert_attn_close(out, ref, f"fp8 fused lens={list(lens[:4])} q_len={q_len}")


def test_fused_append_decode_fp8_on_the_edge_shape():
    w = workloads.edge_1p1b()
    rng = np.random.default_rng(8)
    kf = rng.standard_normal((w.num_blocks, w.num_kv_heads, w.block_size, 128), np.float32)
    vf = rng.standard_normal((w.num_blocks, w.num_kv_heads, w.block_size, 128), np.float32)
    ks = (np.abs(kf).max(axis=(0, 2, 3)) / 448.0).astype(np.float32)
    vs = (np.abs(vf).max(axis=(0, 2, 3)) / 448.0).astype(np.float32)
    k8, v8 = _quantise(kf, ks), _quantise(vf, vs)
    q = w.query(0, DEV)
    kn, vn = w.new_kv(0, DEV)
    k8_d, v8_d = _dev(k8), _dev(v8)
    out = torch.empty_like(q)
    ws = pkv.make_workspace(w.num_seqs, w.q_len, w.num_q_heads, w.num_kv_heads)
    pkv.paged_attn_decode_append_fp8(out, q, kn, vn, k8_d, v8_d, _dev(ks), _dev(vs),
                                     _dev(w.block_tables, torch.int32),
                                     _dev(w.context_lens, torch.int32), w.scale, ws)
    torch.cuda.synchronize()
    slots = _new_slots(w.block_tables, w.context_lens, w.q_len, w.block_size)
    oracle.kv_append_fp8(f16_host(kn), f16_host(vn), slots, k8, v8, w.block_size, ks, vs)
    assert np.array_equal(k8_d.cpu().numpy(), k8) and np.array_equal(v8_d.cpu().numpy(), v8)
    ref = oracle.paged_attention_fp8(f16_host(q), k8, v8, ks, vs, w.block_tables, w.context_lens,
                                     w.block_size, w.scale)
    assert_attn_close(out, ref, "fp8 fused edge_1p1b")


def test_decode_fp8_bad_block_id_sets_the_error_bit_without_fault():
    # a table entry past the pool in the second chunk of a two-chunk stage: it reads as zeros,
    # the block-id bit is set, and the other sequences are exact
    k8, v8, ks, vs, tables, lens, q = _fp8_case([300, 47, 90], seed=31)
    bad = tables.copy()
    bad[0, 3] = k8.shape[0] + 9
    qd = _dev(q)
    out = torch.empty_like(qd)
    ws = pkv.make_workspace(q.shape[0], q.shape[1], q.shape[2], k8.shape[1])
    pkv.paged_attn_decode_fp8(out, qd, _dev(k8), _dev(v8), _dev(ks), _dev(vs),
                              _dev(bad, torch.int32), _dev(lens, torch.int32), 0.1, ws)
    torch.cuda.synchronize()
    assert pkv.device_error(clear=True) & pkv.DEVERR_BLOCK_ID
    ref = oracle.paged_attention_fp8(q, k8, v8, ks, vs, tables, lens, 16, 0.1)
    assert_attn_close(out[1:], ref[1:], "fp8 beside a sequence with a bad block id")
