"""GPU parity when the scores climb along the context by more than 2^8 at a time.

The decode keeps each row's running maximum until a score exceeds it by more than 2^8, and
only then reduces the step's maxima across the warp and rescales l and O. On random data that
happens almost only at a segment's first step. Here the keys of each (sequence, kv head) carry
a component along the group's query direction that rises in levels across the context (and
falls back once), plus a few isolated spikes above every level, so that the maximum grows by
far more than 2^8 in the middle of segments, of stages and of split units. The fp16 cache is
run through the 8-row transposed tile (GQA 6 and 8, MHA with 64-token blocks), the 16-row tile
(R = 12) and the two-m-tile form (R = 18); the E4M3 cache through its two-chunk stages; and
the chunked prefill, which rescales O in tensor memory past the same margin.
Results must meet the attention bar of tests/_util.py against the fp64 oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_147_gb300 import pkv

from _util import assert_attn_close

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCALE = 1 / math.sqrt(128)
LOG2E = 1.4426950408889634
LEVELS = (0, 2, 1, 3)        # the level of each quarter of a context
STEP = 22.0                  # key component per level along the unit query direction
QDIR = 4.0                   # query component along that direction


def _dev(a, dtype=None):
    t = torch.as_tensor(np.ascontiguousarray(a))
    return t.to(DEV) if dtype is None else t.to(device=DEV, dtype=dtype)


def _climbing(lens, bs, hq, hkv, q_len, seed, extra_blocks=3):
    """fp32 K/V pools [NB, Hkv, bs, 128] (unused slots NaN), tables, lengths and fp16 queries
    whose scores climb along each context."""
    rng = np.random.default_rng(seed)
    G = hq // hkv
    lens = np.asarray(lens, dtype=np.int32)
    nblk = [(int(l) + bs - 1) // bs for l in lens]
    nb = sum(nblk) + extra_blocks
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(lens), max(nblk)), -1, dtype=np.int32)
    cur = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = perm[cur:cur + n]
        cur += n
    u = rng.standard_normal((len(lens), hkv, 128))
    u /= np.linalg.norm(u, axis=-1, keepdims=True)
    q = 0.3 * rng.standard_normal((len(lens), q_len, hq, 128))
    q += QDIR * np.repeat(u, G, axis=1)[:, None]
    k = rng.standard_normal((nb, hkv, bs, 128))
    v = rng.standard_normal((nb, hkv, bs, 128))
    used = np.zeros((nb, bs), bool)
    for b, L in enumerate(lens):
        pos = np.arange(int(L))
        beta = STEP * np.asarray(LEVELS, float)[(len(LEVELS) * pos) // max(int(L), 1)]
        if L >= 64:   # spikes past the first two chunks and the first eighth
            s0 = max(int(L) // 8, 32)
            spikes = s0 + rng.choice(int(L) - s0, size=3, replace=False)
            beta[spikes] = STEP * (max(LEVELS) + 1.5)
        blk, off = tables[b, pos // bs], pos % bs
        k[blk, :, off, :] += beta[:, None, None] * u[b][None, :, :]
        used[blk, off] = True
    mask = ~used[:, None, :, None].repeat(hkv, 1).repeat(128, 3)
    k[mask] = np.nan
    v[mask] = np.nan
    return k.astype(np.float32), v.astype(np.float32), tables, lens, q.astype(np.float16)


def _assert_climbs(k, tables, lens, q, bs, hkv):
    """The case does what it is for: in every sequence of 64+ tokens, some head's scores (log2
    units, as the kernel forms them) rise more than 2^8 above everything in its first 16."""
    G = q.shape[2] // hkv
    for b, L in enumerate(lens):
        if L < 64:
            continue
        pos = np.arange(int(L))
        kb = np.nan_to_num(k[tables[b, pos // bs], :, pos % bs, :].astype(np.float64))  # [L, Hkv, D]
        x = np.einsum("hd,lhd->lh", q[b, -1, ::G].astype(np.float64), kb) * SCALE * LOG2E
        assert (x[16:].max(axis=0) - x[:16].max(axis=0)).max() > 8.0, f"sequence {b}"


@pytest.fixture(autouse=True)
def _clean_device_error():
    pkv.device_error(clear=True)
    yield
    assert pkv.device_error(clear=True) == 0, "a kernel bounds guard fired"


@pytest.mark.parametrize("lens,bs,hq,hkv,q_len", [
    ([3000, 700, 41, 1], 16, 12, 2, 1),       # transposed tile, GQA 6
    ([2000, 333], 16, 64, 8, 1),              # transposed tile, GQA 8
    ([2500, 900], 64, 32, 32, 1),             # MHA, 64-token blocks (one 3-D box per K / V)
    ([1500, 257], 16, 8, 2, 3),               # 16-row tile (R = 12), causal queries
    ([1500, 257], 16, 12, 2, 3),              # two 16-row m-tiles (R = 18), causal queries
    ([6000], 16, 12, 2, 1),                   # one sequence split over many CTAs
])
def test_decode_fp16_scores_climbing_along_the_context(lens, bs, hq, hkv, q_len):
    k, v, tables, lens, q = _climbing(lens, bs, hq, hkv, q_len, seed=sum(lens) + q_len)
    k16, v16 = k.astype(np.float16), v.astype(np.float16)
    _assert_climbs(k16, tables, lens, q, bs, hkv)
    qd = _dev(q)
    out = torch.empty_like(qd)
    ws = pkv.make_workspace(q.shape[0], q_len, hq, hkv)
    pkv.paged_attn_decode(out, qd, _dev(k16), _dev(v16), _dev(tables, torch.int32),
                          _dev(lens, torch.int32), SCALE, ws)
    torch.cuda.synchronize()
    ref = oracle.paged_attention(q, k16, v16, tables, lens, bs, SCALE)
    assert_attn_close(out, ref, f"fp16 lens={list(lens[:3])} G={hq // hkv} q_len={q_len}")


def _quantise(x, scale):
    y = torch.from_numpy(np.nan_to_num(x) / scale[None, :, None, None]).clamp(-448.0, 448.0)
    return y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("lens,bs,hq,hkv,q_len", [
    ([3000, 700, 41], 16, 12, 2, 1),          # GQA 6
    ([2000, 333], 16, 64, 8, 1),              # GQA 8
    ([1200, 77], 16, 8, 4, 2),                # causal pair of queries (R = 4)
    ([6000], 16, 12, 2, 1),                   # one sequence split over many CTAs
])
def test_decode_fp8_scores_climbing_along_the_context(lens, bs, hq, hkv, q_len):
    k, v, tables, lens, q = _climbing(lens, bs, hq, hkv, q_len, seed=sum(lens) + 7 * q_len)
    ks = (np.nanmax(np.abs(k), axis=(0, 2, 3)) / 448.0 * 1.5).astype(np.float32)
    vs = (np.nanmax(np.abs(v), axis=(0, 2, 3)) / 448.0 * 1.5).astype(np.float32)
    k8, v8 = _quantise(k, ks), _quantise(v, vs)
    unused = np.isnan(k)
    k8[unused] = 0x7F                         # NaN codes: any read of them shows
    v8[unused] = 0xFF
    kq = torch.from_numpy(k8).view(torch.float8_e4m3fn).double().numpy() * ks[None, :, None, None]
    _assert_climbs(kq, tables, lens, q, bs, hkv)
    qd = _dev(q)
    out = torch.empty_like(qd)
    ws = pkv.make_workspace(q.shape[0], q_len, hq, hkv)
    pkv.paged_attn_decode_fp8(out, qd, _dev(k8), _dev(v8), _dev(ks), _dev(vs),
                              _dev(tables, torch.int32), _dev(lens, torch.int32), SCALE, ws)
    torch.cuda.synchronize()
    ref = oracle.paged_attention_fp8(q, k8, v8, ks, vs, tables, lens, bs, SCALE)
    assert_attn_close(out, ref, f"fp8 lens={list(lens[:3])} G={hq // hkv} q_len={q_len}")


@pytest.mark.parametrize("lens,bs,hq,hkv,q_len", [
    ([1500, 513], 16, 12, 2, 128),            # GQA 6, 128-token chunks
    ([4096, 700], 16, 16, 2, 512),            # GQA 8, 512-token chunks at the end of 4096
    ([900, 300], 64, 8, 8, 64),               # MHA, 64-token blocks
])
def test_prefill_scores_climbing_along_the_context(lens, bs, hq, hkv, q_len):
    """The chunked prefill raises a row's maximum, and rescales O and the row sum in tensor
    memory, only past the same 2^8 margin."""
    k, v, tables, lens, q = _climbing(lens, bs, hq, hkv, q_len, seed=sum(lens) + 11 * q_len)
    k16, v16 = k.astype(np.float16), v.astype(np.float16)
    _assert_climbs(k16, tables, lens, q, bs, hkv)
    qd = _dev(q)
    out = torch.full_like(qd, float("nan"))
    pkv.paged_prefill(out, qd, _dev(k16), _dev(v16), _dev(tables, torch.int32),
                      _dev(lens, torch.int32), SCALE)
    torch.cuda.synchronize()
    ref = oracle.paged_attention(q, k16, v16, tables, lens, bs, SCALE)
    assert_attn_close(out, ref, f"prefill lens={list(lens)} G={hq // hkv} q_len={q_len}")
