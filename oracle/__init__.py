"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle of paged KV-cache decode attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may import
this package. The product (``paged_kv_cache_147_gb300``) never imports it, and it never
imports the product: the two share only the seeded input generator module.

The arithmetic lives in ``pkv_oracle.cpp`` (plain loops in fp64, each function citing the
page passage it restates); this module loads it with ctypes, building it with the host C++
compiler when the shared object is missing or older than its source. fp16 arrays cross the
boundary as their raw ``uint16`` bit patterns.

The FP8 (E4M3) cache functions are pinned against torch's float8_e4m3fn decoding and rounding,
the format's landmark values, a brute-force nearest search and the fp16 oracle on an exactly
representable cache.

Parity status: pinned by the CPU tests, except the ring valid-set rule after a rollback, a
reading of the streaming page that the pages themselves do not fix (parity unpinned against
the pages there; pinned only by an independent linear-history simulation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.cpp")
_LIB = os.path.join(_HERE, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (-O2, no fast-math: fp64 semantics as written)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
                        "-o", tmp, _SRC], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, u64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_double
            lib.pkv_orc_kv_bytes.restype = u64
            lib.pkv_orc_kv_bytes.argtypes = [u64] * 6
            lib.pkv_orc_f16_to_f64.restype = f64
            lib.pkv_orc_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.pkv_orc_f16_array_to_f64.argtypes = [P, P, i64]
            lib.pkv_orc_slot_mapping.argtypes = [P, P, i32, P, i32, i32, P]
            lib.pkv_orc_ring_slot.restype = i64
            lib.pkv_orc_ring_slot.argtypes = [i64, i64, i64]
            lib.pkv_orc_ring_slot_mapping.argtypes = [P, P, i32, P, i32, i32, i32, i32, P]
            lib.pkv_orc_ring_valid.restype = i32
            lib.pkv_orc_ring_valid.argtypes = [i64, i64, i32, i32, i32, i32, P]
            lib.pkv_orc_kv_append.argtypes = [P, P, P, i32, P, P, i32, i32, i32]
            lib.pkv_orc_copy_blocks.argtypes = [P, P, P, P, i32, i64, i32, i64]
            lib.pkv_orc_paged_attention.restype = i32
            lib.pkv_orc_paged_attention.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                                    i32, i32, f64, P, i32]
            lib.pkv_orc_rope.argtypes = [P, i32, f64, f64]
            lib.pkv_orc_e4m3_to_f64.restype = f64
            lib.pkv_orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.pkv_orc_f64_to_e4m3.restype = ctypes.c_uint8
            lib.pkv_orc_f64_to_e4m3.argtypes = [f64]
            lib.pkv_orc_kv_append_fp8.argtypes = [P, P, P, i32, P, P, i32, i32, i32, P, P]
            lib.pkv_orc_spec_verify.argtypes = [P, P, P, P, P, i32, i32, i32, P, P]
            lib.pkv_orc_paged_attention_fp8.restype = i32
            lib.pkv_orc_paged_attention_fp8.argtypes = [P, P, P, P, P, P, P, i32, P, i32, i32,
                                                        i32, i32, i32, i32, f64, i32]
            lib.pkv_orc_ring_attention.restype = i32
            lib.pkv_orc_ring_attention.argtypes = [P, P, P, P, P, i32, P, P, i32, i32, i32,
                                                   i32, i32, i32, i32, i32, f64, i32, f64, P,
                                                   i32]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _u16(a: np.ndarray) -> np.ndarray:
    """fp16 (or uint16) array -> contiguous uint16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int64)


# --------------------------------------------------------------------------- ledger
def kv_bytes(num_layers, seq_len, num_kv_heads, head_dim, dtype_bytes, batch) -> int:
    """KV bytes = 2 x layers x seq x kv_heads x head_dim x dtype_bytes x batch."""
    return int(_load().pkv_orc_kv_bytes(num_layers, seq_len, num_kv_heads, head_dim,
                                        dtype_bytes, batch))


# --------------------------------------------------------------------------- fp16
def f16_to_f64(bits) -> np.ndarray:
    b = _u16(np.asarray(bits))
    out = np.empty(b.shape, dtype=np.float64)
    _load().pkv_orc_f16_array_to_f64(_ptr(b), _ptr(out), b.size)
    return out


# --------------------------------------------------------------------------- addressing
def slot_mapping(seq_ids, positions, block_tables, block_size) -> np.ndarray:
    seq_ids, positions, bt = _i32(seq_ids), _i64(positions), _i32(block_tables)
    out = np.empty(len(positions), dtype=np.int64)
    _load().pkv_orc_slot_mapping(_ptr(seq_ids), _ptr(positions), len(positions), _ptr(bt),
                                 bt.shape[1], block_size, _ptr(out))
    return out


def ring_slot(pos: int, sink: int, window: int) -> int:
    return int(_load().pkv_orc_ring_slot(pos, sink, window))


def ring_slot_mapping(seq_ids, positions, block_tables, sink, window, block_size) -> np.ndarray:
    seq_ids, positions, bt = _i32(seq_ids), _i64(positions), _i32(block_tables)
    out = np.empty(len(positions), dtype=np.int64)
    _load().pkv_orc_ring_slot_mapping(_ptr(seq_ids), _ptr(positions), len(positions), _ptr(bt),
                                      bt.shape[1], sink, window, block_size, _ptr(out))
    return out


def ring_valid(L: int, hw: int, sink: int, window: int, q_len: int = 1, qi: int = 0) -> np.ndarray:
    buf = np.empty(sink + window + 1, dtype=np.int64)
    n = _load().pkv_orc_ring_valid(L, hw, sink, window, q_len, qi, _ptr(buf))
    return buf[:n].copy()


# --------------------------------------------------------------------------- cache edits
def kv_append(k, v, slots, k_cache, v_cache, block_size) -> None:
    """In-place byte scatter of k, v [T, Hkv, D] (fp16) into one layer's pools."""
    k, v, slots = _u16(k), _u16(v), _i64(slots)
    kc, vc = _u16(k_cache), _u16(v_cache)
    assert np.shares_memory(kc, k_cache) and np.shares_memory(vc, v_cache), "pools must be contiguous"
    _load().pkv_orc_kv_append(_ptr(k), _ptr(v), _ptr(slots), len(slots), _ptr(kc), _ptr(vc),
                              k.shape[1], k.shape[2], block_size)


def copy_blocks(k_cache, v_cache, src, dst, num_layers, layer_stride_elems, block_elems) -> None:
    src, dst = _i32(src), _i32(dst)
    kc, vc = _u16(k_cache), _u16(v_cache)
    assert np.shares_memory(kc, k_cache) and np.shares_memory(vc, v_cache), "pools must be contiguous"
    _load().pkv_orc_copy_blocks(_ptr(kc), _ptr(vc), _ptr(src), _ptr(dst), len(src),
                                layer_stride_elems, num_layers, block_elems)


# --------------------------------------------------------------------------- attention
def paged_attention(q, k_cache, v_cache, block_tables, context_lens, block_size, scale,
                    seq_mask=None, num_threads=0, return_threads=False):
    """q [B, q_len, Hq, D] fp16; caches [NB, Hkv, bs, D] fp16 -> out fp64 [B, q_len, Hq, D]."""
    q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, cl = _i32(block_tables), _i32(context_lens)
    B, q_len, Hq, D = q.shape
    Hkv = kc.shape[1]
    out = np.zeros(q.shape, dtype=np.float64)
    mask = None if seq_mask is None else np.ascontiguousarray(seq_mask, dtype=np.uint8)
    nt = _load().pkv_orc_paged_attention(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                         bt.shape[1], _ptr(cl), B, q_len, Hq, Hkv, D,
                                         block_size, float(scale), _ptr(mask), num_threads)
    return (out, nt) if return_threads else out


def rope(x, index: float, base: float = 10000.0) -> np.ndarray:
    x = np.array(x, dtype=np.float64, copy=True)
    _load().pkv_orc_rope(_ptr(x), x.shape[-1], float(index), float(base))
    return x


ROPE_CACHE_INDEX, ROPE_LOGICAL_POSITION, ROPE_NONE = 0, 1, 2


def ring_attention(q, k_cache, v_cache, block_tables, logical_len, high_water, block_size,
                   sink, window, scale, rope_mode=ROPE_CACHE_INDEX, rope_base=10000.0,
                   seq_mask=None, num_threads=0, return_threads=False):
    q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
    bt, L, hw = _i32(block_tables), _i64(logical_len), _i64(high_water)
    B, q_len, Hq, D = q.shape
    Hkv = kc.shape[1]
    out = np.zeros(q.shape, dtype=np.float64)
    mask = None if seq_mask is None else np.ascontiguousarray(seq_mask, dtype=np.uint8)
    nt = _load().pkv_orc_ring_attention(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt),
                                        bt.shape[1], _ptr(L), _ptr(hw), B, q_len, Hq, Hkv, D,
                                        block_size, sink, window, float(scale), rope_mode,
                                        float(rope_base), _ptr(mask), num_threads)
    return (out, nt) if return_threads else out


# --------------------------------------------------------------------------- FP8 (E4M3) cache
def e4m3_to_f64(codes) -> np.ndarray:
    """E4M3 byte codes -> fp64 values (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8)
    f = _load().pkv_orc_e4m3_to_f64
    return np.array([f(int(x)) for x in c.ravel()], dtype=np.float64).reshape(c.shape)


def f64_to_e4m3(x) -> np.ndarray:
    """Round to nearest E4M3 (ties to the even code), saturating finite values to +-448."""
    a = np.asarray(x, dtype=np.float64)
    f = _load().pkv_orc_f64_to_e4m3
    return np.array([f(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def kv_append_fp8(k, v, slots, k_cache, v_cache, block_size, k_scale, v_scale) -> None:
    """In-place FP8 append: k, v [T, Hkv, D] fp16 -> E4M3(x / scale[h]) bytes in one layer's
    uint8 pools [NB, Hkv, bs, D]; the division is done in binary32."""
    k, v, slots = _u16(k), _u16(v), _i64(slots)
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    _load().pkv_orc_kv_append_fp8(_ptr(k), _ptr(v), _ptr(slots), len(slots), _ptr(k_cache),
                                  _ptr(v_cache), k.shape[1], k.shape[2], block_size, _ptr(ks),
                                  _ptr(vs))


def paged_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                        block_size, scale, num_threads=0):
    """q [B, q_len, Hq, D] fp16; uint8 E4M3 caches [NB, Hkv, bs, D] with per-kv-head scales
    -> out fp64 [B, q_len, Hq, D]."""
    q = _u16(q)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
    vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    bt, cl = _i32(block_tables), _i32(context_lens)
    B, q_len, Hq, D = q.shape
    Hkv = kc.shape[1]
    out = np.zeros(q.shape, dtype=np.float64)
    _load().pkv_orc_paged_attention_fp8(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(ks),
                                        _ptr(vs), _ptr(bt), bt.shape[1], _ptr(cl), B, q_len, Hq,
                                        Hkv, D, block_size, float(scale), num_threads)
    return out


# --------------------------------------------------------------------------- speculative verify
def spec_verify(target_logits, draft_logits, drafts, u_accept, u_sample):
    """target [B, K+1, V], draft [B, K, V] float32 logits; drafts [B, K]; u_accept [B, K],
    u_sample [B] in [0, 1) -> (n_accept [B], next_token [B]) int32."""
    t = np.ascontiguousarray(target_logits, dtype=np.float32)
    d = np.ascontiguousarray(draft_logits, dtype=np.float32)
    x = _i32(drafts)
    ua = np.ascontiguousarray(u_accept, dtype=np.float32)
    us = np.ascontiguousarray(u_sample, dtype=np.float32)
    B, K1, V = t.shape
    n = np.zeros(B, np.int32)
    nxt = np.zeros(B, np.int32)
    _load().pkv_orc_spec_verify(_ptr(t), _ptr(d), _ptr(x), _ptr(ua), _ptr(us), B, K1 - 1, V,
                                _ptr(n), _ptr(nxt))
    return n, nxt
