"""Thin Python binding of libpkv.so (the C ABI declared in include/pkv.h).

Each function has the name of its C entry point without the ``pkv_`` prefix and only
marshals arguments: it reads shapes and device pointers off torch tensors, passes the
current CUDA stream, and turns a negative status into :class:`PkvError`. Every step of the
computation runs in the library's CUDA kernels; there is no fallback path. Loading fails
loudly if the library is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# PKV_LIB selects another build of the library (e.g. a pipeline-depth variant).
LIB_PATH = os.environ.get("PKV_LIB") or os.path.join(_HERE, "libpkv.so")

# Symbols the header declares (kept in sync with include/pkv.h; the CPU tests check both).
SYMBOLS = (
    "pkv_version", "pkv_device_error", "pkv_slot_mapping", "pkv_ring_slot_mapping",
    "pkv_kv_append", "pkv_copy_blocks", "pkv_decode_workspace_bytes", "pkv_workspace_init",
    "pkv_paged_attn_decode", "pkv_rope_table", "pkv_ring_attn_decode", "pkv_check_tables",
    "pkv_check_slots", "pkv_paged_attn_decode_noalloc", "pkv_paged_attn_decode_append",
    "pkv_kv_append_fp8", "pkv_paged_attn_decode_fp8", "pkv_paged_attn_decode_append_fp8",
    "pkv_pool_create", "pkv_pool_destroy", "pkv_pool_allocate", "pkv_pool_warm",
    "pkv_pool_release", "pkv_pool_fork", "pkv_pool_append", "pkv_pool_stats",
    "pkv_pool_refcount", "pkv_spec_verify", "pkv_set_early_start", "pkv_paged_prefill",
    "pkv_ring_attn_decode_append",
)

OK, EINVAL, ERANGE, ENOSPC, ECUDA_BASE = 0, -22, -34, -28, -1000
DEVERR_BLOCK_ID, DEVERR_CONTEXT, DEVERR_SLOT, DEVERR_TIMEOUT, DEVERR_SEQ, DEVERR_POSITION = \
    1, 2, 4, 8, 16, 32
DEVERR_TOKEN = 64


class PkvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        if status <= ECUDA_BASE:
            what = f"CUDA error {ECUDA_BASE - status}"
        else:
            what = {EINVAL: "invalid argument", ERANGE: "index out of range",
                    ENOSPC: "workspace too small"}.get(status, "error")
        super().__init__(f"{fn} failed: {what} (status {status})")


_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Loads libpkv.so (built by paged_kv_cache_147_gb300.build); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m paged_kv_cache_147_gb300.build` (no CPU fallback)")
        _lib = _configure(ctypes.CDLL(LIB_PATH))
        return _lib


def load_variant(path: str) -> ctypes.CDLL:
    """Loads another build of the library (e.g. one compiled with different tuning macros)
    next to the default one, with the same signatures; the tests compare the two."""
    return _configure(ctypes.CDLL(path))


def _configure(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Sets the argument and result types of every entry point on a loaded library."""
    P, i32, i64, sz, f32, f64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                 ctypes.c_size_t, ctypes.c_float, ctypes.c_double)
    sig = {
        "pkv_version": (i32, []),
        "pkv_device_error": (i32, [P, i32, P]),
        "pkv_slot_mapping": (i32, [P, P, i32, P, i32, i32, i32, P, P]),
        "pkv_ring_slot_mapping": (i32, [P, P, i32, P, i32, i32, i32, i32, i32, P, P]),
        "pkv_kv_append": (i32, [P, P, P, i32, P, P, i32, i32, i32, i32, P]),
        "pkv_copy_blocks": (i32, [P, P, P, P, i32, i64, i32, i32, i32, i32, i32, P]),
        "pkv_decode_workspace_bytes": (sz, [i32, i32, i32, i32, i32]),
        "pkv_workspace_init": (i32, [P, sz, P]),
        "pkv_paged_attn_decode": (i32, [P, P, P, P, i32, P, i32, P, i32, i32, i32, i32, i32,
                                        i32, f32, P, sz, P]),
        "pkv_rope_table": (i32, [P, i32, i32, f64]),
        "pkv_ring_attn_decode": (i32, [P, P, P, P, i32, P, i32, P, P, i32, i32, i32, i32,
                                       i32, i32, i32, i32, P, f32, P, sz, P]),
        "pkv_check_tables": (i32, [P, P, i32, i32, i32, i32, P]),
        "pkv_check_slots": (i32, [P, i32, i32, i32, P]),
        "pkv_paged_attn_decode_noalloc": (i32, [P, P, P, P, i32, P, i32, P, i32, i32, i32,
                                                i32, i32, i32, f32, P]),
        "pkv_paged_attn_decode_append": (i32, [P, P, P, P, P, P, i32, P, i32, P, i32, i32,
                                               i32, i32, i32, i32, f32, P, sz, P]),
        "pkv_kv_append_fp8": (i32, [P, P, P, i32, P, P, i32, i32, i32, i32, P, P, P]),
        "pkv_paged_attn_decode_fp8": (i32, [P, P, P, P, P, P, i32, P, i32, P, i32, i32, i32,
                                            i32, i32, i32, f32, P, sz, P]),
        "pkv_paged_attn_decode_append_fp8": (i32, [P, P, P, P, P, P, P, P, i32, P, i32, P, i32,
                                                   i32, i32, i32, i32, i32, f32, P, sz, P]),
        "pkv_set_early_start": (i32, [i32]),
        "pkv_ring_attn_decode_append": (i32, [P, P, P, P, P, P, i32, P, i32, P, P, i32, i32, i32,
                                              i32, i32, i32, i32, i32, P, f32, P, sz, P]),
        "pkv_paged_prefill": (i32, [P, P, P, P, i32, P, i32, P, i32, i32, i32, i32, i32, i32, f32,
                                    P]),
        "pkv_pool_create": (i32, [i32, i32, i32, P]),
        "pkv_pool_destroy": (None, [P]),
        "pkv_pool_allocate": (i32, [P, P, i32, i32, P, i32, P, P]),
        "pkv_pool_warm": (i32, [P, P, i32]),
        "pkv_pool_release": (i32, [P, P, i32]),
        "pkv_pool_fork": (i32, [P, P, i32]),
        "pkv_pool_append": (i32, [P, P, P, i32, i32, i32, P, P, P, i32, P]),
        "pkv_pool_stats": (i32, [P, P, P, P, P, P]),
        "pkv_pool_refcount": (i32, [P, i32]),
        "pkv_spec_verify": (i32, [P, P, P, P, P, i32, i32, i32, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name, None)    # an older build may lack newer entry points
        if f is not None:
            f.restype, f.argtypes = res, args
    return lib


def _check(fn: str, status: int) -> None:
    if status != OK:
        raise PkvError(fn, status)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def version() -> int:
    return load().pkv_version()


def device_error(clear: bool = True, stream=None) -> int:
    out = ctypes.c_uint(0)
    _check("pkv_device_error", load().pkv_device_error(ctypes.byref(out), int(clear),
                                                        _stream(stream)))
    return out.value


# ------------------------------------------------------------------------------ slot mapping
def slot_mapping(seq_ids, positions, block_tables, block_size, out=None, stream=None):
    n = positions.numel()
    out = torch.empty(n, dtype=torch.int64, device=positions.device) if out is None else out
    _check("pkv_slot_mapping", load().pkv_slot_mapping(
        _p(seq_ids), _p(positions), n, _p(block_tables), block_tables.shape[0],
        block_tables.shape[1], block_size, _p(out), _stream(stream)))
    return out


def ring_slot_mapping(seq_ids, positions, block_tables, sink, window, block_size, out=None,
                      stream=None):
    n = positions.numel()
    out = torch.empty(n, dtype=torch.int64, device=positions.device) if out is None else out
    _check("pkv_ring_slot_mapping", load().pkv_ring_slot_mapping(
        _p(seq_ids), _p(positions), n, _p(block_tables), block_tables.shape[0],
        block_tables.shape[1], sink, window, block_size, _p(out), _stream(stream)))
    return out


# ------------------------------------------------------------------------------ cache edits
def kv_append(k, v, slots, k_cache, v_cache, stream=None):
    """k, v [T, Hkv, D]; k_cache, v_cache one layer [NB, Hkv, bs, D]."""
    nb, hkv, bs, d = k_cache.shape
    _check("pkv_kv_append", load().pkv_kv_append(
        _p(k), _p(v), _p(slots), slots.numel(), _p(k_cache), _p(v_cache), nb, hkv, d, bs,
        _stream(stream)))


def kv_append_fp8(k, v, slots, k_cache, v_cache, k_scale, v_scale, stream=None):
    """k, v fp16 [T, Hkv, D]; k_cache, v_cache one layer of uint8 E4M3 codes [NB, Hkv, bs, D];
    k_scale, v_scale float32 [Hkv] on the device."""
    nb, hkv, bs, d = k_cache.shape
    _check("pkv_kv_append_fp8", load().pkv_kv_append_fp8(
        _p(k), _p(v), _p(slots), slots.numel(), _p(k_cache), _p(v_cache), nb, hkv, d, bs,
        _p(k_scale), _p(v_scale), _stream(stream)))


def copy_blocks(k_cache, v_cache, src, dst, stream=None):
    """k_cache, v_cache [layers, NB, Hkv, bs, D] (or one layer [NB, Hkv, bs, D])."""
    kc = k_cache if k_cache.dim() == 5 else k_cache.unsqueeze(0)
    layers, nb, hkv, bs, d = kc.shape
    _check("pkv_copy_blocks", load().pkv_copy_blocks(
        _p(k_cache), _p(v_cache), _p(src), _p(dst), src.numel(), kc.stride(0), layers, nb, hkv,
        d, bs, _stream(stream)))


# ------------------------------------------------------------------------------ attention
def set_early_start(enable: bool) -> bool:
    """Lets the fused-append calls start while the previous kernel finishes (True, the
    default) or not; returns the previous setting. Process-wide."""
    return bool(load().pkv_set_early_start(1 if enable else 0))


def decode_workspace_bytes(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim=128) -> int:
    n = load().pkv_decode_workspace_bytes(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim)
    if n == 0:
        raise PkvError("pkv_decode_workspace_bytes", EINVAL)
    return int(n)


def workspace_init(workspace, stream=None):
    _check("pkv_workspace_init", load().pkv_workspace_init(
        _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def make_workspace(num_seqs, q_len, num_q_heads, num_kv_heads, device="cuda", stream=None):
    """Allocates (through torch) and zeroes a decode workspace."""
    ws = torch.empty(decode_workspace_bytes(num_seqs, q_len, num_q_heads, num_kv_heads),
                     dtype=torch.uint8, device=device)
    workspace_init(ws, stream)
    return ws


def paged_attn_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale, workspace,
                      stream=None):
    """q, out [B, q_len, Hq, D]; k_cache, v_cache one layer [NB, Hkv, bs, D]."""
    B, q_len, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_paged_attn_decode", load().pkv_paged_attn_decode(
        _p(out), _p(q), _p(k_cache), _p(v_cache), nb, _p(block_tables), block_tables.shape[1],
        _p(context_lens), B, q_len, hq, hkv, d, bs, float(scale), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def paged_attn_decode_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                          scale, workspace, stream=None):
    """paged_attn_decode over an E4M3 cache: uint8 pools [NB, Hkv, bs, D], float32 per-kv-head
    scales [Hkv] (element value = code * scale)."""
    B, q_len, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_paged_attn_decode_fp8", load().pkv_paged_attn_decode_fp8(
        _p(out), _p(q), _p(k_cache), _p(v_cache), _p(k_scale), _p(v_scale), nb,
        _p(block_tables), block_tables.shape[1], _p(context_lens), B, q_len, hq, hkv, d, bs,
        float(scale), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out


def paged_attn_decode_append_fp8(out, q, k_new, v_new, k_cache, v_cache, k_scale, v_scale,
                                 block_tables, context_lens, scale, workspace, stream=None):
    """paged_attn_decode_append over an E4M3 cache: the new fp16 rows are stored as
    kv_append_fp8 stores them and attended over with the rest of the cache."""
    B, q_len, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_paged_attn_decode_append_fp8", load().pkv_paged_attn_decode_append_fp8(
        _p(out), _p(q), _p(k_new), _p(v_new), _p(k_cache), _p(v_cache), _p(k_scale),
        _p(v_scale), nb, _p(block_tables), block_tables.shape[1], _p(context_lens), B, q_len, hq,
        hkv, d, bs, float(scale), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out


def paged_attn_decode_append(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                             scale, workspace, stream=None):
    """Decode step with the KV append fused in: k_new, v_new [B*q_len, Hkv, D] go to the slots of
    positions context_lens[b] - q_len + i, then attention runs over the cache including them.

    WARNING: by default this launch may start before the kernel ahead of it on the stream has
    finished, and it reads the K/V pools, block_tables and context_lens early. If the kernel
    right before it writes any of those (a torch op that advances context_lens, copy_blocks,
    ...), put another launch or a copy in between, or call set_early_start(False) first."""
    B, q_len, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_paged_attn_decode_append", load().pkv_paged_attn_decode_append(
        _p(out), _p(q), _p(k_new), _p(v_new), _p(k_cache), _p(v_cache), nb, _p(block_tables),
        block_tables.shape[1], _p(context_lens), B, q_len, hq, hkv, d, bs, float(scale),
        _p(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def paged_prefill(out, q, k_cache, v_cache, block_tables, context_lens, scale, stream=None):
    """Chunked-prefill attention: q, out [B, q_len, Hq, D]; the chunk's K/V rows are already in
    the one-layer caches [NB, Hkv, bs, D]; query i of sequence b attends causally up to position
    context_lens[b] - q_len + i."""
    B, q_len, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_paged_prefill", load().pkv_paged_prefill(
        _p(out), _p(q), _p(k_cache), _p(v_cache), nb, _p(block_tables), block_tables.shape[1],
        _p(context_lens), B, q_len, hq, hkv, d, bs, float(scale), _stream(stream)))
    return out


def paged_attn_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                              stream=None):
    """paged_attn_decode for callers that cannot allocate device memory: the library's fixed
    8 MiB scratch array replaces the workspace. Calls sharing it must not overlap on the GPU;
    the first call on a device must come before any stream capture."""
    B, q_len, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_paged_attn_decode_noalloc", load().pkv_paged_attn_decode_noalloc(
        _p(out), _p(q), _p(k_cache), _p(v_cache), nb, _p(block_tables), block_tables.shape[1],
        _p(context_lens), B, q_len, hq, hkv, d, bs, float(scale), _stream(stream)))
    return out


def rope_table(n_index, head_dim=128, base=10000.0) -> torch.Tensor:
    """Host float32 [n_index, head_dim/2, 2] (cos, sin) table; move it to the device."""
    t = torch.empty((n_index, head_dim // 2, 2), dtype=torch.float32)
    _check("pkv_rope_table", load().pkv_rope_table(_p(t), n_index, head_dim, float(base)))
    return t


def ring_attn_decode(out, q, k_cache, v_cache, block_tables, logical_len, high_water, sink,
                     window, rope_cos_sin, scale, workspace, stream=None):
    B, q_len, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_ring_attn_decode", load().pkv_ring_attn_decode(
        _p(out), _p(q), _p(k_cache), _p(v_cache), nb, _p(block_tables), block_tables.shape[1],
        _p(logical_len), _p(high_water), B, q_len, hq, hkv, d, bs, sink, window,
        _p(rope_cos_sin), float(scale), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def ring_attn_decode_append(out, q, k_new, v_new, k_cache, v_cache, block_tables, logical_len,
                            high_water, sink, window, rope_cos_sin, scale, workspace,
                            stream=None):
    """Sink + ring decode step with the append fused in: k_new, v_new [B*q_len, Hkv, D] (before
    RoPE) go to the ring slots of positions logical_len[b] - q_len + i, then ring attention runs
    over the cache including them. Early-start caveat as for paged_attn_decode_append."""
    B, q_len, hq, d = q.shape
    nb, hkv, bs, _ = k_cache.shape
    _check("pkv_ring_attn_decode_append", load().pkv_ring_attn_decode_append(
        _p(out), _p(q), _p(k_new), _p(v_new), _p(k_cache), _p(v_cache), nb, _p(block_tables),
        block_tables.shape[1], _p(logical_len), _p(high_water), B, q_len, hq, hkv, d, bs, sink,
        window, _p(rope_cos_sin), float(scale), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


# ------------------------------------------------------------------------------ host checks
def check_tables(block_tables, context_lens, block_size, num_blocks) -> int | None:
    """Host validation; returns None if valid, else the first bad sequence index."""
    bt = block_tables.detach().to("cpu", torch.int32).contiguous()
    cl = context_lens.detach().to("cpu", torch.int32).contiguous()
    bad = ctypes.c_int(-1)
    st = load().pkv_check_tables(_p(bt), _p(cl), bt.shape[0], bt.shape[1], block_size,
                                 num_blocks, ctypes.byref(bad))
    if st == ERANGE:
        return bad.value
    _check("pkv_check_tables", st)
    return None


def check_slots(slots, num_blocks, block_size) -> int | None:
    s = slots.detach().to("cpu", torch.int64).contiguous()
    bad = ctypes.c_int(-1)
    st = load().pkv_check_slots(_p(s), s.numel(), num_blocks, block_size, ctypes.byref(bad))
    if st == ERANGE:
        return bad.value
    _check("pkv_check_slots", st)
    return None


# ------------------------------------------------------------------------------ speculative verify
def spec_verify(target_logits, draft_logits, drafts, u_accept, u_sample, n_accept=None,
                next_token=None, stream=None):
    """target [B, K+1, V], draft [B, K, V] float32; drafts int32 [B, K]; u_accept [B, K],
    u_sample [B] float32 -> (n_accept, next_token) int32 [B] (device tensors)."""
    B, K1, V = target_logits.shape
    if n_accept is None:
        n_accept = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=target_logits.device)
    _check("pkv_spec_verify", load().pkv_spec_verify(
        _p(target_logits), _p(draft_logits), _p(drafts), _p(u_accept), _p(u_sample), B, K1 - 1,
        V, _p(n_accept), _p(next_token), _stream(stream)))
    return n_accept, next_token


# ------------------------------------------------------------------------------ host block pool
class BlockPool:
    """The library's host block pool (pkv_pool_*): block tables with prefix sharing, reference
    counts and copy-on-write pairs for pkv_copy_blocks. Tables are int32 numpy arrays."""

    def __init__(self, num_blocks: int, block_size: int, hash_bits: int = 64):
        self._lib = load()
        h = ctypes.c_void_p()
        _check("pkv_pool_create", self._lib.pkv_pool_create(num_blocks, block_size, hash_bits,
                                                             ctypes.byref(h)))
        self._h, self.num_blocks, self.block_size = h, num_blocks, block_size

    def close(self):
        if self._h:
            self._lib.pkv_pool_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @staticmethod
    def _i32(a):
        return np.ascontiguousarray(np.asarray(a, dtype=np.int32))

    def allocate(self, tokens, max_tokens=None, table_cap=None):
        """-> (table, reused): the sequence's blocks and how many were shared."""
        t = self._i32(tokens)
        mt = len(t) if max_tokens is None else int(max_tokens)
        cap = table_cap or (max(mt, len(t)) // self.block_size + 2)
        table = np.empty(cap, np.int32)
        n, reused = ctypes.c_int(0), ctypes.c_int(0)
        _check("pkv_pool_allocate", self._lib.pkv_pool_allocate(
            self._h, t.ctypes.data, len(t), mt, table.ctypes.data, cap, ctypes.byref(n),
            ctypes.byref(reused)))
        return table[:n.value].copy(), reused.value

    def warm(self, tokens):
        t = self._i32(tokens)
        _check("pkv_pool_warm", self._lib.pkv_pool_warm(self._h, t.ctypes.data, len(t)))

    def release(self, table):
        t = self._i32(table)
        _check("pkv_pool_release", self._lib.pkv_pool_release(self._h, t.ctypes.data, len(t)))

    def fork(self, table):
        t = self._i32(table)
        _check("pkv_pool_fork", self._lib.pkv_pool_fork(self._h, t.ctypes.data, len(t)))
        return t.copy()

    def append(self, table, length, n_new, all_tokens=None):
        """-> (table, copies): copies is an int32 [n, 2] array of (src, dst) block pairs."""
        cap = (length + n_new) // self.block_size + 2
        t = np.empty(max(cap, len(table)), np.int32)
        t[:len(table)] = table
        n = ctypes.c_int(len(table))
        src, dst = np.empty(cap, np.int32), np.empty(cap, np.int32)
        nc = ctypes.c_int(0)
        at = None if all_tokens is None else self._i32(all_tokens)
        _check("pkv_pool_append", self._lib.pkv_pool_append(
            self._h, t.ctypes.data, ctypes.byref(n), len(t), int(length), int(n_new),
            None if at is None else at.ctypes.data, src.ctypes.data, dst.ctypes.data, cap,
            ctypes.byref(nc)))
        return t[:n.value].copy(), np.stack([src[:nc.value], dst[:nc.value]], axis=1)

    def stats(self) -> dict:
        v = [ctypes.c_int(0) for _ in range(5)]
        _check("pkv_pool_stats", self._lib.pkv_pool_stats(self._h, *[ctypes.byref(x) for x in v]))
        return dict(zip(("total", "used", "shared", "free", "warm"), (x.value for x in v)))

    def refcount(self, block: int) -> int:
        r = self._lib.pkv_pool_refcount(self._h, int(block))
        if r < 0:
            raise PkvError("pkv_pool_refcount", r)
        return r
