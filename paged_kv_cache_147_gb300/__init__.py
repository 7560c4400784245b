"""Paged KV-cache decode attention for GB300 (sm_103a).

The compute lives in ``libpkv.so`` (hand-written CUDA behind a C ABI, declared in
``include/pkv.h``); :mod:`paged_kv_cache_147_gb300.pkv` is the thin ctypes binding that
marshals torch tensors into it. :mod:`paged_kv_cache_147_gb300.workloads` draws the seeded
synthetic inputs. The library is loaded on first use and a missing or unloadable library is
an error: there is no CPU fallback.
"""
__all__ = ["pkv", "workloads"]
