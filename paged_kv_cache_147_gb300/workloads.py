"""Seeded synthetic workloads for paged decode attention.

This module only draws inputs: shapes, context lengths, block allocations (which physical
block each sequence owns and how many tokens each block holds) and N(0, 1) fp16 tensors.
It holds none of the attention, addressing or slot arithmetic; the CUDA library and the
CPU oracle both take what it produces as plain arrays.

Recipes (the shapes follow the workloads the pages discuss):

* ``tiny``     1 layer, 12 q / 2 KV heads, d 128, 64 blocks x 16 tokens, 2 sequences with
               37 and 100 cached tokens, one appended token each (context 38 and 101); the
               two block tables are disjoint slices of one seeded permutation of the pool.
* ``edge_1p1b`` the 1.1B edge model of the embedded PagedAttention page: 24 layers,
               12 q / 2 KV heads, d 128, 16-token blocks, 64 sequences with context
               U_int[16, 2048] (after the append), blocks shuffled across the pool.
* ``llama70b_b16`` / ``llama70b_mixed`` one 70B-class attention stack as in the vLLM memory
               page's example: 80 layers, 64 q / 8 KV heads, d 128, 16-token blocks; batch 16
               at 4096 tokens, or batch 32 with lognormal lengths clipped to [50, 8000]
               (median 632.5, sigma 1.269, which puts 50 and 8000 at -/+ 2 sigma).
* ``prefix``   1 layer, MHA 32 / 32 heads, d 128, 64-token blocks; 64 sequences whose tables
               start with the same 4 blocks (256 shared tokens) and continue with private
               suffixes of U_int[32, 1024] tokens; sequences 60..63 are the four children of
               one forked parent whose partly filled last block they share.
* ``prefill_70b`` a chunked-prefill step of the 70B-class stack (the vLLM memory page's
               chunked prefill): 64 q / 8 KV heads, d 128, 16-token blocks, 16 sequences whose
               512-token chunk ends at context 4096 (3584 tokens cached before it), 4 layers.
               ``prefill(...)`` builds smaller chunked-prefill cases with given lengths.
* ``ring``     sink + ring streaming cache: 12 q / 2 KV heads, d 128, 16-token blocks, sink
               4, window 1020 (64 shuffled blocks per sequence), 32 sequences at logical
               lengths U_int[2000, 100000] (every ring slot holds data).

Context lengths count the tokens in cache after this step's append. fp16 values are drawn
as float32 N(0, 1) from a seeded ``torch.Generator`` and rounded to fp16; integer structure
comes from numpy's PCG64 with the recipe's seed.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int                 # physical blocks per layer
    q_len: int                      # new tokens (queries) per sequence this step
    context_lens: np.ndarray        # int32 [B], after the append
    block_tables: np.ndarray        # int32 [B, max_blocks], -1 where unused
    block_fill: np.ndarray          # int32 [num_blocks], tokens held before the append
    free_blocks: np.ndarray         # int32, unowned block ids (for copy-on-write targets)
    refcount: np.ndarray            # int32 [num_blocks], tables referencing each block
    # streaming-cache fields (ring workloads only)
    sink: int = 0
    window: int = 0
    ring_len0: np.ndarray | None = None   # int64 [B], logical length before this step

    # ------------------------------------------------------------------ shape helpers
    @property
    def num_seqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def prior_lens(self) -> np.ndarray:
        return (self.context_lens - self.q_len).astype(np.int32)

    def pool_shape(self) -> tuple:
        return (self.num_layers, self.num_blocks, self.num_kv_heads, self.block_size,
                self.head_dim)

    def new_token_positions(self) -> tuple[np.ndarray, np.ndarray]:
        """(seq_ids int32 [B*q_len], positions int64 [B*q_len]) of this step's tokens."""
        if self.ring_len0 is not None:
            base = self.ring_len0.astype(np.int64)
        else:
            base = self.prior_lens.astype(np.int64)
        seq = np.repeat(np.arange(self.num_seqs, dtype=np.int32), self.q_len)
        pos = (base[:, None] + np.arange(self.q_len, dtype=np.int64)[None, :]).reshape(-1)
        return seq, pos

    # ------------------------------------------------------------------ tensors
    def _gen(self, layer: int, tag: int, device) -> torch.Generator:
        g = torch.Generator(device=device)
        g.manual_seed(self.seed * 1_000_003 + layer * 101 + tag)
        return g

    def _randn(self, shape, layer, tag, device) -> torch.Tensor:
        g = self._gen(layer, tag, device)
        return torch.randn(shape, generator=g, device=device, dtype=torch.float32).half()

    def draw(self, shape, layer: int, tag: int, device="cpu") -> torch.Tensor:
        """An extra seeded N(0, 1) fp16 tensor (tags >= 100 are free for callers)."""
        return self._randn(shape, layer, tag, device)

    def pools(self, device="cpu", poison: bool = False, layers=None):
        """K and V pools [num_layers, NB, Hkv, bs, D] fp16 (one tensor each, layer-strided).

        With ``poison`` the slots a block does not hold yet (per ``block_fill``) and every
        unowned block are NaN, so any read of them shows up in the output.
        """
        layers = range(self.num_layers) if layers is None else layers
        shape = self.pool_shape()
        k = torch.empty(shape, dtype=torch.float16, device=device)
        v = torch.empty(shape, dtype=torch.float16, device=device)
        for l in layers:
            k[l] = self._randn(shape[1:], l, 1, device)
            v[l] = self._randn(shape[1:], l, 2, device)
        if poison:
            fill = torch.as_tensor(self.block_fill, device=device)
            empty = torch.arange(self.block_size, device=device)[None, :] >= fill[:, None]
            mask = empty[None, :, None, :, None]
            k.masked_fill_(mask, float("nan"))
            v.masked_fill_(mask, float("nan"))
        return k, v

    def layer_pool(self, layer: int, device="cpu"):
        """One layer's K and V pools [NB, Hkv, bs, D] (the same values pools() puts there)."""
        shape = self.pool_shape()[1:]
        return self._randn(shape, layer, 1, device), self._randn(shape, layer, 2, device)

    def query(self, layer: int, device="cpu") -> torch.Tensor:
        """q [B, q_len, Hq, D] fp16."""
        return self._randn((self.num_seqs, self.q_len, self.num_q_heads, self.head_dim),
                           layer, 3, device)

    def new_kv(self, layer: int, device="cpu", tag: int = 0) -> tuple[torch.Tensor, torch.Tensor]:
        """This step's K, V rows [B*q_len, Hkv, D] fp16 (tag selects a later step's draw)."""
        shape = (self.num_seqs * self.q_len, self.num_kv_heads, self.head_dim)
        return (self._randn(shape, layer, 4 + 2 * tag, device),
                self._randn(shape, layer, 5 + 2 * tag, device))

    def kv_read_bytes(self) -> int:
        """fp16 K+V bytes one decode step reads over all layers (algorithmic, logical)."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_dim * 2 * 2 * self.num_layers


# ---------------------------------------------------------------------- allocation helper
def _allocate(rng: np.random.Generator, lens_after: np.ndarray, q_len: int, block_size: int,
              max_blocks: int, spare: int = 0):
    """Give each sequence ceil(len / bs) blocks drawn from one shuffled permutation.

    Returns (num_blocks, tables, fill, free, refcount); fill counts the tokens each block
    holds before the step's q_len appended tokens.
    """
    nblk = (lens_after + block_size - 1) // block_size
    total = int(nblk.sum()) + spare
    perm = rng.permutation(total).astype(np.int32)
    tables = np.full((len(lens_after), max_blocks), -1, dtype=np.int32)
    fill = np.zeros(total, dtype=np.int32)
    ref = np.zeros(total, dtype=np.int32)
    cur = 0
    for b, (n, L) in enumerate(zip(nblk, lens_after)):
        ids = perm[cur:cur + n]
        cur += n
        tables[b, :n] = ids
        prior = int(L) - q_len
        for j, blk in enumerate(ids):
            fill[blk] = max(0, min(block_size, prior - j * block_size))
            ref[blk] += 1
    return total, tables, fill, perm[cur:].copy(), ref


def tiny(seed: int = 0) -> Workload:
    rng = np.random.default_rng(seed)
    lens = np.array([38, 101], dtype=np.int32)
    perm = rng.permutation(64).astype(np.int32)
    tables = np.full((2, 7), -1, dtype=np.int32)
    tables[0, :3] = perm[0:3]
    tables[1, :7] = perm[3:10]
    fill = np.zeros(64, dtype=np.int32)
    ref = np.zeros(64, dtype=np.int32)
    for b in range(2):
        prior = int(lens[b]) - 1
        for j in range(int((lens[b] + 15) // 16)):
            fill[tables[b, j]] = max(0, min(16, prior - 16 * j))
            ref[tables[b, j]] += 1
    return Workload("tiny", seed, 1, 12, 2, 128, 16, 64, 1, lens, tables, fill, perm[10:].copy(),
                    ref)


def edge_1p1b(seed: int = 1, num_seqs: int = 64, num_layers: int = 24) -> Workload:
    rng = np.random.default_rng(seed)
    lens = rng.integers(16, 2048, size=num_seqs, endpoint=True).astype(np.int32)
    nb, tables, fill, free, ref = _allocate(rng, lens, 1, 16, 2048 // 16)
    return Workload("edge_1p1b", seed, num_layers, 12, 2, 128, 16, nb, 1, lens, tables, fill,
                    free, ref)


def llama70b_b16(seed: int = 2, num_layers: int = 80) -> Workload:
    rng = np.random.default_rng(seed)
    lens = np.full(16, 4096, dtype=np.int32)
    nb, tables, fill, free, ref = _allocate(rng, lens, 1, 16, 4096 // 16)
    return Workload("llama70b_b16", seed, num_layers, 64, 8, 128, 16, nb, 1, lens, tables, fill,
                    free, ref)


def llama70b_mixed(seed: int = 2, num_layers: int = 80) -> Workload:
    rng = np.random.default_rng(seed + 10_000)
    mu, sigma = math.log(632.5), 1.269
    lens = np.clip(np.rint(rng.lognormal(mu, sigma, size=32)), 50, 8000).astype(np.int32)
    nb, tables, fill, free, ref = _allocate(rng, lens, 1, 16, 8000 // 16)
    return Workload("llama70b_mixed", seed, num_layers, 64, 8, 128, 16, nb, 1, lens, tables,
                    fill, free, ref)


def prefix(seed: int = 3, private: bool = False) -> Workload:
    """64 sequences over one shared 4-block prefix; sequences 60..63 are forked children.
    With ``private`` every sequence gets its own copy of the 4 prefix blocks instead (the same
    lengths and fork, no cross-sequence sharing of the prefix): the comparison case for what
    sharing saves in DRAM traffic."""
    rng = np.random.default_rng(seed)
    bs, shared_blocks, n = 64, 4, 64
    suffix = rng.integers(32, 1024, size=n, endpoint=True).astype(np.int32)
    # the forked parent (used by sequences 60..63) must end inside a block: its prior
    # length (one token before the append) is not a multiple of the block size
    while (256 + int(suffix[60]) - 1) % bs == 0:
        suffix[60] += 1
    suffix[61:64] = suffix[60]
    lens = (256 + suffix).astype(np.int32)
    max_blocks = (256 + 1024 + bs - 1) // bs + 1
    # private blocks: sequences 0..59 one set each, 60..63 one set shared
    priv_counts = [(int(lens[b]) - 256 + bs - 1) // bs for b in range(61)]
    n_prefix = shared_blocks * (61 if private else 1)
    total = n_prefix + sum(priv_counts) + 8               # 8 spare blocks for copy-on-write
    perm = rng.permutation(total).astype(np.int32)
    shared = perm[:shared_blocks]
    cur = n_prefix
    tables = np.full((n, max_blocks), -1, dtype=np.int32)
    fill = np.zeros(total, dtype=np.int32)
    ref = np.zeros(total, dtype=np.int32)
    fill[shared] = bs
    for b in range(61):
        ids = perm[cur:cur + priv_counts[b]]
        cur += priv_counts[b]
        prior_priv = int(lens[b]) - 1 - 256
        for j, blk in enumerate(ids):
            fill[blk] = max(0, min(bs, prior_priv - j * bs))
        owners = [b] if b < 60 else [60, 61, 62, 63]
        if private:
            shared = perm[b * shared_blocks:(b + 1) * shared_blocks]
            fill[shared] = bs
        for o in owners:
            tables[o, :shared_blocks] = shared
            tables[o, shared_blocks:shared_blocks + len(ids)] = ids
            ref[shared] += 1
            ref[ids] += 1
    free = perm[cur:].copy()
    return Workload("prefix_private" if private else "prefix", seed, 1, 32, 32, 128, bs, total, 1,
                    lens, tables, fill, free, ref)


def prefill(seed: int, lens, q_len: int, num_q_heads: int, num_kv_heads: int,
            block_size: int = 16, num_layers: int = 1, name: str = "prefill") -> Workload:
    """A chunk of q_len new tokens per sequence; lens are the context lengths including the
    chunk (a length below q_len leaves the chunk's first queries with nothing to see)."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    max_blocks = int((lens.max() + block_size - 1) // block_size) + 1
    nb, tables, fill, free, ref = _allocate(rng, lens, q_len, block_size, max_blocks, spare=2)
    return Workload(name, seed, num_layers, num_q_heads, num_kv_heads, 128, block_size, nb,
                    q_len, lens, tables, fill, free, ref)


def prefill_70b(seed: int = 5, num_layers: int = 4) -> Workload:
    return prefill(seed, [4096] * 16, 512, 64, 8, 16, num_layers, name="prefill_70b")


def ring(seed: int = 4, num_seqs: int = 32, num_layers: int = 1, q_len: int = 4) -> Workload:
    """Sink + ring cache; ring_len0 = logical length before this step's q_len drafts."""
    rng = np.random.default_rng(seed)
    sink, window, bs = 4, 1020, 16
    cap_blocks = (sink + window) // bs
    L0 = rng.integers(2000, 100000, size=num_seqs, endpoint=True).astype(np.int64)
    perm = rng.permutation(num_seqs * cap_blocks).astype(np.int32)
    tables = perm.reshape(num_seqs, cap_blocks).copy()
    total = num_seqs * cap_blocks
    fill = np.full(total, bs, dtype=np.int32)            # every ring slot holds data
    ref = np.ones(total, dtype=np.int32)
    lens = (L0 + q_len).astype(np.int32)
    return Workload("ring", seed, num_layers, 12, 2, 128, bs, total, q_len, lens, tables, fill,
                    np.zeros(0, np.int32), ref, sink=sink, window=window, ring_len0=L0)


WORKLOADS = {
    "tiny": tiny,
    "edge_1p1b": edge_1p1b,
    "llama70b_b16": llama70b_b16,
    "llama70b_mixed": llama70b_mixed,
    "prefix": prefix,
    "ring": ring,
    "prefill_70b": prefill_70b,
}
