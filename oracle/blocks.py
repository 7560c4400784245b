"""TEST INFRASTRUCTURE ONLY: a plain Python model of the host KV block pool.

Only ``tests/`` may import this module. It restates, in the simplest form, the block pool of
the Ollama memory-management page (§三 KV Cache内存管理的工程实现 and §三's copy-on-write
paragraph), with the readings the page leaves open made explicit:

* A pool of ``num_blocks`` fixed-size blocks; a FIFO free list (allocation takes the front,
  freed blocks go to the back); a reference count per block.
* Prefix index: the page hashes token ids with 64-bit FNV-1a (offset basis
  0xcbf29ce484222325, prime 0x100000001b3, each u32 token xor-ed in whole, then multiplied)
  over block-sized windows and calls the result a hash chain. Reading: block k of a sequence
  is keyed by the FNV-1a state after its last token, continued from block k-1's (the hash of
  the whole prefix), so that a block is only ever shared under the same preceding tokens. Only
  full blocks are indexed. A candidate is accepted only if its token ids and its parent block
  (the block matched just before it) equal the request's: the token-level verification the
  page asks for against collisions.
* allocate(tokens, max_tokens): walk the prompt's full blocks from the start, reusing indexed
  blocks while they match (reference +1), stop at the first miss; then take
  ceil((max_tokens - reused tokens) / block_size) new blocks (reference 1) and index the new
  full prompt blocks.
* release(table): reference -1 per block; a block that reaches 0 goes to the back of the free
  list and leaves the index.
* Leaving the index: a block's indexed descendants (children matched under it, their children,
  ...) leave the index with it, because its id may then be handed out for other tokens and a
  child's parent check would no longer prove its prefix. Descendants no sequence holds go to
  the back of the free list, a block before its own descendants, children in registration
  order.
* warm(tokens): index a prompt's full blocks without a sequence holding them (reference 0,
  off the free list): the page's pre-warmed system prompt.
* eviction: while the free list is short, the oldest (by allocation) indexed block no sequence
  holds (a warm one) is reclaimed (the page's LRU proxy); blocks a sequence holds are never
  taken. Fewer free and warm blocks than asked for: out of memory (no change).
* fork(table): a child sharing every block of its parent (reference +1 each).
* append(table, length, n_new, new_tokens): make room for positions [length, length + n_new):
  a position past the table takes a new block; a position in a block other sequences also
  hold (reference > 1) first copies that block to a new one (the page's copy-on-write: the
  shared block stays read-only for the others) and the sequence switches to the copy. Blocks
  that become full are indexed when their parent is.
"""
from __future__ import annotations

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a(tokens, h: int = FNV_OFFSET) -> int:
    for t in tokens:
        h ^= int(t) & 0xFFFFFFFF
        h = (h * FNV_PRIME) & MASK64
    return h


class OutOfBlocks(Exception):
    pass


class BlockPool:
    def __init__(self, num_blocks: int, block_size: int, hash_bits: int = 64):
        self.nb, self.bs = num_blocks, block_size
        self.hash_mask = MASK64 if hash_bits >= 64 else (1 << hash_bits) - 1
        self.ref = [0] * num_blocks
        self.free = list(range(num_blocks))
        self.key = [None] * num_blocks          # index key of an indexed block
        self.chain = [0] * num_blocks           # FNV state after the block's last token
        self.toks = [None] * num_blocks         # token ids of an indexed block
        self.parent = [-1] * num_blocks         # block matched before it (-1: first block)
        self.kids = [[] for _ in range(num_blocks)]   # indexed children, registration order
        self.stamp = [0] * num_blocks           # allocation order
        self.clock = 0
        self.index = {}                         # key -> [blocks], in registration order

    # ---------------------------------------------------------------- internals
    def _take(self, n):
        warm = [b for b in range(self.nb) if self.ref[b] == 0 and self.key[b] is not None]
        if len(self.free) + len(warm) < n:
            raise OutOfBlocks()
        while len(self.free) < n:
            oldest = min((self.stamp[b], b) for b in range(self.nb)
                         if self.ref[b] == 0 and self.key[b] is not None)[1]
            self.free.append(oldest)
            self._unindex(oldest)
        out = []
        for _ in range(n):
            b = self.free.pop(0)
            self.clock += 1
            self.stamp[b] = self.clock
            out.append(b)
        return out

    def _unindex(self, b):
        k = self.key[b]
        if k is None:
            return
        lst = self.index[k]
        lst.remove(b)
        if not lst:
            del self.index[k]
        if self.parent[b] >= 0 and b in self.kids[self.parent[b]]:
            self.kids[self.parent[b]].remove(b)
        self.key[b] = None
        self.toks[b] = None
        kids, self.kids[b] = self.kids[b], []
        for c in kids:
            if self.key[c] is None:
                continue
            self.parent[c] = -1
            if self.ref[c] == 0:
                self.free.append(c)
            self._unindex(c)

    def _index_block(self, b, parent, chain, toks):
        k = chain & self.hash_mask
        self.key[b], self.chain[b], self.toks[b], self.parent[b] = k, chain, list(toks), parent
        self.index.setdefault(k, []).append(b)
        if parent >= 0:
            self.kids[parent].append(b)

    def _match(self, parent, chain, toks):
        for b in self.index.get(chain & self.hash_mask, []):
            if self.toks[b] == list(toks) and self.parent[b] == parent:
                return b
        return -1

    # ---------------------------------------------------------------- operations
    def allocate(self, tokens, max_tokens=None):
        tokens = [int(t) for t in tokens]
        max_tokens = len(tokens) if max_tokens is None else max(max_tokens, len(tokens))
        bs = self.bs
        table, parent, h, pos = [], -1, FNV_OFFSET, 0
        while pos + bs <= len(tokens):
            h2 = fnv1a(tokens[pos:pos + bs], h)
            b = self._match(parent, h2, tokens[pos:pos + bs])
            if b < 0:
                break
            table.append(b)
            parent, h, pos = b, h2, pos + bs
        reused = len(table)
        need = -(-(max_tokens - pos) // bs)
        for b in table:                 # held first, so that eviction cannot take them
            self.ref[b] += 1
        try:
            new = self._take(need)
        except OutOfBlocks:
            for b in table:
                self.ref[b] -= 1
            raise
        for b in new:
            self.ref[b] = 1
            if pos + bs <= len(tokens):
                h2 = fnv1a(tokens[pos:pos + bs], h)
                self._index_block(b, parent, h2, tokens[pos:pos + bs])
                parent, h = b, h2
            pos += bs
            table.append(b)
        return table, reused

    def warm(self, tokens):
        full = (len(tokens) // self.bs) * self.bs
        table, reused = self.allocate(list(tokens)[:full])
        for b in table:
            self.ref[b] -= 1
        return table, reused

    def release(self, table):
        for b in table:
            self.ref[b] -= 1
            assert self.ref[b] >= 0
            if self.ref[b] == 0:
                self.free.append(b)
                self._unindex(b)

    def fork(self, table):
        for b in table:
            self.ref[b] += 1
        return list(table)

    def append(self, table, length, n_new, new_tokens=None, all_tokens=None):
        """Returns (table, copies): copies are (src, dst) block pairs to copy before writing."""
        table = list(table)
        bs = self.bs
        if n_new == 0:
            return table, []
        first, last = length // bs, (length + n_new - 1) // bs
        # the blocks this append writes: past the table (new) or held by others (copied)
        todo = [j for j in range(first, last + 1)
                if j >= len(table) or self.ref[table[j]] > 1]
        fresh = self._take(len(todo))           # all or nothing
        copies = []
        for j, d in zip(todo, fresh):
            self.ref[d] = 1
            if j < len(table):
                self.ref[table[j]] -= 1
                copies.append((table[j], d))
                table[j] = d
            else:
                table.append(d)
        if all_tokens is not None:
            self._index_filled(table, length, n_new, all_tokens)
        return table, copies

    def _index_filled(self, table, length, n_new, all_tokens):
        bs = self.bs
        for j in range(length // bs, (length + n_new) // bs):
            if (j + 1) * bs > length + n_new or self.key[table[j]] is not None:
                continue
            parent = table[j - 1] if j > 0 else -1
            if j > 0 and self.key[parent] is None:
                continue
            h = self.chain[parent] if j > 0 else FNV_OFFSET
            toks = [int(t) for t in all_tokens[j * bs:(j + 1) * bs]]
            self._index_block(table[j], parent, fnv1a(toks, h), toks)

    def stats(self):
        used = sum(1 for r in self.ref if r > 0)
        shared = sum(1 for r in self.ref if r > 1)
        warm = sum(1 for b in range(self.nb) if self.ref[b] == 0 and self.key[b] is not None)
        return {"total": self.nb, "used": used, "shared": shared, "free": len(self.free),
                "warm": warm}
