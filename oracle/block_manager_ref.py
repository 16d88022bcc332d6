"""Reference model of the host block manager: free pool, refcounts, copy-on-write.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Semantics restated from the pages:
- "PagedAttention" (robocikowo.com), "Komponenty": a block manager hands out and
  takes back physical blocks and keeps a pool of free ones; prefix blocks are
  shared through per-block reference counts and duplicated lazily when one
  sharer modifies them.  "Jak dziala": blocks are allocated on demand as a
  sequence grows, and a write into a shared block triggers the copy.
- analyticslegends.ai concept sheet, "Pourquoi c'est important": pages are
  allocated on demand and freed one by one when the request ends.
- ayinedjimi-consultants.fr glossary, "Definition": unused blocks are recycled
  immediately; N sampled candidates share the prompt's blocks until they diverge.

Allocation policy (a choice made here, stated so the model and the library
can be compared id for id): the free pool is a stack; it starts so that block
0 is handed out first, then 1, 2, ...; a freed block is pushed on top and is
the next one handed out; a sequence's blocks are released from its last
logical block to its first.

Prefix caching (restated from "PagedAttention et RadixAttention : parlons de
KV Cache", aitalk.it, "Deux couches, pas deux rivaux" and "Au-dela"): each
full block gets a key hashed from its parent's key, a per-tenant salt and its
own tokens, so equal prefixes give equal key chains.  The hash is 64-bit
FNV-1a, written here from its published definition (offset basis
0xcbf29ce484222325, prime 0x100000001b3, xor then multiply, per byte) over the
little-endian bytes of (parent key, salt, each token as int32).  A hit also
compares the stored tokens, parent key and salt.  Only the leading run of hits
is shared; fresh full blocks are keyed unless their key is already taken.  A
keyed block at refcount 0 stays cached; allocation takes a free block first,
else evicts the least recently released cached block.
"""
from __future__ import annotations

from collections import OrderedDict

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    h = FNV_OFFSET
    for b in data:
        h = ((h ^ b) * FNV_PRIME) & MASK64
    return h


def block_key(parent: int, salt: int, tokens) -> int:
    data = parent.to_bytes(8, "little") + (salt & MASK64).to_bytes(8, "little")
    data += b"".join((int(t) & 0xFFFFFFFF).to_bytes(4, "little") for t in tokens)
    return fnv1a64(data)


class NoBlocks(Exception):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("bad pool")
        self.block_size = block_size
        self.free = list(range(num_blocks - 1, -1, -1))  # top of stack = end of list
        self.ref = [0] * num_blocks
        self.seqs: dict[int, tuple[list[int], int]] = {}
        self.key: dict[int, tuple] = {}          # block -> (key, parent, salt, tokens)
        self.index: dict[int, int] = {}          # key -> block
        self.lru: OrderedDict[int, None] = OrderedDict()   # cached blocks, first = evicted first

    def _available(self) -> int:
        return len(self.free) + len(self.lru)

    def _alloc(self) -> int:
        if self.free:
            b = self.free.pop()
        elif self.lru:
            b, _ = self.lru.popitem(last=False)
            k = self.key.pop(b)
            if self.index.get(k[0]) == b:
                del self.index[k[0]]
        else:
            raise NoBlocks()
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        if b in self.key:
            self.lru[b] = None
        else:
            self.free.append(b)

    def _lookup(self, key, parent, salt, tokens):
        b = self.index.get(key)
        if b is None:
            return None
        k = self.key[b]
        return b if (k[1], k[2], k[3]) == (parent, salt & MASK64, tuple(tokens)) else None

    def add_seq_cached(self, seq_id: int, tokens, salt: int = 0) -> int:
        if seq_id in self.seqs:
            raise ValueError("bad seq")
        bs, n = self.block_size, len(tokens)
        nfull, nblocks = n // bs, -(-n // bs)
        keys, hits, parent, hitting = [], [], 0, True
        for i in range(nfull):
            tk = tokens[i * bs:(i + 1) * bs]
            k = block_key(parent, salt, tk)
            keys.append(k)
            if hitting:
                b = self._lookup(k, parent, salt, tk)
                if b is None:
                    hitting = False
                else:
                    hits.append(b)
            parent = k
        lru_hits = sum(1 for b in hits if b in self.lru)
        if nblocks - len(hits) > self._available() - lru_hits:
            raise NoBlocks()
        blocks = []
        for b in hits:
            self.lru.pop(b, None)
            self.ref[b] += 1
            blocks.append(b)
        for i in range(len(hits), nblocks):
            b = self._alloc()
            blocks.append(b)
            if i < nfull and keys[i] not in self.index:
                self.key[b] = (keys[i], keys[i - 1] if i else 0, salt & MASK64,
                               tuple(tokens[i * bs:(i + 1) * bs]))
                self.index[keys[i]] = b
        self.seqs[seq_id] = (blocks, n)
        return len(hits) * bs

    def register_blocks(self, seq_id: int, tokens, salt: int = 0) -> int:
        blocks, n = self.seqs[seq_id]
        if n != len(tokens):
            raise ValueError("length mismatch")
        bs, parent, added = self.block_size, 0, 0
        for i in range(n // bs):
            tk = tokens[i * bs:(i + 1) * bs]
            k = block_key(parent, salt, tk)
            b = blocks[i]
            if b not in self.key and k not in self.index:
                self.key[b] = (k, parent, salt & MASK64, tuple(tk))
                self.index[k] = b
                added += 1
            parent = k
        return added

    def num_cached(self) -> int:
        return len(self.lru)

    def add_seq(self, seq_id: int, num_tokens: int) -> None:
        if seq_id in self.seqs or num_tokens < 0:
            raise ValueError("bad seq")
        need = -(-num_tokens // self.block_size)
        if need > self._available():
            raise NoBlocks()
        self.seqs[seq_id] = ([self._alloc() for _ in range(need)], num_tokens)

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.seqs or child in self.seqs:
            raise ValueError("bad fork")
        blocks, n = self.seqs[parent]
        for b in blocks:
            self.ref[b] += 1
        self.seqs[child] = (list(blocks), n)

    def append_slot(self, seq_id: int):
        """Reserve the slot of the sequence's next token.  Returns
        (slot, cow_src, cow_dst); cow_* are -1 when no copy is needed."""
        blocks, n = self.seqs[seq_id]
        off = n % self.block_size
        cow = (-1, -1)
        if off == 0:
            blocks.append(self._alloc())
        else:
            last = blocks[-1]
            if self.ref[last] > 1:
                new = self._alloc()
                self.ref[last] -= 1
                blocks[-1] = new
                cow = (last, new)
        self.seqs[seq_id] = (blocks, n + 1)
        return blocks[-1] * self.block_size + off, cow[0], cow[1]

    def free_seq(self, seq_id: int) -> None:
        blocks, _ = self.seqs.pop(seq_id)
        for b in reversed(blocks):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self._release(b)

    def block_table(self, seq_id: int) -> list[int]:
        return list(self.seqs[seq_id][0])

    def num_tokens(self, seq_id: int) -> int:
        return self.seqs[seq_id][1]

    def num_free(self) -> int:
        return self._available()

    def refcount(self, block: int) -> int:
        return self.ref[block]

    def move_seq(self, to: "BlockManagerModel", seq_id: int):
        """Move a sequence to another pool; returns the (from, to) block pairs.
        Every block must be unshared; fails without changes otherwise or when
        the target is short."""
        blocks, n = self.seqs[seq_id]
        if seq_id in to.seqs or to.block_size != self.block_size:
            raise ValueError("bad move")
        if any(self.ref[b] != 1 for b in blocks):
            raise ValueError("shared block")
        if len(blocks) > to._available():
            raise NoBlocks()
        new = [to._alloc() for _ in blocks]
        for b in reversed(blocks):
            self.ref[b] = 0
            self._release(b)
        del self.seqs[seq_id]
        to.seqs[seq_id] = (new, n)
        return list(zip(blocks, new))
