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

Allocation policy (a choice of this build, stated so the model and the library
can be compared id for id): the free pool is a stack; it starts so that block
0 is handed out first, then 1, 2, ...; a freed block is pushed on top and is
the next one handed out; a sequence's blocks are released from its last
logical block to its first.
"""
from __future__ import annotations


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

    def _alloc(self) -> int:
        if not self.free:
            raise NoBlocks()
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def add_seq(self, seq_id: int, num_tokens: int) -> None:
        if seq_id in self.seqs or num_tokens < 0:
            raise ValueError("bad seq")
        need = -(-num_tokens // self.block_size)
        if need > len(self.free):
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
                self.free.append(b)

    def block_table(self, seq_id: int) -> list[int]:
        return list(self.seqs[seq_id][0])

    def num_tokens(self, seq_id: int) -> int:
        return self.seqs[seq_id][1]

    def num_free(self) -> int:
        return len(self.free)

    def refcount(self, block: int) -> int:
        return self.ref[block]
