"""Plain-Python model of the KV block manager -- TEST INFRASTRUCTURE ONLY.

What it models (pages: "anthology-of-the-sota note-023", Method and Concepts; "Paged
Attention" glossary, paragraphs 1-3; "PagedAttention & Continuous Batching", the
shared-system-prompt paragraph):

* a sequence's tokens fill fixed-size blocks; a block is taken only when a token
  needs it (on-demand allocation);
* sequences may share physical blocks by reference (a fork: parallel sampling or
  beam search from one prompt);
* a sequence about to write into a block that others still share first gets its
  own copy of it (copy-on-write); the others keep the original;
* a finished sequence drops its references; blocks nobody references are free again
  and are the first handed out next.

Policy the pages leave open, fixed here the same way as the library: free blocks
form a stack whose top is handed out first, initially yielding 0, 1, 2, ...; a
finished sequence's blocks are pushed back last-block-first, so its first block is
reused first.  Only the tests import this module.
"""
from __future__ import annotations


class OutOfBlocks(Exception):
    pass


class BlockManagerModel:
    def __init__(self, num_blocks: int, block_size: int):
        self.num_blocks, self.block_size = num_blocks, block_size
        self.free = list(range(num_blocks - 1, -1, -1))  # top of the stack = end of the list
        self.refs = [0] * num_blocks
        self.filled = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        self.swapped: dict[int, int] = {}
        self.copies = 0

    def _take(self) -> int:
        b = self.free.pop()
        self.refs[b] = 1
        self.filled[b] = 0
        return b

    def add_sequence(self, seq: int, tokens: int) -> None:
        assert seq not in self.tables and seq not in self.swapped
        need = -(-tokens // self.block_size)
        if need > len(self.free):
            raise OutOfBlocks
        blocks = []
        for i in range(need):
            b = self._take()
            self.filled[b] = min(self.block_size, tokens - i * self.block_size)
            blocks.append(b)
        self.tables[seq], self.lens[seq] = blocks, tokens

    def fork(self, parent: int, child: int) -> None:
        assert child not in self.tables and child not in self.swapped
        for b in self.tables[parent]:
            self.refs[b] += 1
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]

    def append(self, seqs: list[int]):
        """One new token for each sequence, in order: (slots, copy-on-write pairs)."""
        assert len(set(seqs)) == len(seqs)
        # count fresh blocks first so that a failure changes nothing
        refs = dict()
        need = 0
        for s in seqs:
            if self.lens[s] % self.block_size == 0:
                need += 1
            else:
                b = self.tables[s][-1]
                r = refs.get(b, self.refs[b])
                if r > 1:
                    need += 1
                    r -= 1
                refs[b] = r
        if need > len(self.free):
            raise OutOfBlocks
        slots, pairs = [], []
        for s in seqs:
            row = self.lens[s] % self.block_size
            if row == 0:
                self.tables[s].append(self._take())
            elif self.refs[self.tables[s][-1]] > 1:
                old = self.tables[s][-1]
                fresh = self._take()
                self.filled[fresh] = self.filled[old]
                self.refs[old] -= 1
                self.tables[s][-1] = fresh
                pairs.append((old, fresh))
                self.copies += 1
            b = self.tables[s][-1]
            slots.append(b * self.block_size + row)
            self.filled[b] = max(self.filled[b], row + 1)
            self.lens[s] += 1
        return slots, pairs

    def free_sequence(self, seq: int) -> None:
        for b in reversed(self.tables.pop(seq)):
            self.refs[b] -= 1
            if self.refs[b] == 0:
                self.filled[b] = 0
                self.free.append(b)
        del self.lens[seq]

    def swap_out(self, seq: int) -> list[int]:
        """Preempted: its blocks (to copy to CPU memory) are released; the length is kept."""
        blocks = self.tables[seq]
        n = self.lens[seq]
        self.free_sequence(seq)
        self.swapped[seq] = n
        return blocks

    def swap_in(self, seq: int) -> list[int]:
        """Restored into fresh private blocks (to copy the saved data back into)."""
        n = self.swapped[seq]
        if -(-n // self.block_size) > len(self.free):
            raise OutOfBlocks
        del self.swapped[seq]
        self.add_sequence(seq, n)
        return list(self.tables[seq])

    def stats(self) -> dict:
        used = [b for b in range(self.num_blocks) if self.refs[b] > 0]
        return dict(num_blocks=self.num_blocks, free_blocks=len(self.free), used_blocks=len(used),
                    num_sequences=len(self.tables),
                    shared_blocks=sum(1 for b in used if self.refs[b] > 1),
                    stored_tokens=sum(self.filled[b] for b in used),
                    logical_tokens=sum(self.lens.values()),
                    allocated_slots=len(used) * self.block_size,
                    max_len=max(self.lens.values(), default=0), copies=self.copies, swapped=len(self.swapped))
