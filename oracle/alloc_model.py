"""Reference model of the paged KV-cache block manager (host side).

TEST INFRASTRUCTURE ONLY: the tests compare the C++ allocator of the library
against this model operation by operation.

Semantics, restated from the block manager described on the blog page
("アルゴリズムの擬似コード" section of the PagedAttention post) and from the
paper summary (sections 5 and 6: on-demand blocks, return to the pool when a
sequence ends, reference counts and copy-on-write for parallel sampling and
beam search):
  * the pool starts with every block free; the free list is ordered
    0..N-1 and a block is taken from its END, so the first block handed out
    is N-1;
  * a taken block has reference count 1; releasing a reference decrements
    it, and a block whose count reaches 0 is appended to the free list;
  * appending a token to a sequence: with no block yet, take one; if the
    last block is full, take a new one; otherwise, if the last block is
    shared (count > 1), take a new block, record (old, new) as a block copy,
    drop one reference from the old block and put the new one in its place
    (copy-on-write); the token goes to slot (length mod B) of the last block;
  * fork: a child sequence receives the parent's block list and length and
    every block gains a reference (the sharing of section 6);
  * freeing a sequence releases its blocks in logical order.
Taking a block from an empty free list is an error (the pseudo-code raises
MemoryError); a batch of appends that cannot be served changes nothing.
"""
from __future__ import annotations

import copy


class RefCountError(RuntimeError):
    pass


class BlockAllocatorModel:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = list(range(num_blocks))
        self.ref = [0] * num_blocks
        self.seqs: dict[int, dict] = {}

    # -- pool ---------------------------------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise MemoryError("no free KV cache blocks")
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        if self.ref[b] <= 0:
            raise RefCountError(f"block {b} released with count {self.ref[b]}")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    # -- sequences ----------------------------------------------------------
    def add_seq(self, seq_id: int) -> None:
        if seq_id in self.seqs:
            raise ValueError(f"sequence {seq_id} exists")
        self.seqs[seq_id] = {"blocks": [], "len": 0}

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.seqs or child in self.seqs:
            raise ValueError("bad fork")
        p = self.seqs[parent]
        for b in p["blocks"]:
            self.ref[b] += 1
        self.seqs[child] = {"blocks": list(p["blocks"]), "len": p["len"]}

    def free_seq(self, seq_id: int) -> None:
        if seq_id not in self.seqs:
            raise ValueError(f"no sequence {seq_id}")
        for b in self.seqs[seq_id]["blocks"]:
            self._release(b)
        del self.seqs[seq_id]

    def _append_one(self, seq_id: int, pairs: list) -> int:
        sq = self.seqs[seq_id]
        B = self.block_size
        if not sq["blocks"]:
            sq["blocks"].append(self._take())
        filled = sq["len"] - (len(sq["blocks"]) - 1) * B
        if filled >= B:
            sq["blocks"].append(self._take())
            filled = 0
        elif self.ref[sq["blocks"][-1]] > 1:
            old = sq["blocks"][-1]
            new = self._take()
            pairs.append((old, new))
            self.ref[old] -= 1
            sq["blocks"][-1] = new
        slot = sq["blocks"][-1] * B + filled
        sq["len"] += 1
        return slot

    def append_slots(self, seq_ids):
        """One new token for each listed sequence, in list order.  Returns
        (slots, copy_pairs).  All-or-nothing on MemoryError."""
        for s in seq_ids:
            if s not in self.seqs:
                raise ValueError(f"no sequence {s}")
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence is listed twice")
        saved = (list(self.free), list(self.ref), copy.deepcopy(self.seqs))
        pairs: list = []
        try:
            slots = [self._append_one(s, pairs) for s in seq_ids]
        except MemoryError:
            self.free, self.ref, self.seqs = saved
            raise
        return slots, pairs

    # -- queries ------------------------------------------------------------
    def table(self, seq_id: int):
        return list(self.seqs[seq_id]["blocks"])

    def length(self, seq_id: int) -> int:
        return self.seqs[seq_id]["len"]

    def num_free(self) -> int:
        return len(self.free)
