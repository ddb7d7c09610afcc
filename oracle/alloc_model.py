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

Prefix caching (optional), restated from the continuous-batching page's
"Prefix 캐싱" and "제거" (eviction) sections:
  * a sequence created with known prompt ids and extended with known token
    ids has each block that becomes full recorded under its whole prefix (the
    tuple of ids from position 0 to the block's end) unless that prefix is
    already recorded;
  * a new sequence with a prompt takes, block by block from the first, the
    recorded block of each full-block prefix of the prompt while there is
    one (one more reference each); the tokens they cover need no prefill;
  * a recorded block whose count reaches 0 keeps its record and goes to a
    list of initialized free blocks instead of the free list; taking a block
    uses the free list first, and when it is empty the most recently freed
    initialized block loses its record and is taken;
  * appending without an id ends the recording for that sequence.
The keys here are the exact id tuples (no hashing).
"""
from __future__ import annotations

import copy


class RefCountError(RuntimeError):
    pass


class BlockAllocatorModel:
    def __init__(self, num_blocks: int, block_size: int, prefix_cache: bool = False):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.prefix_cache = prefix_cache
        self.free = list(range(num_blocks))
        self.ref = [0] * num_blocks
        self.seqs: dict[int, dict] = {}
        self.init: list = []             # initialized free blocks, oldest first
        self.record: dict = {}           # prefix id tuple -> block
        self.key_of: dict = {}           # block -> its prefix id tuple

    # -- pool ---------------------------------------------------------------
    def _take(self) -> int:
        if self.free:
            b = self.free.pop()
        elif self.init:
            b = self.init.pop()
            del self.record[self.key_of.pop(b)]
        else:
            raise MemoryError("no free KV cache blocks")
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        if self.ref[b] <= 0:
            raise RefCountError(f"block {b} released with count {self.ref[b]}")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            (self.init if b in self.key_of else self.free).append(b)

    # -- sequences ----------------------------------------------------------
    def add_seq(self, seq_id: int) -> None:
        if seq_id in self.seqs:
            raise ValueError(f"sequence {seq_id} exists")
        self.seqs[seq_id] = {"blocks": [], "len": 0, "ids": None}

    def add_seq_prefix(self, seq_id: int, prompt) -> int:
        """New sequence with known prompt ids; returns the tokens covered by
        recorded blocks it takes over."""
        if seq_id in self.seqs:
            raise ValueError(f"sequence {seq_id} exists")
        B = self.block_size
        blocks = []
        prompt = [int(t) for t in prompt]
        if self.prefix_cache:
            while (len(blocks) + 1) * B <= len(prompt):
                key = tuple(prompt[: (len(blocks) + 1) * B])
                if key not in self.record:
                    break
                b = self.record[key]
                if self.ref[b] == 0:
                    self.init.remove(b)
                self.ref[b] += 1
                blocks.append(b)
        n = len(blocks) * B
        self.seqs[seq_id] = {"blocks": blocks, "len": n, "ids": prompt[:n]}
        return n

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.seqs or child in self.seqs:
            raise ValueError("bad fork")
        p = self.seqs[parent]
        for b in p["blocks"]:
            self.ref[b] += 1
        self.seqs[child] = {"blocks": list(p["blocks"]), "len": p["len"],
                            "ids": None if p["ids"] is None else list(p["ids"])}

    def free_seq(self, seq_id: int) -> None:
        if seq_id not in self.seqs:
            raise ValueError(f"no sequence {seq_id}")
        for b in self.seqs[seq_id]["blocks"]:
            self._release(b)
        del self.seqs[seq_id]

    def _append_one(self, seq_id: int, pairs: list, token=None) -> int:
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
        if sq["ids"] is not None:
            if token is None:
                sq["ids"] = None
            else:
                sq["ids"].append(int(token))
                if self.prefix_cache and sq["len"] % B == 0:
                    key = tuple(sq["ids"])
                    if key not in self.record:
                        self.record[key] = sq["blocks"][-1]
                        self.key_of[sq["blocks"][-1]] = key
        return slot

    def append_slots(self, seq_ids, token_ids=None):
        """One new token for each listed sequence, in list order (with its id
        if ``token_ids`` is given).  Returns (slots, copy_pairs).
        All-or-nothing on MemoryError."""
        for s in seq_ids:
            if s not in self.seqs:
                raise ValueError(f"no sequence {s}")
        if len(set(seq_ids)) != len(seq_ids):
            raise ValueError("a sequence is listed twice")
        toks = [None] * len(seq_ids) if token_ids is None else list(token_ids)
        saved = copy.deepcopy((self.free, self.ref, self.seqs, self.init, self.record, self.key_of))
        pairs: list = []
        try:
            slots = [self._append_one(s, pairs, t) for s, t in zip(seq_ids, toks)]
        except MemoryError:
            self.free, self.ref, self.seqs, self.init, self.record, self.key_of = saved
            raise
        return slots, pairs

    # -- queries ------------------------------------------------------------
    def table(self, seq_id: int):
        return list(self.seqs[seq_id]["blocks"])

    def length(self, seq_id: int) -> int:
        return self.seqs[seq_id]["len"]

    def num_free(self) -> int:
        return len(self.free) + len(self.init)

    def prefix_stats(self):
        return len(self.record), len(self.init)
