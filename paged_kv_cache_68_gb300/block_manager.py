"""Host-side block manager: free list, per-sequence block tables, reference
counts, copy-on-write planning and slot mapping.

This is the CPU half of the paged KV cache: it decides where every token's
K/V row lives and hands the GPU three small arrays -- block tables, a slot
mapping and a list of (src, dst) block copies -- which the CUDA library
consumes (``kv_append``, ``paged_attention_decode``, ``copy_blocks``).

Sources (page title and section):

* "Lecture 3: memory and prefix reuse in serving engines" (semidirectx.com,
  CS349D notes), sec. 3.1: blocks are handed out on demand, only when the
  last block is full, from anywhere in the pool; sec. 4.1: parallel sampling
  forks the table and sets every reference count to n; a write into a shared
  block allocates, copies, remaps and decrements before writing, so n samples
  cost n - 1 copies; sec. 4.2: a dropped branch decrements, a block returns
  to the free list at zero.
* "Lecture 24: PagedAttention and vLLM" (semidirectx.com, CMU 11-868 notes),
  answer 4: no copy at all when the prompt length is a multiple of the block
  size.
* "Part 3: single node" (random-liu.github.io), ch. 11 sec. 3 (block table)
  and ch. 13 sec. 1 (slot_mapping computed on the CPU).
* "S06 memory and KV cache: PagedAttention" (llminference.xinbetween.com),
  "block manager" (any free block will do; out of blocks -> the caller
  preempts) and the reference-count invariant: after every operation, the
  number of tables holding a block equals its count.
* The kwkr.cn blog's toy ``KVCacheManager``: prefill takes ceil(L / bs)
  blocks, decode takes one more block exactly when the new token starts a
  block, and running out raises ``RuntimeError("OOM")``.
* "Lecture 3", sec. 5.2 and "Part 3: single node", ch. 14 sec. 3: a preempted
  request's blocks are swapped out to CPU memory, handed out by a CPU block
  allocator, and swapped back in when it resumes; the swap space needed is
  bounded by the GPU pool.
"""

from __future__ import annotations

from collections import Counter
from typing import Dict, Iterable, List, Optional, Tuple


class OutOfBlocks(RuntimeError):
    """Raised when the free list is empty; the message carries "OOM"."""

    def __init__(self, what: str = ""):
        super().__init__(f"OOM: no free KV block{': ' + what if what else ''}")


class BlockManager:
    """Reference-counted allocator of fixed-size KV blocks.

    ``free_order`` fixes the order blocks leave the free list (the pages draw
    it shuffled); ``pop`` chooses the end they leave from: ``"front"``
    (first-in, first-out) or ``"back"`` (last-in, first-out).
    """

    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Optional[Iterable[int]] = None, pop: str = "front",
                 num_cpu_blocks: int = 0):
        if block_size < 1 or num_blocks < 0:
            raise ValueError("block_size must be >= 1 and num_blocks >= 0")
        if pop not in ("front", "back"):
            raise ValueError("pop must be 'front' or 'back'")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free: List[int] = list(range(num_blocks) if free_order is None else free_order)
        if sorted(self.free) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the block ids")
        self._pop_front = pop == "front"
        self.ref: List[int] = [0] * num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self.copies_made = 0
        # swap space: CPU blocks, their counts, and the sequences living there
        self.num_cpu_blocks = num_cpu_blocks
        self.cpu_free: List[int] = list(range(num_cpu_blocks))
        self.cpu_ref: List[int] = [0] * num_cpu_blocks
        self.swapped: set = set()

    # -- allocation ------------------------------------------------------
    def _take(self) -> int:
        if not self.free:
            raise OutOfBlocks()
        blk = self.free.pop(0) if self._pop_front else self.free.pop()
        self.ref[blk] = 1
        return blk

    def _release(self, blk: int) -> None:
        self.ref[blk] -= 1
        if self.ref[blk] < 0:
            raise AssertionError(f"reference count of block {blk} went negative")
        if self.ref[blk] == 0:
            self.free.append(blk)

    def num_free(self) -> int:
        return len(self.free)

    def blocks_for(self, n_tokens: int) -> int:
        return -(-n_tokens // self.block_size)

    def allocate_prompt(self, seq_id: int, n_tokens: int) -> List[int]:
        """Prefill: take ceil(n_tokens / bs) blocks at once (all or nothing)."""
        if seq_id in self.tables:
            raise ValueError(f"sequence {seq_id} already exists")
        need = self.blocks_for(n_tokens)
        if need > len(self.free):
            raise OutOfBlocks(f"prompt of {n_tokens} tokens needs {need} blocks")
        self.tables[seq_id] = [self._take() for _ in range(need)]
        self.lens[seq_id] = n_tokens
        return list(self.tables[seq_id])

    # -- swap to host ----------------------------------------------------
    def _group_blocks(self, seq_ids, on_cpu: bool) -> List[int]:
        """Distinct blocks of the group's tables, in first-use order; every one
        must be held by group members only (a block shared with a sequence
        outside the group cannot move)."""
        ids = list(seq_ids)
        for sid in ids:
            if (sid in self.swapped) != on_cpu:
                raise ValueError(f"sequence {sid} is {'not ' if on_cpu else ''}swapped out")
        held = Counter(b for sid in ids for b in self.tables[sid])
        refs = self.cpu_ref if on_cpu else self.ref
        for b, n in held.items():
            if refs[b] != n:
                raise ValueError(f"block {b} is shared outside the group")
        return list(dict.fromkeys(b for sid in ids for b in self.tables[sid]))

    def swap_out(self, seq_ids) -> List[Tuple[int, int]]:
        """Move a group's blocks to CPU blocks (all or nothing); returns the
        (gpu_block, cpu_block) pairs to copy device -> host, after which the
        GPU blocks are free."""
        blocks = self._group_blocks(seq_ids, on_cpu=False)
        if len(blocks) > len(self.cpu_free):
            raise OutOfBlocks(f"swap space: {len(blocks)} blocks needed")
        cpu = {b: self.cpu_free.pop(0) for b in blocks}
        for b in blocks:
            self.cpu_ref[cpu[b]] = self.ref[b]
            self.ref[b] = 0
            self.free.append(b)
        for sid in seq_ids:
            self.tables[sid] = [cpu[b] for b in self.tables[sid]]
            self.swapped.add(sid)
        return [(b, cpu[b]) for b in blocks]

    def swap_in(self, seq_ids) -> List[Tuple[int, int]]:
        """Bring a swapped-out group back into fresh GPU blocks (all or
        nothing); returns the (gpu_block, cpu_block) pairs to copy host ->
        device, after which the CPU blocks are free."""
        blocks = self._group_blocks(seq_ids, on_cpu=True)
        if len(blocks) > len(self.free):
            raise OutOfBlocks(f"swap-in: {len(blocks)} blocks needed")
        gpu = {c: self._take() for c in blocks}
        for c in blocks:
            self.ref[gpu[c]] = self.cpu_ref[c]
            self.cpu_ref[c] = 0
            self.cpu_free.append(c)
        for sid in seq_ids:
            self.tables[sid] = [gpu[c] for c in self.tables[sid]]
            self.swapped.discard(sid)
        return [(gpu[c], c) for c in blocks]

    def append_slot(self, seq_id: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot of the next token of ``seq_id``.

        Returns ``(slot, cow)``: the absolute slot
        ``table[pos // bs] * bs + pos % bs`` for position ``pos`` = current
        length, and ``(src, dst)`` when the write lands in a shared block and
        a copy-on-write was planned (else ``None``).  The caller must run the
        copy before writing the slot.
        """
        if seq_id in self.swapped:
            raise ValueError(f"sequence {seq_id} is swapped out")
        table = self.tables[seq_id]
        pos = self.lens[seq_id]
        j = pos // self.block_size
        cow = None
        if j == len(table):                       # the last block is full
            table.append(self._take())
        elif self.ref[table[j]] > 1:              # shared: copy, remap, decrement
            old = table[j]
            new = self._take()
            table[j] = new
            self.ref[old] -= 1
            cow = (old, new)
            self.copies_made += 1
        self.lens[seq_id] = pos + 1
        return table[j] * self.block_size + pos % self.block_size, cow

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (reference count + 1)."""
        if child in self.tables:
            raise ValueError(f"sequence {child} already exists")
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for blk in self.tables[child]:
            self.ref[blk] += 1

    def free_seq(self, seq_id: int) -> None:
        """Drop a sequence; blocks whose count reaches zero return to the pool."""
        if seq_id in self.swapped:
            self.swapped.discard(seq_id)
            for c in self.tables.pop(seq_id):
                self.cpu_ref[c] -= 1
                if self.cpu_ref[c] == 0:
                    self.cpu_free.append(c)
        else:
            for blk in self.tables.pop(seq_id):
                self._release(blk)
        del self.lens[seq_id]

    # -- views -----------------------------------------------------------
    def slot_of(self, seq_id: int, pos: int) -> int:
        if not 0 <= pos < self.lens[seq_id]:
            raise IndexError("position outside the sequence")
        return self.tables[seq_id][pos // self.block_size] * self.block_size + pos % self.block_size

    def table(self, seq_id: int) -> List[int]:
        return list(self.tables[seq_id])

    def shared_prefix_blocks(self, seq_ids) -> int:
        """Leading table entries that every sequence of ``seq_ids`` holds in
        common (the same physical block ids), counting only blocks whose
        reference count covers them all."""
        tables = [self.tables[s] for s in seq_ids]
        n = 0
        while all(len(t) > n for t in tables) and len({t[n] for t in tables}) == 1 \
                and self.ref[tables[0][n]] >= len(tables):
            n += 1
        return n

    def check_invariant(self) -> None:
        """Tables holding each block == its reference count; free <=> count 0
        (GPU blocks and, for swapped-out sequences, CPU blocks)."""
        cpu_holders = Counter(c for sid, t in self.tables.items() if sid in self.swapped for c in t)
        for c in range(self.num_cpu_blocks):
            if cpu_holders.get(c, 0) != self.cpu_ref[c]:
                raise AssertionError(f"cpu block {c}: held by {cpu_holders.get(c, 0)}, count {self.cpu_ref[c]}")
            if (c in set(self.cpu_free)) != (self.cpu_ref[c] == 0):
                raise AssertionError(f"cpu block {c}: free-list membership disagrees with count")
        holders = Counter(blk for sid, t in self.tables.items() if sid not in self.swapped for blk in t)
        for blk in range(self.num_blocks):
            if holders.get(blk, 0) != self.ref[blk]:
                raise AssertionError(
                    f"block {blk}: held by {holders.get(blk, 0)} tables, count {self.ref[blk]}")
        free = set(self.free)
        if len(free) != len(self.free):
            raise AssertionError("a block is on the free list twice")
        for blk in range(self.num_blocks):
            if (blk in free) != (self.ref[blk] == 0):
                raise AssertionError(f"block {blk}: free-list membership disagrees with count")
        for sid, t in self.tables.items():
            if len(t) != self.blocks_for(self.lens[sid]):
                raise AssertionError(f"sequence {sid}: table length disagrees with its length")
