"""Reference model of the paged cache's block manager (plain Python lists).

TEST INFRASTRUCTURE ONLY: the tests compare the C-ABI block manager against
this model call by call; nothing on the product path imports it.

Semantics, after the pages ("跟着 Claude Code，我用 Python 实现了一个轻量级的
vLLM", section "核心机制一：分页 KV Cache": fixed 16-token blocks taken on
demand, all returned when a sequence ends; "从零实现一个 mini vLLM--开篇",
section 5, phase 4: a block table per request; "v0版本介绍", section
"为什么需要推理框架": a block is taken only when the current one is full, and
requests may share a prompt's blocks), with the readings the library
documents: reference counts for sharing, copy-on-write of a shared partly
filled last block, a first-in first-out free list that takes from the front
and returns a sequence's blocks to the back in table order, and calls that
change nothing when they fail.
"""
from __future__ import annotations

BLOCK = 16


class NoFreeBlocks(Exception):
    pass


class ModelBlockManager:
    def __init__(self, num_blocks: int, initial_free_order=None):
        order = list(range(num_blocks)) if initial_free_order is None else [int(x) for x in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("initial order must be a permutation")
        self.num_blocks = num_blocks
        self.free = order
        self.refs = [0] * num_blocks
        self.blocks: dict[int, list[int]] = {}
        self.length: dict[int, int] = {}

    def _take(self) -> int:
        b = self.free.pop(0)
        self.refs[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.refs[b] -= 1
        if self.refs[b] == 0:
            self.free.append(b)

    def num_free(self) -> int:
        return len(self.free)

    def add_sequence(self, seq_id: int, num_tokens: int) -> list[int]:
        if seq_id < 0 or seq_id in self.blocks or num_tokens < 0:
            raise ValueError("bad sequence")
        need = -(-num_tokens // BLOCK)
        if need > len(self.free):
            raise NoFreeBlocks
        self.blocks[seq_id] = [self._take() for _ in range(need)]
        self.length[seq_id] = num_tokens
        return [self.blocks[seq_id][p // BLOCK] * BLOCK + p % BLOCK for p in range(num_tokens)]

    def append_slots(self, seq_ids) -> tuple[list[int], list[tuple[int, int]]]:
        seq_ids = [int(s) for s in seq_ids]
        if len(set(seq_ids)) != len(seq_ids) or any(s not in self.blocks for s in seq_ids):
            raise ValueError("bad sequence list")
        # Dry run on copies of the state to see whether the pool suffices.
        refs = list(self.refs)
        need = 0
        for s in seq_ids:
            if self.length[s] % BLOCK == 0:
                need += 1
            elif refs[self.blocks[s][-1]] > 1:
                need += 1
                refs[self.blocks[s][-1]] -= 1
        if need > len(self.free):
            raise NoFreeBlocks
        slots, copies = [], []
        for s in seq_ids:
            pos = self.length[s]
            if pos % BLOCK == 0:
                self.blocks[s].append(self._take())
            elif self.refs[self.blocks[s][-1]] > 1:
                old = self.blocks[s][-1]
                new = self._take()
                copies.append((old, new))
                self._release(old)
                self.blocks[s][-1] = new
            slots.append(self.blocks[s][-1] * BLOCK + pos % BLOCK)
            self.length[s] = pos + 1
        return slots, copies

    def fork(self, parent: int, child: int) -> None:
        if parent not in self.blocks or child in self.blocks or child < 0:
            raise ValueError("bad fork")
        self.blocks[child] = list(self.blocks[parent])
        self.length[child] = self.length[parent]
        for b in self.blocks[child]:
            self.refs[b] += 1

    def free_sequence(self, seq_id: int) -> None:
        if seq_id not in self.blocks:
            raise ValueError("unknown sequence")
        for b in self.blocks.pop(seq_id):
            self._release(b)
        del self.length[seq_id]

    def block_tables(self, seq_ids, width: int):
        rows, lens = [], []
        for s in seq_ids:
            bl = self.blocks[int(s)]
            if len(bl) > width:
                raise ValueError("table too narrow")
            rows.append(bl + [-1] * (width - len(bl)))
            lens.append(self.length[int(s)])
        return rows, lens
