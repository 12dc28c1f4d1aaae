"""Host-side block manager: free list, per-sequence block tables, slot mapping.

"How does TensorRT-LLM work?", "The paged KV cache": memory is a pool of
equal blocks handed out one at a time when a request needs more room; a small
table remembers which blocks belong to which request, in order; the moment a
request finishes, all its blocks go back to the free pool.
"TensorRT-LLM, in depth", "In-flight batching and the scheduler": a running
request that cannot get a block for its next token is paused.

The slot of position p of a sequence is table[p // block_size] * block_size +
p % block_size.
"""
from __future__ import annotations

from collections import deque
from typing import Dict, Iterable, List, Optional, Sequence

import numpy as np
import torch


class OutOfBlocks(RuntimeError):
    """The free list cannot cover a request; the caller pauses it."""


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int,
                 free_order: Optional[Iterable[int]] = None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.max_blocks_per_seq = int(max_blocks_per_seq)
        order = range(self.num_blocks) if free_order is None else [int(x) for x in free_order]
        self.free: deque = deque(order)
        if sorted(self.free) != list(range(self.num_blocks)):
            raise ValueError("free_order must be a permutation of the pool's block ids")
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}

    # ------------------------------------------------------------ lifecycle
    def add(self, seq_id: int) -> None:
        if seq_id in self.tables:
            raise KeyError("sequence %d already present" % seq_id)
        self.tables[seq_id] = []
        self.lens[seq_id] = 0

    def free_sequence(self, seq_id: int) -> None:
        """Return every block of the sequence to the free list."""
        for blk in self.tables.pop(seq_id):
            self.free.append(blk)
        del self.lens[seq_id]

    @property
    def num_free(self) -> int:
        return len(self.free)

    def can_grow(self, seq_id: int, n_tokens: int) -> bool:
        need = self._blocks_for(self.lens[seq_id] + n_tokens) - len(self.tables[seq_id])
        return need <= len(self.free) and self._blocks_for(self.lens[seq_id] + n_tokens) <= self.max_blocks_per_seq

    def _blocks_for(self, n_tokens: int) -> int:
        return (n_tokens + self.block_size - 1) // self.block_size

    # ---------------------------------------------------------- slot mapping
    def grow(self, seq_id: int, n_tokens: int) -> np.ndarray:
        """Reserve the next n_tokens positions of the sequence and return their
        slots (int64).  Raises OutOfBlocks, leaving the sequence unchanged, if
        the free list or the table width cannot cover them."""
        L = self.lens[seq_id]
        table = self.tables[seq_id]
        need = self._blocks_for(L + n_tokens) - len(table)
        if self._blocks_for(L + n_tokens) > self.max_blocks_per_seq or need > len(self.free):
            raise OutOfBlocks("sequence %d needs %d more blocks, %d free" % (seq_id, need, len(self.free)))
        for _ in range(max(0, need)):
            table.append(self.free.popleft())
        pos = np.arange(L, L + n_tokens, dtype=np.int64)
        tab = np.asarray(table, dtype=np.int64)
        slots = tab[pos // self.block_size] * self.block_size + pos % self.block_size
        self.lens[seq_id] = L + n_tokens
        return slots

    def decode_slots(self, seq_ids: Sequence[int]) -> np.ndarray:
        """One new token for each listed sequence: its slot (int64 [B])."""
        return np.concatenate([self.grow(s, 1) for s in seq_ids]) if len(seq_ids) else np.zeros(0, np.int64)

    # ------------------------------------------------------------- tensors
    def block_tables(self, seq_ids: Sequence[int], width: Optional[int] = None) -> torch.Tensor:
        width = self.max_blocks_per_seq if width is None else width
        t = torch.full((len(seq_ids), width), -1, dtype=torch.int32)
        for i, s in enumerate(seq_ids):
            tab = self.tables[s]
            t[i, :len(tab)] = torch.tensor(tab, dtype=torch.int32)
        return t

    def seq_lens(self, seq_ids: Sequence[int]) -> torch.Tensor:
        return torch.tensor([self.lens[s] for s in seq_ids], dtype=torch.int32)

    def check(self) -> None:
        """Invariants: every block is held by exactly one sequence or free, and
        each sequence holds exactly the blocks its length needs."""
        held = [b for tab in self.tables.values() for b in tab]
        allb = held + list(self.free)
        if sorted(allb) != list(range(self.num_blocks)):
            raise AssertionError("block ids lost or duplicated")
        for s, tab in self.tables.items():
            if len(tab) != self._blocks_for(self.lens[s]):
                raise AssertionError("sequence %d holds %d blocks for %d tokens" % (s, len(tab), self.lens[s]))
