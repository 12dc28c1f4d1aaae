"""Python face of the native host block manager (``kv_block_manager_*`` /
``kv_bm_*`` in include/pkv.h, implemented in csrc/block_manager.cpp).

"How does TensorRT-LLM work?", "The paged KV cache": memory is a pool of
equal blocks handed out one at a time when a request needs more room; a small
table remembers which blocks belong to which request, in order; the moment a
request finishes, its blocks go back to the free pool; requests that begin
with the same text point at the same blocks.  "TensorRT-LLM, in depth",
"In-flight batching and the scheduler": a running request that cannot get a
block for its next token is paused.

The slot of position p of a sequence is table[p // block_size] * block_size +
p % block_size.  Sequence keys may be any hashable Python value.
"""
from __future__ import annotations

import ctypes
from typing import Dict, Hashable, Iterable, List, Optional, Sequence

import numpy as np
import torch

from . import binding as pk

OUT_OF_BLOCKS = 6


class OutOfBlocks(RuntimeError):
    """The free list cannot cover a request; the caller pauses it."""


def _lib():
    L = pk.lib()
    if not getattr(L, "_bm_ready", False):
        c, P = ctypes, ctypes.c_void_p
        L.kv_block_manager_create.restype = c.c_int
        L.kv_block_manager_create.argtypes = [c.c_int32, c.c_int32, c.c_int32, P, c.POINTER(P)]
        L.kv_block_manager_destroy.restype = None
        L.kv_block_manager_destroy.argtypes = [P]
        L.kv_bm_num_free.restype = c.c_int32
        L.kv_bm_num_free.argtypes = [P]
        L.kv_bm_add_sequence.restype = c.c_int
        L.kv_bm_add_sequence.argtypes = [P, c.c_int64]
        L.kv_bm_free_sequence.restype = c.c_int
        L.kv_bm_free_sequence.argtypes = [P, c.c_int64]
        L.kv_bm_grow.restype = c.c_int
        L.kv_bm_grow.argtypes = [P, c.c_int64, c.c_int32, P, P]
        L.kv_bm_decode_slots.restype = c.c_int
        L.kv_bm_decode_slots.argtypes = [P, P, c.c_int32, P, c.POINTER(c.c_int32)]
        L.kv_bm_match_prefix.restype = c.c_int
        L.kv_bm_match_prefix.argtypes = [P, c.c_int64, P, c.c_int32, c.POINTER(c.c_int32)]
        L.kv_bm_seq_len.restype = c.c_int32
        L.kv_bm_seq_len.argtypes = [P, c.c_int64]
        L.kv_bm_block_tables.restype = c.c_int
        L.kv_bm_block_tables.argtypes = [P, P, c.c_int32, c.c_int32, P, P]
        L.kv_bm_free_list.restype = c.c_int32
        L.kv_bm_free_list.argtypes = [P, P, c.c_int32]
        L.kv_bm_block_ref.restype = c.c_int32
        L.kv_bm_block_ref.argtypes = [P, c.c_int32]
        L.kv_bm_check.restype = c.c_int
        L.kv_bm_check.argtypes = [P]
        L._bm_ready = True
    return L


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a.size else ctypes.c_void_p()


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int,
                 free_order: Optional[Iterable[int]] = None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.max_blocks_per_seq = int(max_blocks_per_seq)
        order = None
        if free_order is not None:
            order = np.ascontiguousarray(np.asarray(list(free_order), dtype=np.int32))
            if order.size != self.num_blocks:
                raise ValueError("free_order must be a permutation of the pool's block ids")
        h = ctypes.c_void_p()
        rc = _lib().kv_block_manager_create(self.num_blocks, self.block_size, self.max_blocks_per_seq,
                                            _ptr(order) if order is not None else None, ctypes.byref(h))
        if rc != 0:
            raise ValueError("kv_block_manager_create failed (%d): free_order must be a permutation" % rc)
        self._h = h
        self._ids: Dict[Hashable, int] = {}
        self._next_id = 0

    def __del__(self):
        try:
            if getattr(self, "_h", None) is not None and self._h.value:
                _lib().kv_block_manager_destroy(self._h)
                self._h = None
        except Exception:
            pass

    def _id(self, seq: Hashable) -> int:
        if seq not in self._ids:
            raise KeyError("unknown sequence %r" % (seq,))
        return self._ids[seq]

    # ------------------------------------------------------------ lifecycle
    def add(self, seq: Hashable) -> None:
        if seq in self._ids:
            raise KeyError("sequence %r already present" % (seq,))
        self._ids[seq] = self._next_id
        self._next_id += 1
        if _lib().kv_bm_add_sequence(self._h, self._ids[seq]) != 0:
            raise RuntimeError("kv_bm_add_sequence failed")

    def free_sequence(self, seq: Hashable) -> None:
        """Drop a finished sequence; its blocks lose one reference each."""
        if _lib().kv_bm_free_sequence(self._h, self._id(seq)) != 0:
            raise RuntimeError("kv_bm_free_sequence failed")
        del self._ids[seq]

    @property
    def num_free(self) -> int:
        return int(_lib().kv_bm_num_free(self._h))

    def seq_len(self, seq: Hashable) -> int:
        return int(_lib().kv_bm_seq_len(self._h, self._id(seq)))

    def _blocks_for(self, n_tokens: int) -> int:
        return (n_tokens + self.block_size - 1) // self.block_size

    def can_grow(self, seq: Hashable, n_tokens: int) -> bool:
        L = self.seq_len(seq)
        total = self._blocks_for(L + n_tokens)
        return total <= self.max_blocks_per_seq and total - self._blocks_for(L) <= self.num_free

    # ---------------------------------------------------------- slot mapping
    def grow(self, seq: Hashable, n_tokens: int, token_ids: Optional[Sequence[int]] = None) -> np.ndarray:
        """Reserve the next n_tokens positions of the sequence and return their
        slots (int64).  Raises OutOfBlocks, leaving the sequence unchanged, if
        the free list or the table width cannot cover them."""
        slots = np.empty(n_tokens, dtype=np.int64)
        ids = None if token_ids is None else np.ascontiguousarray(np.asarray(token_ids, dtype=np.int32))
        if ids is not None and ids.size != n_tokens:
            raise ValueError("token_ids must have n_tokens entries")
        rc = _lib().kv_bm_grow(self._h, self._id(seq), n_tokens, _ptr(ids) if ids is not None else None,
                               _ptr(slots))
        if rc == OUT_OF_BLOCKS:
            raise OutOfBlocks("sequence %r cannot get blocks for %d more tokens (%d free)"
                              % (seq, n_tokens, self.num_free))
        if rc != 0:
            raise RuntimeError("kv_bm_grow failed (%d)" % rc)
        return slots

    def decode_slots(self, seqs: Sequence[Hashable]) -> np.ndarray:
        """One new token per listed sequence: its slot, or -1 for a sequence
        that has to pause (no free block for it this step)."""
        ids = np.ascontiguousarray(np.array([self._id(s) for s in seqs], dtype=np.int64))
        slots = np.empty(len(seqs), dtype=np.int64)
        paused = ctypes.c_int32(0)
        rc = _lib().kv_bm_decode_slots(self._h, _ptr(ids), len(seqs), _ptr(slots), ctypes.byref(paused))
        if rc != 0:
            raise RuntimeError("kv_bm_decode_slots failed (%d)" % rc)
        self.last_paused = paused.value
        return slots

    def match_prefix(self, seq: Hashable, token_ids: Sequence[int]) -> int:
        """For an empty sequence about to hold these prompt ids: share the
        cached full blocks of the longest matching prefix; returns the number
        of reused tokens (the sequence's new length)."""
        ids = np.ascontiguousarray(np.asarray(token_ids, dtype=np.int32))
        reused = ctypes.c_int32(0)
        rc = _lib().kv_bm_match_prefix(self._h, self._id(seq), _ptr(ids), ids.size, ctypes.byref(reused))
        if rc != 0:
            raise RuntimeError("kv_bm_match_prefix failed (%d)" % rc)
        return reused.value

    # ------------------------------------------------------------- tensors
    def block_tables(self, seqs: Sequence[Hashable], width: Optional[int] = None) -> torch.Tensor:
        width = self.max_blocks_per_seq if width is None else width
        ids = np.ascontiguousarray(np.array([self._id(s) for s in seqs], dtype=np.int64))
        t = np.empty((len(seqs), width), dtype=np.int32)
        rc = _lib().kv_bm_block_tables(self._h, _ptr(ids), len(seqs), width, _ptr(t), None)
        if rc != 0:
            raise RuntimeError("kv_bm_block_tables failed (%d)" % rc)
        return torch.from_numpy(t)

    def seq_lens(self, seqs: Sequence[Hashable]) -> torch.Tensor:
        return torch.tensor([self.seq_len(s) for s in seqs], dtype=torch.int32)

    @property
    def tables(self) -> Dict[Hashable, List[int]]:
        out = {}
        for s in self._ids:
            n = self._blocks_for(self.seq_len(s))
            out[s] = self.block_tables([s], max(1, self.max_blocks_per_seq))[0, :n].tolist()
        return out

    @property
    def lens(self) -> Dict[Hashable, int]:
        return {s: self.seq_len(s) for s in self._ids}

    @property
    def free(self) -> List[int]:
        n = int(_lib().kv_bm_free_list(self._h, None, 0))
        buf = np.empty(max(1, n), dtype=np.int32)
        _lib().kv_bm_free_list(self._h, _ptr(buf), n)
        return buf[:n].tolist()

    def ref(self, block: int) -> int:
        return int(_lib().kv_bm_block_ref(self._h, block))

    def check(self) -> None:
        """Invariants: a block's reference count equals the number of tables
        holding it; free blocks are exactly the unreferenced ones; each
        sequence holds exactly the blocks its length needs."""
        if _lib().kv_bm_check(self._h) != 0:
            raise AssertionError("block manager invariant violated")
