"""In-flight (continuous) batching over the paged KV cache.

"TensorRT-LLM, in depth", "In-flight batching and the scheduler": each
iteration rebuilds the batch -- running requests contribute one decode token
each (a request that cannot get a block for its next token is paused and
retried later), then waiting requests are admitted with a prefill chunk after
their cached prefix is matched, within two limits: max_batch_size requests
and max_num_tokens tokens per iteration.  "How does TensorRT-LLM work?", "In-
flight batching": a finished request leaves at once and its blocks return to
the free pool.

This module only plans iterations (which tokens go to which slots); the
caller writes the planned tokens' K/V with ``kv_append`` and runs
``paged_decode_attention`` for the decoding requests.  It is the host side of
the decode hot path: no model, no sampling.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field
from typing import Deque, Dict, List, Optional, Sequence, Tuple

import numpy as np

from .block_manager import BlockManager, OutOfBlocks


@dataclass
class Request:
    rid: int
    prompt: List[int]            # prompt token ids
    max_new_tokens: int
    prefilled: int = 0           # prompt tokens already in the cache (written or reused)
    reused: int = 0              # of which shared from cached blocks
    generated: int = 0           # decode tokens appended so far
    admitted: bool = False

    @property
    def length(self) -> int:
        return self.prefilled + self.generated

    @property
    def done(self) -> bool:
        return self.generated >= self.max_new_tokens


@dataclass
class Iteration:
    """One planned forward pass."""
    decode: List[Tuple[Request, int, int]] = field(default_factory=list)   # (request, position, slot)
    prefill: List[Tuple[Request, int, np.ndarray]] = field(default_factory=list)  # (request, first position, slots)
    paused: List[Request] = field(default_factory=list)
    retired: List[Request] = field(default_factory=list)

    @property
    def num_tokens(self) -> int:
        return len(self.decode) + sum(len(s) for _, _, s in self.prefill)


class InFlightScheduler:
    def __init__(self, bm: BlockManager, max_batch_size: int, max_num_tokens: int):
        self.bm = bm
        self.max_batch_size = int(max_batch_size)
        self.max_num_tokens = int(max_num_tokens)
        self.running: List[Request] = []     # prompt fully cached: decoding
        self.waiting: Deque[Request] = deque()
        self.finished: List[Request] = []
        self.preempted = 0

    def submit(self, req: Request) -> None:
        self.waiting.append(req)

    def idle(self) -> bool:
        return not self.running and not self.waiting

    def plan(self) -> Iteration:
        """Plan one iteration (the pages' schedule() sketch)."""
        it = Iteration()
        batch, budget = 0, self.max_num_tokens
        for r in self.running:                      # decoding requests: 1 token each
            if batch == self.max_batch_size or budget == 0:
                break
            pos = r.length
            slot = int(self.bm.decode_slots([r.rid])[0])
            if slot < 0:                            # out of blocks: pause, retry later
                it.paused.append(r)
                continue
            r.generated += 1
            it.decode.append((r, pos, slot))
            batch += 1
            budget -= 1
        for r in list(self.waiting):                # new requests: prefill, maybe chunked
            if batch == self.max_batch_size or budget == 0:
                break
            if not r.admitted:
                self.bm.add(r.rid)
                r.reused = r.prefilled = self.bm.match_prefix(r.rid, r.prompt)
                r.admitted = True
            chunk = min(len(r.prompt) - r.prefilled, budget)
            try:
                slots = self.bm.grow(r.rid, chunk, token_ids=r.prompt[r.prefilled:r.prefilled + chunk])
            except OutOfBlocks:
                break
            it.prefill.append((r, r.prefilled, slots))
            r.prefilled += chunk
            batch += 1
            budget -= chunk
            if r.prefilled == len(r.prompt):        # whole prompt cached: decode from the next pass
                self.waiting.remove(r)
                self.running.append(r)
        if it.num_tokens == 0 and it.paused:
            # every running request is paused and nothing could be admitted:
            # the newest running request gives its blocks back and starts over
            # (recompute), so the others can make progress
            victim = self.running.pop()
            self.bm.free_sequence(victim.rid)
            victim.prefilled = victim.reused = victim.generated = 0
            victim.admitted = False
            self.waiting.appendleft(victim)
            self.preempted += 1
        return it

    def retire(self, it: Optional[Iteration] = None) -> List[Request]:
        """After the pass: finished requests leave and free their blocks."""
        done = [r for r in self.running if r.done]
        for r in done:
            self.running.remove(r)
            self.bm.free_sequence(r.rid)
            self.finished.append(r)
        if it is not None:
            it.retired = done
        return done

    def decode_view(self, it: Iteration, width: int):
        """Tables and lengths of this pass's decoding requests (host tensors)."""
        rids = [r.rid for r, _, _ in it.decode]
        return rids, self.bm.block_tables(rids, width), self.bm.seq_lens(rids)
