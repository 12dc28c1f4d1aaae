"""In-flight (continuous) batching over the paged KV cache: the host side of
the decode hot path.

Policy, from "TensorRT-LLM, in depth", section "In-flight batching and the
scheduler", and "How does TensorRT-LLM work?", section "In-flight batching":
the batch is rebuilt before every forward pass under two caps, a number of
requests and a number of tokens; requests already generating take priority
over new ones; a request whose next token needs a block the pool cannot give
waits for a later pass instead of failing; a new request first reuses the
cached blocks of its longest matching prefix and may have its prompt cut
into chunks across passes; a request that has finished leaves at once and
its blocks go back to the pool.

Design.  A pass walks one queue of candidates in priority order -- the
generating requests in the order they started, then the admitted-but-not-
yet-generating and the new requests in arrival order -- and grants each what
it asks for from one shared ``Budget`` (seats and tokens): one token for a
generating request, as much of the remaining prompt as the budget allows for
a prompt.  A grant that the pool cannot back with blocks either pauses the
request (generating ones) or ends admission for the pass (prompts: later
arrivals must not overtake an earlier one).  Where the pages leave a gap:
if a pass would do nothing at all because every generating request is
paused, the most recently started one releases its blocks and goes back to
the front of the queue to be recomputed, so the loop always progresses.

This module only plans (which token goes to which slot); the caller writes
the planned tokens' K/V with ``kv_append`` and runs
``paged_decode_attention`` for the generating requests.  No model, no
sampling.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field
from typing import Deque, Iterator, List, Optional, Tuple

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
    admitted: bool = False       # holds a sequence in the block manager

    @property
    def length(self) -> int:
        return self.prefilled + self.generated

    @property
    def done(self) -> bool:
        return self.generated >= self.max_new_tokens

    @property
    def prompt_left(self) -> int:
        return len(self.prompt) - self.prefilled


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


@dataclass
class Budget:
    """What one pass may still hand out."""
    seats: int
    tokens: int

    def exhausted(self) -> bool:
        return self.seats <= 0 or self.tokens <= 0

    def take(self, tokens: int) -> None:
        self.seats -= 1
        self.tokens -= tokens


class InFlightScheduler:
    def __init__(self, bm: BlockManager, max_batch_size: int, max_num_tokens: int):
        self.bm = bm
        self.max_batch_size = int(max_batch_size)
        self.max_num_tokens = int(max_num_tokens)
        self.running: List[Request] = []     # whole prompt cached: one token per pass
        self.waiting: Deque[Request] = deque()  # prompt not (fully) cached yet, arrival order
        self.finished: List[Request] = []
        self.preempted = 0

    def submit(self, req: Request) -> None:
        self.waiting.append(req)

    def idle(self) -> bool:
        return not self.running and not self.waiting

    # ------------------------------------------------------------ planning
    def _queue(self) -> Iterator[Tuple[Request, bool]]:
        """Candidates in priority order, each with whether it is generating."""
        for r in list(self.running):
            yield r, True
        for r in list(self.waiting):
            yield r, False

    def _grant_token(self, r: Request, it: Iteration, budget: Budget) -> None:
        """A generating request asks for the slot of its next token."""
        slot = int(self.bm.decode_slots([r.rid])[0])
        if slot < 0:  # no block for it this pass: it waits, costing nothing
            it.paused.append(r)
            return
        it.decode.append((r, r.length, slot))
        r.generated += 1
        budget.take(1)

    def _grant_prompt(self, r: Request, it: Iteration, budget: Budget) -> bool:
        """A prompt asks for its next chunk; False when the pool cannot back
        it (admission stops for this pass)."""
        if not r.admitted:
            self.bm.add(r.rid)
            r.prefilled = r.reused = self.bm.match_prefix(r.rid, r.prompt)
            r.admitted = True
        n = min(r.prompt_left, budget.tokens)
        first = r.prefilled
        try:
            slots = self.bm.grow(r.rid, n, token_ids=r.prompt[first:first + n])
        except OutOfBlocks:
            return False
        it.prefill.append((r, first, slots))
        r.prefilled += n
        budget.take(n)
        return True

    def plan(self) -> Iteration:
        """Plan one forward pass."""
        it = Iteration()
        budget = Budget(self.max_batch_size, self.max_num_tokens)
        admitting = True
        for r, generating in self._queue():
            if budget.exhausted():
                break
            if generating:
                self._grant_token(r, it, budget)
            elif admitting:
                admitting = self._grant_prompt(r, it, budget)
        # prompts cached in full this pass generate from the next one on
        for r, _, _ in it.prefill:
            if r.prompt_left == 0:
                self.waiting.remove(r)
                self.running.append(r)
        if it.num_tokens == 0 and it.paused:
            self._recompute_newest()
        return it

    def _recompute_newest(self) -> None:
        """Every generating request is stuck and nothing was admitted: the one
        that started last gives its blocks back and re-enters the queue first,
        to be prefilled again."""
        victim = self.running.pop()
        self.bm.free_sequence(victim.rid)
        victim.prefilled = victim.reused = victim.generated = 0
        victim.admitted = False
        self.waiting.appendleft(victim)
        self.preempted += 1

    # ------------------------------------------------------------ after a pass
    def retire(self, it: Optional[Iteration] = None) -> List[Request]:
        """Finished requests leave and free their blocks."""
        done = [r for r in self.running if r.done]
        for r in done:
            self.running.remove(r)
            self.bm.free_sequence(r.rid)
            self.finished.append(r)
        if it is not None:
            it.retired = done
        return done

    def decode_view(self, it: Iteration, width: int):
        """Tables and lengths of this pass's generating requests (host tensors)."""
        rids = [r.rid for r, _, _ in it.decode]
        return rids, self.bm.block_tables(rids, width), self.bm.seq_lens(rids)
