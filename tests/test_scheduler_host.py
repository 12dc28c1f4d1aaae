"""Host tests of the in-flight scheduler (no GPU): the pages' iteration
limits, pausing when blocks run out, prefix reuse, retirement and free-list
conservation."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_194_gb300.block_manager import BlockManager
from paged_kv_cache_194_gb300.scheduler import InFlightScheduler, Request


def _requests(rng, n, system, vocab=50):
    reqs = []
    for i in range(n):
        user = [int(x) for x in rng.integers(0, vocab, int(rng.integers(1, 40)))]
        prompt = (system if rng.random() < 0.6 else []) + user
        reqs.append(Request(i, prompt, int(rng.integers(1, 30))))
    return reqs


@pytest.mark.parametrize("num_blocks", [24, 200])
def test_scheduler_runs_every_request_to_completion(num_blocks):
    rng = np.random.default_rng(num_blocks)
    bs, width = 8, 16
    bm = BlockManager(num_blocks, bs, width)
    sch = InFlightScheduler(bm, max_batch_size=6, max_num_tokens=48)
    system = list(range(1000, 1024))  # a 24-token shared system prompt: 3 full blocks
    reqs = _requests(rng, 25, system)
    for r in reqs:
        sch.submit(r)
    iters, paused, reused = 0, 0, 0
    while not sch.idle():
        it = sch.plan()
        iters += 1
        assert len(it.decode) + len(it.prefill) <= 6
        assert it.num_tokens <= 48
        # planned slots of this pass are distinct and agree with the tables
        slots = [s for _, _, s in it.decode] + [int(x) for _, _, ss in it.prefill for x in ss]
        assert len(slots) == len(set(slots))
        for r, pos, slot in it.decode:
            t = bm.block_tables([r.rid], width).numpy()
            assert oracle.slot_mapping(t, bs, [0], [pos])[0] == slot
        paused += len(it.paused)
        sch.retire(it)
        bm.check()
        assert iters < 5000
    reused = sum(r.reused for r in reqs)
    assert all(r.generated == r.max_new_tokens and r.prefilled == len(r.prompt) for r in reqs)
    assert bm.num_free == num_blocks  # every block is back (freed or cached-and-free)
    if num_blocks == 24:
        assert paused > 0  # the small pool makes requests wait for blocks
    assert reused > 0  # the shared system prompt was matched
