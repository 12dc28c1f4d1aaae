"""GPU: the failure path of the bounded pipeline waits, made to happen on
demand (no fault, no hang).

Every wait of the tensor-core decode design is bounded; an expired one sets
PKV_ERRBIT_TIMEOUT in the pool's error word, stops the CTA's pipeline, waits
for the copies the CTA has in flight, skips its output and returns.  The test
hook shortens the first stage wait of the consumer warps (of one CTA, or of
all of them) to zero polls.  The call must return promptly with the bit set,
every output row it did write must still be right, and after the caller
clears the error word and the workspace counters the next call must be exact
("TensorRT-LLM, in depth", "In-flight batching and the scheduler": a request
that cannot go on is paused, not failed).
"""
import math
import time

import numpy as np
import pytest
import torch

from paged_kv_cache_194_gb300 import binding as pk
from paged_kv_cache_194_gb300 import workloads as wl
from paged_kv_cache_194_gb300.decode import DecodeBatch

from parity import TOL, compare, oracle_reference

pytestmark = pytest.mark.gpu

LENS = (5000, 1, 0, 64, 700, 4096, 129, 2000, 3000, 17, 900, 1500)


def _setup(kv):
    w = wl.Workload("timeout_" + kv, 51, len(LENS), 16, 4, 128, 16, kv, "bf16", 1.0 / math.sqrt(128.0),
                    lens="fixed", fixed_lens=LENS)
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    slots = batch.next_token_slots()
    q, kn, vn = batch.step_inputs(0)
    pk.kv_append(batch.pool, 0, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    tables, lens = batch.tables(), batch.seq_lens()
    ref, _ = oracle_reference(w, inst.k_scale, inst.v_scale, 0, q, tables, lens.tolist(), list(range(w.num_seqs)))
    return w, batch, q.cuda(), tables.cuda(), lens.cuda(), int(lens.max()), ref


def _call(w, batch, q, tables, lens, max_len, split, ws, polls=None, cta=-1):
    out = torch.full_like(q, float("nan"))
    try:
        if polls is not None:
            pk.set_first_wait_limit_for_testing(polls, cta)
        t0 = time.perf_counter()
        pk.paged_decode_attention(q, batch.pool, 0, tables, lens, max_len, w.scale, out=out, workspace=ws,
                                  split_tokens=split, algo="mma")
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    finally:
        pk.set_first_wait_limit_for_testing(-1)
    return out, dt


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_one_cta_gives_up_balanced(kv, record_property):
    w, batch, q, tables, lens, max_len, ref = _setup(kv)
    ws = pk.workspace_for(batch.pool, w.num_seqs, w.num_q_heads, max_len)
    out, dt = _call(w, batch, q, tables, lens, max_len, 0, ws, polls=0, cta=0)
    record_property("seconds", dt)
    assert dt < 5.0
    assert batch.pool.errors() & pk.ERRBIT_TIMEOUT
    # CTA 0 skipped its output: the (sequence, KV head) units it took part in
    # are unwritten; every other row was written and is right
    o = out.float().cpu()
    skipped = torch.isnan(o).any(dim=2)  # [B, Hq]
    assert skipped.any() and not skipped.all()
    keep = ~skipped.numpy()
    compare(out.double().cpu()[torch.from_numpy(keep)], ref[keep], TOL[kv], "rows written beside the stopped CTA")
    # the units CTA 0 shared with other CTAs keep a non-zero piece counter
    counters = ws[:4 * w.num_seqs * w.num_kv_heads].view(torch.int32)
    assert int(counters.count_nonzero()) > 0
    # the caller clears the error word and the counters; the next call is exact
    batch.pool.clear_errors()
    ws.zero_()
    out2, _ = _call(w, batch, q, tables, lens, max_len, 0, ws)
    assert batch.pool.errors() == 0
    compare(out2, ref, TOL[kv], "after recovery")
    fresh = pk.paged_decode_attention(q, batch.pool, 0, tables, lens, max_len, w.scale, algo="mma")
    torch.cuda.synchronize()
    assert torch.equal(out2, fresh)
    assert int(counters.count_nonzero()) == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_every_cta_gives_up(kv):
    w, batch, q, tables, lens, max_len, ref = _setup(kv)
    ws = pk.workspace_for(batch.pool, w.num_seqs, w.num_q_heads, max_len)
    out, dt = _call(w, batch, q, tables, lens, max_len, 0, ws, polls=0, cta=-1)
    assert dt < 5.0
    assert batch.pool.errors() & pk.ERRBIT_TIMEOUT
    # nothing was written except the zero rows of the empty sequence, which
    # every launch writes before its pipeline starts
    empty = torch.tensor([L == 0 for L in LENS])
    assert torch.all(out[empty] == 0)
    assert torch.isnan(out[~empty].float()).all()
    assert int(ws[:4 * w.num_seqs * w.num_kv_heads].count_nonzero()) == 0  # no piece was published
    batch.pool.clear_errors()
    out2, _ = _call(w, batch, q, tables, lens, max_len, 0, ws)
    assert batch.pool.errors() == 0
    compare(out2, ref, TOL[kv], "after recovery")


def test_one_cta_gives_up_fixed_splits():
    """Fixed splits: CTA 0 is split 0 of the first KV-head unit of sequence 0;
    the other sequences' rows are right, and so is the next call."""
    w, batch, q, tables, lens, max_len, ref = _setup("bf16")
    ws = pk.workspace_for(batch.pool, w.num_seqs, w.num_q_heads, max_len, 256)
    out, dt = _call(w, batch, q, tables, lens, max_len, 256, ws, polls=0, cta=0)
    assert dt < 5.0
    assert batch.pool.errors() & pk.ERRBIT_TIMEOUT
    compare(out[1:], ref[1:], TOL["bf16"], "other sequences")
    batch.pool.clear_errors()
    out2, _ = _call(w, batch, q, tables, lens, max_len, 256, ws)
    assert batch.pool.errors() == 0
    compare(out2, ref, TOL["bf16"], "after recovery")


def test_hook_off_by_default_and_after_reset():
    w, batch, q, tables, lens, max_len, ref = _setup("bf16")
    pk.set_first_wait_limit_for_testing(-1)
    out, _ = _call(w, batch, q, tables, lens, max_len, 0, None)
    assert batch.pool.errors() == 0
    compare(out, ref, TOL["bf16"], "normal call")
