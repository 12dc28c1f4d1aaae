"""GPU test of the in-flight loop: the scheduler plans each pass, the prompt
chunks' and decode tokens' K/V go through kv_append, and paged decode
attention runs through the C ABI for the decoding requests; every pass is
compared with the fp64 oracle.  Requests share a system prompt (prefix
reuse: several block tables point at the same blocks) and the pool is small
enough that requests pause for blocks."""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_194_gb300 import binding as pk
from paged_kv_cache_194_gb300 import workloads as wl
from paged_kv_cache_194_gb300.block_manager import BlockManager
from paged_kv_cache_194_gb300.scheduler import InFlightScheduler, Request

from parity import TOL, compare, oracle_reference

pytestmark = pytest.mark.gpu

D, HKV, G, BS, WIDTH = 128, 2, 4, 16, 16


_TAGS = {"sys": 1, "own": 2, "q": 3}


def _gen(tag, *key):
    s = _TAGS[tag]
    for k in key:
        s = (s * 1000003 + int(k) + 1) % (2**61 - 1)
    g = torch.Generator()
    g.manual_seed(s)
    return g


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_in_flight_loop_with_prefix_reuse(kv):
    rng = np.random.default_rng(7)
    w = wl.Workload("inflight_" + kv, 9, 1, G * HKV, HKV, D, BS, kv, "bf16", 1.0 / math.sqrt(D))
    system = [int(x) for x in rng.integers(0, 2**30, 40)]  # 2 full blocks + 8 tokens
    sys_k = torch.randn(len(system), HKV, D, generator=_gen("sys", 0)).to(torch.bfloat16)
    sys_v = torch.randn(len(system), HKV, D, generator=_gen("sys", 1)).to(torch.bfloat16)
    reqs, own = [], {}
    for i in range(18):
        user = [int(x) for x in rng.integers(0, 2**30, int(rng.integers(1, 50)))]
        prompt = (system if i % 3 else []) + user
        r = Request(i, prompt, int(rng.integers(2, 12)))
        n = len(prompt) + r.max_new_tokens
        own[i] = (torch.randn(n, HKV, D, generator=_gen("own", i, 0)).to(torch.bfloat16),
                  torch.randn(n, HKV, D, generator=_gen("own", i, 1)).to(torch.bfloat16))
        reqs.append(r)

    def rows(r, L):  # K/V of positions 0..L-1: the system prompt's rows are shared
        k, v = own[r.rid][0][:L].clone(), own[r.rid][1][:L].clone()
        if r.prompt[:len(system)] == system:
            m = min(L, len(system))
            k[:m], v[:m] = sys_k[:m], sys_v[:m]
        return k, v

    k_scale = v_scale = 1.0
    if kv == "fp8":  # per-tensor scales over everything the test may store
        allk = torch.cat([sys_k] + [own[i][0] for i in own]).float().abs().max()
        allv = torch.cat([sys_v] + [own[i][1] for i in own]).float().abs().max()
        k_scale, v_scale = float(allk / 448.0), float(allv / 448.0)
    NB = 16  # small enough that running requests pause for blocks
    pool = pk.KVPool(1, NB, BS, HKV, D, kv, k_scale, v_scale)
    bm = BlockManager(NB, BS, WIDTH)
    sch = InFlightScheduler(bm, max_batch_size=8, max_num_tokens=80)
    for r in reqs:
        sch.submit(r)
    checked = paused = 0
    for _ in range(400):
        if sch.idle():
            break
        it = sch.plan()
        paused += len(it.paused)
        ks, vs, ss = [], [], []
        for r, p0, slots in it.prefill:
            k, v = rows(r, p0 + len(slots))
            ks.append(k[p0:])
            vs.append(v[p0:])
            ss.append(torch.from_numpy(slots))
        for r, pos, slot in it.decode:
            k, v = rows(r, pos + 1)
            ks.append(k[pos:])
            vs.append(v[pos:])
            ss.append(torch.tensor([slot], dtype=torch.int64))
        if ss:
            pk.kv_append(pool, 0, torch.cat(ks).cuda(), torch.cat(vs).cuda(), torch.cat(ss).cuda())
        if it.decode:
            rids, tables, lens = sch.decode_view(it, WIDTH)
            q = torch.stack([torch.randn(G * HKV, D, generator=_gen("q", r.rid, r.generated))
                             for r, _, _ in it.decode]).to(torch.bfloat16)
            out = pk.paged_decode_attention(q.cuda(), pool, 0, tables.cuda(), lens.cuda(), int(lens.max()), w.scale)
            torch.cuda.synchronize()
            batch_reqs = [r for r, _, _ in it.decode]
            ref, _ = oracle_reference(w, k_scale, v_scale, 0, q, tables, lens.tolist(), list(range(len(rids))),
                                      rows_fn=lambda b, L: rows(batch_reqs[b], L))
            compare(out, ref, TOL[kv], "in-flight pass")
            checked += len(rids)
        sch.retire(it)
        bm.check()
    assert sch.idle() and len(sch.finished) == len(reqs)
    assert all(r.generated == r.max_new_tokens for r in reqs)
    assert paused > 0 and sum(r.reused for r in reqs) > 0 and checked > 50
    assert pool.errors() == 0 and bm.num_free == NB
