"""The allocation-free decode entry point against the workspace entry point.

paged_decode_attention_static_ws is for callers that may not allocate device
memory where they run decode attention; its split partials live in a fixed
device array inside the library.  This file sorts last so that a run stopping
at its first failure has already run every other test.
"""
import math

import pytest
import torch

from paged_kv_cache_194_gb300 import binding as pk
from paged_kv_cache_194_gb300 import workloads as wl
from paged_kv_cache_194_gb300.decode import DecodeBatch

from parity import TOL, compare

pytestmark = pytest.mark.gpu


def _batch(kv="bf16", lens=(1, 15, 16, 17, 64, 65, 300, 1000, 2047)):
    w = wl.Workload("no_alloc_" + kv, 31, len(lens), 8, 2, 128, 16, kv, "bf16", 1.0 / math.sqrt(128.0),
                    lens="fixed", fixed_lens=tuple(lens))
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    slots = batch.next_token_slots()
    q, kn, vn = batch.step_inputs(0)
    pk.kv_append(batch.pool, 0, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    return w, batch, q.cuda(), batch.tables().cuda(), batch.seq_lens().cuda(), int(batch.seq_lens().max())


@pytest.mark.parametrize("split", [64, 0], ids=["fixed_splits", "balanced"])
@pytest.mark.parametrize("algo", ["simt", "mma"])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_static_scratch_matches_workspace_entry_point(kv, algo, split):
    w, batch, q, tables, lens, max_len = _batch(kv)
    # split 64: 32 fixed splits for the longest sequence; split 0: the
    # tensor-core design's balanced schedule shares sequences between CTAs
    _, ns, need = pk.decode_plan(batch.pool, w.num_seqs, w.num_q_heads, max_len, split)
    assert 0 < need <= pk.STATIC_SCRATCH_BYTES
    ref = pk.paged_decode_attention(q, batch.pool, 0, tables, lens, max_len, w.scale, split_tokens=split, algo=algo)
    for _ in range(2):  # two calls in a row share the library's array
        out = torch.full_like(q, float("nan"))
        pk.paged_decode_attention_static_ws(q, batch.pool, 0, tables, lens, max_len, w.scale, out=out,
                                            split_tokens=split, algo=algo)
        torch.cuda.synchronize()
        compare(out, ref.double().cpu().numpy(), TOL[kv], "static scratch vs workspace (%s, %s)" % (kv, algo))
    assert batch.pool.errors() == 0


def test_static_scratch_rejects_oversized_plans():
    w, batch, q, tables, lens, max_len = _batch("bf16", lens=(2047,) * 4)
    # 4 sequences x 8 heads x 32 splits fits; 2048 sequences x 8 heads x 32 splits does not
    _, _, need = pk.decode_plan(batch.pool, 2048, w.num_q_heads, max_len, 64)
    assert need > pk.STATIC_SCRATCH_BYTES
    big_q = torch.zeros(2048, w.num_q_heads, 128, dtype=torch.bfloat16, device="cuda")
    big_t = tables[:1].expand(2048, -1).contiguous()
    big_l = lens[:1].expand(2048).contiguous()
    with pytest.raises(pk.PkvError) as e:
        pk.paged_decode_attention_static_ws(big_q, batch.pool, 0, big_t, big_l, max_len, w.scale, split_tokens=64)
    assert e.value.status == 3
