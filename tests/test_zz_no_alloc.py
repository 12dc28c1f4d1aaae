"""The allocation-free decode entry point against the workspace entry point.

paged_decode_attention_static_ws serves callers that may not allocate device
memory where they run decode attention (plug-ins whose memory the host
application plans up front, allocator-free loops, fixed memory budgets); its
split partials live in a fixed device array inside the library.  Both entry
points run the same kernels on the same inputs, so their outputs must be
identical bit for bit.  The array keeps what the previous call left, so the
tests chain calls of different shapes, and a call after one whose pipeline
wait expired.  This file sorts last so that a run stopping at its first
failure has already run every other test.
"""
import math

import pytest
import torch

from paged_kv_cache_194_gb300 import binding as pk
from paged_kv_cache_194_gb300 import workloads as wl
from paged_kv_cache_194_gb300.decode import DecodeBatch

pytestmark = pytest.mark.gpu

LENS_A = (1, 15, 16, 17, 64, 65, 300, 1000, 2047)
# more sequences and more KV heads than shape A: its counters reach bytes that
# held shape A's partial sums
LENS_B = (3000, 5, 0, 777, 1500, 64, 2048, 129, 4000, 31, 900, 2600, 1, 450, 1023, 3333)


def _batch(kv="bf16", lens=LENS_A, hkv=2, seed=31):
    w = wl.Workload("no_alloc_%s_%d" % (kv, hkv), seed, len(lens), 4 * hkv, hkv, 128, 16, kv, "bf16",
                    1.0 / math.sqrt(128.0), lens="fixed", fixed_lens=tuple(lens))
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    slots = batch.next_token_slots()
    q, kn, vn = batch.step_inputs(0)
    pk.kv_append(batch.pool, 0, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    return w, batch, q.cuda(), batch.tables().cuda(), batch.seq_lens().cuda(), int(batch.seq_lens().max())


def _static(w, batch, q, tables, lens, max_len, split, algo):
    out = torch.full_like(q, float("nan"))
    pk.paged_decode_attention_static_ws(q, batch.pool, 0, tables, lens, max_len, w.scale, out=out,
                                        split_tokens=split, algo=algo)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("split", [64, 0], ids=["fixed_splits", "balanced"])
@pytest.mark.parametrize("algo", ["simt", "mma", "tc"])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_static_scratch_matches_workspace_entry_point(kv, algo, split):
    if algo == "tc" and (kv != "bf16" or split):
        pytest.skip("the tcgen05 design serves BF16 pools without fixed splits")
    shapes = [_batch(kv, LENS_A, 2), _batch(kv, LENS_B, 4, seed=32), _batch(kv, LENS_A, 2)]
    for i, (w, batch, q, tables, lens, max_len) in enumerate(shapes):
        # split 64: up to 63 fixed splits per sequence; split 0: the balanced
        # schedule shares sequences between CTAs and merges them in the kernel
        _, _, need = pk.decode_plan(batch.pool, w.num_seqs, w.num_q_heads, max_len, split)
        assert 0 < need <= pk.STATIC_SCRATCH_BYTES
        ref = pk.paged_decode_attention(q, batch.pool, 0, tables, lens, max_len, w.scale, split_tokens=split,
                                        algo=algo)
        for rep in range(2):  # two calls in a row share the library's array
            out = _static(w, batch, q, tables, lens, max_len, split, algo)
            assert torch.equal(out, ref), "shape %d call %d (%s, %s, split %d)" % (i, rep, kv, algo, split)
        assert batch.pool.errors() == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_static_scratch_recovers_after_an_expired_wait(kv):
    """A call whose first CTA gives up its first pipeline wait reports
    PKV_ERRBIT_TIMEOUT and can leave per-sequence counters non-zero in the
    library's array; the next call clears its own counters and is exact."""
    w, batch, q, tables, lens, max_len = _batch(kv, LENS_B, 4, seed=33)
    ref = pk.paged_decode_attention(q, batch.pool, 0, tables, lens, max_len, w.scale, algo="mma")
    torch.cuda.synchronize()
    try:
        pk.set_first_wait_limit_for_testing(0, 0)
        _static(w, batch, q, tables, lens, max_len, 0, "mma")
    finally:
        pk.set_first_wait_limit_for_testing(-1)
    assert batch.pool.errors() & pk.ERRBIT_TIMEOUT
    batch.pool.clear_errors()
    for _ in range(2):
        out = _static(w, batch, q, tables, lens, max_len, 0, "mma")
        assert torch.equal(out, ref)
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
