"""GPU: the fused decode step (append the newest token inside the attention
kernel) against the two-launch step (kv_append, then attention) -- output
and the whole pool bit for bit -- and against the oracle."""
import math

import pytest
import torch

from paged_kv_cache_194_gb300 import binding as pk
from paged_kv_cache_194_gb300 import workloads as wl
from paged_kv_cache_194_gb300.decode import DecodeBatch

from parity import TOL, compare, oracle_reference

pytestmark = pytest.mark.gpu

EDGE = (0, 1, 2, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 300, 1000)


def _w(name, G, Hkv, bs, kv, ind, lens, qd=""):
    return wl.Workload(name, 61, len(lens), G * Hkv, Hkv, 128, bs, kv, ind, 1.0 / math.sqrt(128), lens="fixed",
                       fixed_lens=tuple(lens), q_dtype=qd)


CASES = [
    _w("bf16_pair_g4_bs16", 4, 2, 16, "bf16", "bf16", EDGE),         # KV-head pairs
    _w("bf16_pairs_hkv4_g1_bs16", 1, 4, 16, "bf16", "bf16", (1, 16, 17, 90, 0)),
    _w("bf16_pairs_hkv8_g4_bs16", 4, 8, 16, "bf16", "bf16", EDGE),
    _w("bf16_pairs_g2_from_f32_bs16", 2, 4, 16, "bf16", "f32", (33, 1, 400), qd="bf16"),
    _w("bf16_pair_g1_bs16", 1, 2, 16, "bf16", "bf16", (1, 16, 17, 90, 0)),
    _w("bf16_g2_bs32", 2, 3, 32, "bf16", "bf16", (1, 31, 32, 33, 700, 0)),
    _w("bf16_from_f32_g8_bs16", 8, 1, 16, "bf16", "f32", (40, 100, 1), qd="bf16"),
    _w("fp8_g4_bs64", 4, 2, 64, "fp8", "bf16", EDGE),
    _w("fp8_from_f32_g4_bs16", 4, 1, 16, "fp8", "f32", (40, 100, 1, 16), qd="bf16"),
]


@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fused_equals_two_launches(w, split):
    inst = wl.instance(w)
    a, b = DecodeBatch(inst, fill_byte=0x3C), DecodeBatch(inst, fill_byte=0x3C)  # identical pools and tables
    assert torch.equal(a.pool.k, b.pool.k) and torch.equal(a.pool.v, b.pool.v)
    slots = a.next_token_slots()
    b.next_token_slots()  # same block-manager growth, slots unused: the kernel takes them from the table
    q, kn, vn = a.step_inputs(0)
    tables, lens = a.tables().cuda(), a.seq_lens().cuda()
    assert torch.equal(tables.cpu(), b.tables())
    max_len = int(lens.max())
    pk.kv_append(a.pool, 0, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    out_a = pk.paged_decode_attention(q.cuda(), a.pool, 0, tables, lens, max_len, w.scale, split_tokens=split,
                                      algo="mma")
    out_b = pk.paged_decode_append_attention(q.cuda(), kn.cuda(), vn.cuda(), b.pool, 0, tables, lens, max_len,
                                             w.scale, split_tokens=split, algo="mma")
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(a.pool.k, b.pool.k) and torch.equal(a.pool.v, b.pool.v)
    assert a.pool.errors() == 0 and b.pool.errors() == 0
    ref, _ = oracle_reference(w, inst.k_scale, inst.v_scale, 0, q, tables.cpu(), lens.cpu().tolist(),
                              list(range(w.num_seqs)))
    compare(out_b, ref, TOL[w.kv_dtype], w.name)


def test_fused_full_size_llama(record_property):
    """The benchmark's decode step (one launch: append + attention) at full
    size, every sequence compared with the oracle."""
    w = wl.WORKLOADS["llama"]
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    batch.next_token_slots()
    q, kn, vn = batch.step_inputs(0)
    tables, lens = batch.tables(), batch.seq_lens()
    out = pk.paged_decode_append_attention(q.cuda(), kn.cuda(), vn.cuda(), batch.pool, 0, tables.cuda(),
                                           lens.cuda(), int(lens.max()), w.scale)
    torch.cuda.synchronize()
    seqs = list(range(w.num_seqs))
    ref, _ = oracle_reference(w, inst.k_scale, inst.v_scale, 0, q, tables, lens.tolist(), seqs)
    max_abs, max_rel = compare(out, ref, TOL["bf16"], "llama fused")
    record_property("max_abs_err", max_abs)
    record_property("max_rel_err", max_rel)
    assert batch.pool.errors() == 0


def test_fused_full_size_ragged_steps(record_property):
    """The in-flight batch (256 sequences, 32-token blocks, 4 query heads per
    KV head) for 8 fused decode steps, the block manager growing the tables
    between them; every sequence compared with the oracle at the first and
    the last step."""
    w = wl.WORKLOADS["ragged"]
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    seqs = list(range(w.num_seqs))
    ws = None
    worst = (0.0, 0.0)
    for step in range(w.steps):
        batch.next_token_slots()
        q, kn, vn = batch.step_inputs(0, step)
        tables, lens = batch.tables(), batch.seq_lens()
        if ws is None:
            ws = pk.workspace_for(batch.pool, w.num_seqs, w.num_q_heads, int(inst.lens.max()) + w.steps)
        out = pk.paged_decode_append_attention(q.cuda(), kn.cuda(), vn.cuda(), batch.pool, 0, tables.cuda(),
                                               lens.cuda(), int(lens.max()), w.scale, workspace=ws)
        torch.cuda.synchronize()
        if step in (0, w.steps - 1):
            ref, _ = oracle_reference(w, 1.0, 1.0, 0, q, tables, lens.tolist(), seqs)
            e = compare(out, ref, TOL["bf16"], "ragged fused step %d" % step)
            worst = (max(worst[0], e[0]), max(worst[1], e[1]))
        batch.bm.check()
    record_property("max_abs_err", worst[0])
    record_property("max_rel_err", worst[1])
    assert batch.pool.errors() == 0


def test_fused_unsupported_designs():
    w = _w("f32_pool", 2, 1, 16, "f32", "f32", (5, 9))
    batch = DecodeBatch(wl.instance(w))
    batch.next_token_slots()
    q, kn, vn = batch.step_inputs(0)
    with pytest.raises(pk.PkvError):
        pk.paged_decode_append_attention(q.cuda(), kn.cuda(), vn.cuda(), batch.pool, 0, batch.tables().cuda(),
                                         batch.seq_lens().cuda(), 9, w.scale)


def test_lengths_written_by_the_kernel_before():
    """Decode calls back to back, each reading lengths that a kernel wrote
    just before it on the same stream (no host synchronisation between
    them): every call must match the oracle for the lengths it was given."""
    w = CASES[2]
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    slots = batch.next_token_slots()
    q, kn, vn = batch.step_inputs(0)
    pk.kv_append(batch.pool, 0, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    tables, lens = batch.tables().cuda(), batch.seq_lens().cuda()
    max_len = int(lens.max())
    outs, used = [], []
    for cut in (0, 1, 3, 0, 40):
        lens_dev = torch.clamp(lens - cut, min=0).to(torch.int32)  # a kernel writes them
        outs.append(pk.paged_decode_attention(q.cuda(), batch.pool, 0, tables, lens_dev, max_len, w.scale,
                                              algo="mma"))
        used.append(lens_dev)
    torch.cuda.synchronize()
    assert batch.pool.errors() == 0
    for out, L in zip(outs, used):
        ref, _ = oracle_reference(w, inst.k_scale, inst.v_scale, 0, q, tables.cpu(), L.cpu().tolist(),
                                  list(range(w.num_seqs)))
        compare(out, ref, TOL[w.kv_dtype], "lengths written by the kernel before")
