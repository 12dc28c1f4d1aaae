"""GPU parity of multi-query paged attention (speculative verification /
prompt chunks): the last C tokens of each sequence query causally."""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_194_gb300 import binding as pk
from paged_kv_cache_194_gb300 import workloads as wl
from paged_kv_cache_194_gb300.decode import DecodeBatch

from parity import TOL, compare, oracle_reference_mq

pytestmark = pytest.mark.gpu


def _w(name, G, Hkv, kv, ind, lens, bs=16, D=128):
    return wl.Workload(name, 41, len(lens), G * Hkv, Hkv, D, bs, kv, ind, 1.0 / math.sqrt(D),
                       lens="fixed", fixed_lens=tuple(lens), dist="uniform" if kv == "f32" else "normal")


def _filled(w):
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    slots = batch.next_token_slots()  # the last position of each sequence
    _, kn, vn = batch.step_inputs(0)
    pk.kv_append(batch.pool, 0, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    return inst, batch


CASES = [  # (G, C, kv, designs); mma launches take up to 64 query rows per KV head, tc 128 per CTA
    (4, 2, "bf16", ("mma", "simt", "tc")),
    (4, 2, "fp8", ("mma",)),
    (2, 4, "bf16", ("mma", "simt")),
    (1, 8, "bf16", ("mma", "simt", "tc")),
    (2, 4, "f32", ("simt",)),
    (4, 4, "bf16", ("mma", "simt")),    # 16 rows: two column groups of warps
    (4, 8, "bf16", ("mma", "simt")),    # 32 rows; SIMT in two launches
    (4, 8, "fp8", ("mma",)),
    (4, 16, "bf16", ("mma", "tc")),     # 64 rows: two n-tiles per warp / half a tcgen05 tile
    (4, 16, "fp8", ("mma",)),
    (4, 40, "bf16", ("mma", "simt", "tc")),  # chunks 16 + 16 + 8 (mma); 160 rows = 2 tcgen05 tiles
    (8, 8, "bf16", ("mma", "tc")),      # 64 rows
    (1, 100, "bf16", ("mma", "tc")),    # chunks 64 + 36 (mma)
    (3, 5, "bf16", ("mma", "tc")),      # 3 query heads per KV head: 15 rows padded to 16
    (4, 100, "bf16", ("tc",)),          # 400 rows: 4 tcgen05 row tiles, the last partial
]


@pytest.mark.parametrize("split", [0, 64])
@pytest.mark.parametrize("G,C,kv,algos", CASES, ids=lambda x: str(x))
def test_multi_query_parity(G, C, kv, algos, split):
    lens = (C - 1, C, C + 1, 17, 64, 65, 300, 1000) if C < 64 else (C - 1, C, C + 1, 17, 130, 300, 1000, 1500)
    if "tc" in algos and split:
        algos = tuple(x for x in algos if x != "tc")  # the tcgen05 design takes no fixed splits
        if not algos:
            pytest.skip("fixed splits: tcgen05 design not used")
    w = _w("mq_%s_g%d_c%d" % (kv, G, C), G, 2, kv, "f32" if kv == "f32" else "bf16", lens,
           D=64 if kv == "f32" else 128)
    inst, batch = _filled(w)
    tables, lens_t = batch.tables(), batch.seq_lens()
    q = torch.randn(w.num_seqs, C, w.num_q_heads, w.head_dim, generator=torch.Generator().manual_seed(C))
    q = q.to(wl.DTYPES[w.query_dtype])
    ref, _ = oracle_reference_mq(w, inst.k_scale, inst.v_scale, 0, q, tables, lens_t.tolist(), list(range(w.num_seqs)))
    for algo in algos:
        out = pk.paged_multi_query_attention(q.cuda(), batch.pool, 0, tables.cuda(), lens_t.cuda(),
                                             int(lens_t.max()), w.scale, split_tokens=split, algo=algo)
        torch.cuda.synchronize()
        compare(out, ref, TOL[kv], "%s algo=%s split=%d" % (w.name, algo, split))
        # queries at negative positions (sequence shorter than C) are zero rows
        assert torch.all(out[0, 0] == 0)
    assert batch.pool.errors() == 0


@pytest.mark.parametrize("bs", [32, 64])
def test_tc_block_sizes(bs):
    """The tcgen05 design at 32- and 64-token blocks: one TMA box per block
    half covers 32 or 64 token rows, so a 64-token tile spans 2 or 1 blocks."""
    G, C = 4, 40
    lens = (C - 1, C, 31, 33, 63, 64, 65, 129, 700, 1500)
    w = _w("mq_tc_bs%d" % bs, G, 2, "bf16", "bf16", lens, bs=bs)
    inst, batch = _filled(w)
    tables, lens_t = batch.tables(), batch.seq_lens()
    q = torch.randn(w.num_seqs, C, w.num_q_heads, w.head_dim, generator=torch.Generator().manual_seed(bs))
    q = q.to(torch.bfloat16)
    assert pk.multi_query_algo(batch.pool, C, w.num_q_heads) == "tc"
    ref, _ = oracle_reference_mq(w, inst.k_scale, inst.v_scale, 0, q, tables, lens_t.tolist(), list(range(w.num_seqs)))
    out = pk.paged_multi_query_attention(q.cuda(), batch.pool, 0, tables.cuda(), lens_t.cuda(),
                                         int(lens_t.max()), w.scale, algo="tc")
    torch.cuda.synchronize()
    compare(out, ref, TOL["bf16"], w.name)
    assert torch.all(out[0, 0] == 0)
    assert batch.pool.errors() == 0


def test_one_query_equals_decode():
    w = _w("mq_one", 4, 2, "bf16", "bf16", (5, 100, 700))
    inst, batch = _filled(w)
    tables, lens = batch.tables().cuda(), batch.seq_lens().cuda()
    q = torch.randn(w.num_seqs, 1, w.num_q_heads, w.head_dim).to(torch.bfloat16).cuda()
    for algo in ("mma", "simt"):
        a = pk.paged_multi_query_attention(q, batch.pool, 0, tables, lens, int(lens.max()), w.scale, algo=algo)
        b = pk.paged_decode_attention(q[:, 0].contiguous(), batch.pool, 0, tables, lens, int(lens.max()), w.scale,
                                      algo=algo)
        assert torch.equal(a[:, 0], b)


@pytest.mark.parametrize("name,algo", [("specverify", "auto"),
                                       ("specverify", "mma"),
                                       ("prefill", "auto")])
def test_multi_query_workload_full_size(name, algo, record_property):
    """The benchmark's multi-query step at full size (append the last C
    positions, then attend), every sequence checked against the oracle."""
    w = wl.WORKLOADS[name]
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    slots = batch.next_token_slots()
    q, kn, vn = batch.step_inputs(0)
    pk.kv_append(batch.pool, 0, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    tables, lens = batch.tables(), batch.seq_lens()
    assert torch.equal(lens, inst.lens)
    out = pk.paged_multi_query_attention(q.cuda(), batch.pool, 0, tables.cuda(), lens.cuda(), int(lens.max()),
                                         w.scale, algo=algo)
    torch.cuda.synchronize()
    ref, _ = oracle_reference_mq(w, inst.k_scale, inst.v_scale, 0, q, tables, lens.tolist(), list(range(w.num_seqs)))
    max_abs, max_rel = compare(out, ref, TOL[w.kv_dtype], "%s algo=%s" % (name, algo))
    record_property("max_abs_err", max_abs)
    record_property("max_rel_err", max_rel)
    assert batch.pool.errors() == 0


@pytest.mark.parametrize("C,lens", [(8, (20000, 9000, 4097, 0, 5)), (1, (30000, 64, 65)), (32, (12345, 31, 2))])
def test_tc_balanced_few_long_sequences(C, lens):
    """A few long sequences: fewer (sequence, KV head) units than CTA slots, so
    the tcgen05 design shares every unit's tiles among many persistent CTAs and
    the last CTA to finish a unit merges its pieces (dozens of them here)."""
    G = 4
    w = _w("mq_tc_long_c%d" % C, G, 2, "bf16", "bf16", lens, bs=32)
    inst, batch = _filled(w)
    tables, lens_t = batch.tables(), batch.seq_lens()
    q = torch.randn(w.num_seqs, C, w.num_q_heads, w.head_dim, generator=torch.Generator().manual_seed(C + 5))
    q = q.to(torch.bfloat16)
    ref, _ = oracle_reference_mq(w, inst.k_scale, inst.v_scale, 0, q, tables, lens_t.tolist(), list(range(w.num_seqs)))
    _, _, wsb = pk.multi_query_plan(batch.pool, w.num_seqs, C, w.num_q_heads, int(lens_t.max()), 0)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    for rep in range(2):  # the merge counters are back at zero for the second call
        out = pk.paged_multi_query_attention(q.cuda(), batch.pool, 0, tables.cuda(), lens_t.cuda(),
                                             int(lens_t.max()), w.scale, algo="tc", workspace=ws)
        torch.cuda.synchronize()
        compare(out, ref, TOL["bf16"], "%s rep %d" % (w.name, rep))
        assert batch.pool.errors() == 0
    assert torch.count_nonzero(ws[: 4 * w.num_seqs * w.num_kv_heads]) == 0


def test_tc_grid_many_sequences():
    """More sequences than the grid schedule ranks by length (128) and more
    (sequence, KV head) units than CTA slots: one CTA per unit in blockIdx
    order, every element checked."""
    G, C, B = 4, 8, 160
    lens = tuple(1 + (37 * b) % 600 for b in range(B))
    w = _w("mq_tc_many", G, 2, "bf16", "bf16", lens, bs=16)
    inst, batch = _filled(w)
    tables, lens_t = batch.tables(), batch.seq_lens()
    q = torch.randn(w.num_seqs, C, w.num_q_heads, w.head_dim, generator=torch.Generator().manual_seed(11))
    q = q.to(torch.bfloat16)
    ref, _ = oracle_reference_mq(w, inst.k_scale, inst.v_scale, 0, q, tables, lens_t.tolist(), list(range(w.num_seqs)))
    out = pk.paged_multi_query_attention(q.cuda(), batch.pool, 0, tables.cuda(), lens_t.cuda(),
                                         int(lens_t.max()), w.scale, algo="tc")
    torch.cuda.synchronize()
    compare(out, ref, TOL["bf16"], w.name)
    assert batch.pool.errors() == 0


@pytest.mark.parametrize("algo", ["tc", "mma"])
def test_all_sequences_empty(algo):
    """No sequence has a visible token: no tiles at all, every output row is zero."""
    w = _w("mq_empty_%s" % algo, 4, 2, "bf16", "bf16", (40, 7, 100), bs=32)  # (a pool needs blocks)
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    tables = batch.tables()
    lens_t = torch.zeros(w.num_seqs, dtype=torch.int32)
    q = torch.randn(w.num_seqs, 8, w.num_q_heads, w.head_dim, generator=torch.Generator().manual_seed(9))
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    pk.paged_multi_query_attention(q.to(torch.bfloat16).cuda(), batch.pool, 0, tables.cuda(), lens_t.cuda(), 0,
                                   w.scale, out=out, algo=algo)
    torch.cuda.synchronize()
    assert torch.all(out == 0)
    assert batch.pool.errors() == 0


@pytest.mark.parametrize("C", [16, 64])
def test_tc_back_to_back_launches(C):
    """Many tcgen05 launches in a row, with nothing between them: no error
    bits, every call bit-identical to the first and close to the warp-level
    design (guards the pipeline's barrier protocol)."""
    w = _w("tc_repeat", 4, 8, "bf16", "bf16", (128, 700, 1500, 4096, 2100, 333, 64 + C, 3000))
    inst, batch = _filled(w)
    tables, lens = batch.tables().cuda(), batch.seq_lens().cuda()
    q = torch.randn(w.num_seqs, C, w.num_q_heads, w.head_dim, generator=torch.Generator().manual_seed(5))
    q = q.to(torch.bfloat16).cuda()
    max_len = int(lens.max())
    first = pk.paged_multi_query_attention(q, batch.pool, 0, tables, lens, max_len, w.scale, algo="tc")
    outs = [torch.empty_like(first) for _ in range(40)]
    for o in outs:
        pk.paged_multi_query_attention(q, batch.pool, 0, tables, lens, max_len, w.scale, out=o, algo="tc")
    torch.cuda.synchronize()
    assert batch.pool.errors() == 0
    for o in outs:
        assert torch.equal(o, first)
    ref = pk.paged_multi_query_attention(q, batch.pool, 0, tables, lens, max_len, w.scale, algo="mma")
    torch.cuda.synchronize()
    assert (first.float() - ref.float()).abs().max().item() < 2e-2
