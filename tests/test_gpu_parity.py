"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases compare every output element; they span several 64-token tiles,
several splits and ragged tails.  Full-size workloads run in the benchmark's
launch configuration and compare every sequence of the batch, every element.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_194_gb300 import binding as pk
from paged_kv_cache_194_gb300 import workloads as wl
from paged_kv_cache_194_gb300.decode import DecodeBatch

from parity import TOL, compare, oracle_reference

pytestmark = pytest.mark.gpu

EDGE_LENS = (1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 300, 1000)


def _w(name, G, Hkv, D, bs, kv, ind, lens, dist="normal", seed=21, qd=""):
    return wl.Workload(name, seed, len(lens), G * Hkv, Hkv, D, bs, kv, ind, 1.0 / math.sqrt(D),
                       lens="fixed", fixed_lens=tuple(lens), dist=dist, q_dtype=qd)


SMALL = [
    wl.WORKLOADS["tiny"],
    _w("bf16_g4_d128_bs16", 4, 2, 128, 16, "bf16", "bf16", EDGE_LENS),
    _w("bf16_g1_d128_bs32", 1, 3, 128, 32, "bf16", "bf16", (5, 64, 200, 33)),
    _w("bf16_g2_d64_bs64", 2, 2, 64, 64, "bf16", "bf16", (1, 64, 65, 500)),
    _w("bf16_g8_d128_bs16", 8, 1, 128, 16, "bf16", "bf16", (7, 130, 257)),
    _w("bf16_g8_d64_bs32", 8, 2, 64, 32, "bf16", "bf16", (31, 32, 96)),
    _w("fp8_g4_d128_bs64", 4, 2, 128, 64, "fp8", "bf16", EDGE_LENS),
    _w("fp8_g2_d64_bs16", 2, 2, 64, 16, "fp8", "bf16", (3, 80, 129)),
    _w("fp8_from_f32_g4", 4, 1, 128, 32, "fp8", "f32", (40, 100), qd="bf16"),
    _w("bf16_from_f32_g4", 4, 1, 128, 16, "bf16", "f32", (40, 100), qd="bf16"),
    _w("f32_g4_d128_bs32", 4, 2, 128, 32, "f32", "f32", (1, 70, 190), dist="uniform"),
    _w("f32_g16_d64_bs16", 16, 1, 64, 16, "f32", "f32", (17, 99), dist="uniform"),
    _w("with_empty_seq", 4, 2, 128, 16, "bf16", "bf16", (0, 5, 0, 77)),
    # KV-head pairs (tensor-core decode at 16-token blocks, even KV-head count)
    _w("pair_g1_bs16", 1, 4, 128, 16, "bf16", "bf16", (1, 16, 33, 200, 0, 511)),
    _w("pair_g2_bs16", 2, 2, 128, 16, "bf16", "bf16", EDGE_LENS),
    _w("pair_g3_bs16", 3, 2, 128, 16, "bf16", "bf16", (2, 17, 64, 129, 700)),
    # several KV-head pairs per sequence (4 and 8 KV heads)
    _w("pairs_hkv4_g4_bs16", 4, 4, 128, 16, "bf16", "bf16", EDGE_LENS),
    _w("pairs_hkv8_g2_bs16", 2, 8, 128, 16, "bf16", "bf16", (1, 16, 17, 250, 0, 2049)),
    _w("pairs_hkv4_g3_bs16", 3, 4, 128, 16, "bf16", "bf16", (2, 17, 64, 129, 700)),
]


def _run_step(batch, layer=0, split=0, algo="auto", step=0):
    """One decode step through the C ABI: append the new token, attend."""
    slots = batch.next_token_slots()
    q, kn, vn = batch.step_inputs(layer, step)
    pk.kv_append(batch.pool, layer, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    tables, lens = batch.tables(), batch.seq_lens()
    out = pk.paged_decode_attention(q.cuda(), batch.pool, layer, tables.cuda(), lens.cuda(),
                                    int(lens.max()), batch.w.scale, split_tokens=split, algo=algo)
    torch.cuda.synchronize()
    return q, tables, lens, out


def _algos(w):
    """Every kernel design that serves the workload."""
    designs = []
    if pk.lib() and w.kv_dtype != "f32" and w.head_dim == 128 and w.block_size in (16, 32, 64) and w.group <= 64:
        designs.append("mma")
    if w.group in (1, 2, 4, 8, 16) and w.group * {"f32": 4, "bf16": 8, "fp8": 16}[w.kv_dtype] <= 64:
        designs.append("simt")
    return designs


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
@pytest.mark.parametrize("split", [0, 64, 128])
def test_small_parity(w, split, record_property):
    if split % w.block_size:
        pytest.skip("split must be a multiple of the block size")
    inst = wl.instance(w)
    for algo in _algos(w):
        batch = DecodeBatch(inst)
        q, tables, lens, out = _run_step(batch, split=split, algo=algo)
        ref, _ = oracle_reference(w, inst.k_scale, inst.v_scale, 0, q, tables, lens.tolist(),
                                  list(range(w.num_seqs)))
        e = compare(out, ref, TOL[w.kv_dtype], "%s split=%d algo=%s" % (w.name, split, algo))
        record_property("max_abs_" + algo, e[0])
        record_property("max_rel_" + algo, e[1])
        assert batch.pool.errors() == 0


@pytest.mark.parametrize("w", [SMALL[1], SMALL[6], SMALL[10], SMALL[0]], ids=lambda w: w.name)
def test_append_bitexact_whole_pool(w):
    """The GPU pool after prefill + one step equals the oracle's pool byte for
    byte, including blocks no token touched (sentinel fill)."""
    inst = wl.instance(w)
    batch = DecodeBatch(inst, fill_byte=0x5A)
    slots = batch.next_token_slots()
    q, kn, vn = batch.step_inputs(0)
    pk.kv_append(batch.pool, 0, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    tables = batch.tables().numpy()
    opool = oracle.OraclePool(1, inst.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype,
                              inst.k_scale, inst.v_scale, fill=0x5A)
    for b in range(w.num_seqs):
        L = int(inst.lens[b])
        if L == 0:
            continue
        k, v = wl.seq_kv(w, 0, b, L)
        oracle.kv_append(opool, 0, k, v, w.in_dtype, oracle.slot_mapping(tables, w.block_size, np.full(L, b), np.arange(L)))
    gk = batch.pool.k.view(torch.uint8).cpu().numpy().ravel()
    gv = batch.pool.v.view(torch.uint8).cpu().numpy().ravel()
    assert np.array_equal(gk, opool.k.view(np.uint8).ravel())
    assert np.array_equal(gv, opool.v.view(np.uint8).ravel())


def test_append_skip_slot_and_bad_slot_flag():
    w = SMALL[1]
    inst = wl.instance(w)
    pool = pk.KVPool(1, 8, 16, 2, 128, "bf16", fill=0)
    k = torch.randn(3, 2, 128, dtype=torch.bfloat16, device="cuda")
    before = pool.k.clone()
    slots = torch.tensor([-1, 8 * 16, 5], dtype=torch.int64, device="cuda")  # skip, out of range, ok
    pk.kv_append(pool, 0, k, k, slots)
    torch.cuda.synchronize()
    assert pool.errors() & pk.ERRBIT_SLOT
    after = pool.k.view(8, 2, 16, 128)
    assert torch.equal(after[0, :, 5], k[2])
    mask = torch.ones(8, 2, 16, dtype=torch.bool, device="cuda")
    mask[0, :, 5] = False
    assert torch.equal(after[mask], before.view(8, 2, 16, 128)[mask])


def test_single_token_is_exact():
    w = _w("len1", 4, 2, 128, 16, "bf16", "bf16", (1, 1, 1, 1))
    inst = wl.instance(w)
    for algo in ("simt", "mma"):
        batch = DecodeBatch(inst)
        q, tables, lens, out = _run_step(batch, algo=algo)
        _, kn, vn = batch.step_inputs(0)
        want = vn.cuda().repeat_interleave(w.group, dim=1)  # [B, Hq, D]
        assert torch.equal(out, want), algo


@pytest.mark.parametrize("algo", ["simt", "mma"])
@pytest.mark.parametrize("idx", [1, 6], ids=["bf16", "fp8"])
def test_block_permutation_gives_identical_output(idx, algo):
    w = SMALL[idx]
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    q, tables, lens, out = _run_step(batch, algo=algo)
    perm = torch.randperm(inst.num_blocks, generator=torch.Generator().manual_seed(5))
    pool2 = pk.KVPool(1, inst.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype,
                      inst.k_scale, inst.v_scale)
    pool2.k[:, perm.cuda()] = batch.pool.k
    pool2.v[:, perm.cuda()] = batch.pool.v
    t2 = torch.where(tables >= 0, perm[tables.clamp(min=0).long()].to(torch.int32), tables)
    out2 = pk.paged_decode_attention(q.cuda(), pool2, 0, t2.cuda(), lens.cuda(), int(lens.max()), w.scale,
                                     algo=algo)
    assert torch.equal(out, out2)


def test_auto_picks_tensor_cores_for_bf16_and_fp8():
    for idx, want in ((1, "mma"), (6, "mma"), (3, "simt"), (0, "simt")):
        w = SMALL[idx]
        inst = wl.instance(w)
        pool = pk.KVPool(1, 4, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, inst.k_scale, inst.v_scale)
        assert pk.decode_algo(pool, w.num_q_heads) == want, w.name


@pytest.mark.parametrize("algo", ["simt", "mma"])
def test_split_equals_no_split(algo):
    w = _w("splits", 4, 2, 128, 16, "bf16", "bf16", (3000, 1234, 64, 4096))
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    q, tables, lens, out_split = _run_step(batch, split=64, algo=algo)
    out_one = pk.paged_decode_attention(q.cuda(), batch.pool, 0, tables.cuda(), lens.cuda(), int(lens.max()),
                                        w.scale, split_tokens=4096, algo=algo)
    np.testing.assert_allclose(out_split.float().cpu().numpy(), out_one.float().cpu().numpy(), rtol=8e-3, atol=2e-3)


@pytest.mark.parametrize("algo", ["simt", "mma"])
def test_device_index_faults_are_flagged_not_fatal(algo):
    w = _w("faults", 4, 2, 128, 16, "bf16", "bf16", (40, 50))
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    q, tables, lens, out = _run_step(batch, algo=algo)
    assert batch.pool.errors() == 0
    bad = tables.clone()
    bad[1, 1] = inst.num_blocks  # one past the pool
    pk.paged_decode_attention(q.cuda(), batch.pool, 0, bad.cuda(), lens.cuda(), int(lens.max()), w.scale, algo=algo)
    torch.cuda.synchronize()
    assert batch.pool.errors() & pk.ERRBIT_BLOCK_ID
    batch.pool.clear_errors()
    long_lens = lens.clone()
    long_lens[0] = int(lens.max()) + 5  # beyond max_seq_len given to the call
    o3 = pk.paged_decode_attention(q.cuda(), batch.pool, 0, tables.cuda(), long_lens.cuda(), int(lens.max()), w.scale,
                                   algo=algo)
    torch.cuda.synchronize()
    assert batch.pool.errors() & pk.ERRBIT_SEQ_LEN
    assert torch.isfinite(o3.float()).all()


# ------------------------------------------------------------- full sizes
# Every sequence of the batch, every head and element, in the launch
# configuration the benchmark times.


@pytest.mark.parametrize("name", ["llama", "fp8"])
def test_full_size_whole_batch(name, record_property):
    w = wl.WORKLOADS[name]
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    q, tables, lens, out = _run_step(batch)  # default schedule, as the benchmark runs it
    seqs = list(range(w.num_seqs))
    ref, _ = oracle_reference(w, inst.k_scale, inst.v_scale, 0, q, tables, lens.tolist(), seqs)
    max_abs, max_rel = compare(out, ref, TOL[w.kv_dtype], name)
    record_property("max_abs", max_abs)
    record_property("max_rel", max_rel)
    record_property("seqs_compared", len(seqs))
    assert batch.pool.errors() == 0


def test_ragged_in_flight_steps(record_property):
    """The in-flight batch: 8 steps of append + attention with the block
    manager growing the tables; every sequence compared at the first and the
    last step."""
    w = wl.WORKLOADS["ragged"]
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    seqs = list(range(w.num_seqs))
    worst = (0.0, 0.0)
    for step in range(w.steps):
        q, tables, lens, out = _run_step(batch, step=step)
        if step in (0, w.steps - 1):
            ref, _ = oracle_reference(w, 1.0, 1.0, 0, q, tables, lens.tolist(), seqs)
            e = compare(out, ref, TOL["bf16"], "ragged step %d" % step)
            worst = (max(worst[0], e[0]), max(worst[1], e[1]))
        batch.bm.check()
    record_property("max_abs", worst[0])
    record_property("max_rel", worst[1])
    assert batch.pool.errors() == 0
    assert lens.tolist() == [int(x) + w.steps - 1 for x in inst.lens]


@pytest.mark.parametrize("split", ["recipe", "balanced"])
def test_long_context_layers(split, record_property):
    """4 sequences of 131072 tokens, layers 0 and 31 of the 32-layer pool,
    every sequence compared: with the recipe's 2048-token splits (fixed
    splits + combine kernel) and with the balanced schedule, which cuts each
    (sequence, KV-head pair) into pieces at data-dependent points and merges
    them in the kernel; its per-unit counters are back at zero after each call."""
    w = wl.WORKLOADS["long"]
    inst = wl.instance(w)
    batch = DecodeBatch(inst, cpu_layers=[0, 31])
    slots = batch.next_token_slots()
    tables, lens = batch.tables(), batch.seq_lens()
    S = w.split_tokens if split == "recipe" else 0
    ws = pk.workspace_for(batch.pool, w.num_seqs, w.num_q_heads, int(lens.max()), S)
    for layer in (0, 31):
        q, kn, vn = batch.step_inputs(layer)
        pk.kv_append(batch.pool, layer, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
        out = pk.paged_decode_attention(q.cuda(), batch.pool, layer, tables.cuda(), lens.cuda(),
                                        int(lens.max()), w.scale, split_tokens=S, workspace=ws)
        torch.cuda.synchronize()
        if S == 0:
            assert int(ws[:4 * w.num_seqs * w.num_kv_heads].count_nonzero()) == 0
        ref, _ = oracle_reference(w, 1.0, 1.0, layer, q, tables, lens.tolist(), list(range(w.num_seqs)))
        e = compare(out, ref, TOL["bf16"], "long layer %d (%s)" % (layer, split))
        record_property("max_abs_layer%d" % layer, e[0])
        record_property("max_rel_layer%d" % layer, e[1])
    assert batch.pool.errors() == 0


@pytest.mark.parametrize("scale_kind", ["huge", "tiny", "mixed"])
@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_query_magnitudes(kv, scale_kind, record_property):
    """BF16 queries far outside f16's range (up to 1e6) and far below its
    normal range (down to 1e-6): the query is never quantised, so every
    design must match the oracle, which uses the exact BF16 values."""
    w = _w("qmag_" + kv, 4, 2, 128, 64 if kv == "fp8" else 16, kv, "bf16", (1, 17, 300, 1000, 2500), seed=44)
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    slots = batch.next_token_slots()
    q0, kn, vn = batch.step_inputs(0)
    pk.kv_append(batch.pool, 0, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    tables, lens = batch.tables(), batch.seq_lens()
    g = torch.Generator().manual_seed(45)
    if scale_kind == "huge":
        mag = torch.tensor([1e6, 3e5, 7e4, 65504.0 * 4])[torch.randint(0, 4, (w.num_seqs, w.num_q_heads, 1), generator=g)]
    elif scale_kind == "tiny":
        mag = torch.tensor([1e-6, 3e-5, 1e-4, 2.0 ** -20])[torch.randint(0, 4, (w.num_seqs, w.num_q_heads, 1), generator=g)]
    else:  # a row mixes huge and tiny entries; rows differ by orders of magnitude
        mag = 10.0 ** torch.randint(-6, 7, (w.num_seqs, w.num_q_heads, w.head_dim), generator=g).double()
    q = (q0.double() * mag).to(torch.bfloat16)
    assert torch.isfinite(q.float()).all()
    ref, _ = oracle_reference(w, inst.k_scale, inst.v_scale, 0, q, tables, lens.tolist(), list(range(w.num_seqs)))
    for algo in _algos(w):
        out = pk.paged_decode_attention(q.cuda(), batch.pool, 0, tables.cuda(), lens.cuda(), int(lens.max()),
                                        w.scale, algo=algo)
        torch.cuda.synchronize()
        e = compare(out, ref, TOL[kv], "%s %s algo=%s" % (kv, scale_kind, algo))
        record_property("max_abs_" + algo, e[0])
    assert batch.pool.errors() == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_balanced_schedule_repeats_and_leaves_counters_zero(kv):
    """Three calls on one workspace give identical bits; the per-sequence
    counters at the front of the workspace are zero after every call."""
    w = _w("balanced_" + kv, 4, 2, 128, 16, kv, "bf16", (5000, 1, 0, 64, 700, 4096, 129), seed=33)
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    q, tables, lens, _ = _run_step(batch, algo="mma")
    ws = pk.workspace_for(batch.pool, w.num_seqs, w.num_q_heads, int(lens.max()))
    outs = []
    for _ in range(3):
        outs.append(pk.paged_decode_attention(q.cuda(), batch.pool, 0, tables.cuda(), lens.cuda(), int(lens.max()),
                                              w.scale, workspace=ws, algo="mma"))
        torch.cuda.synchronize()
        assert int(ws[:4 * w.num_seqs * w.num_kv_heads].count_nonzero()) == 0
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    ref, _ = oracle_reference(w, inst.k_scale, inst.v_scale, 0, q, tables, lens.tolist(), list(range(w.num_seqs)))
    compare(outs[0], ref, TOL[kv], "balanced " + kv)
    assert batch.pool.errors() == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_balanced_schedule_tiny_batch(kv):
    """Fewer tiles than CTAs: most CTAs own nothing (over FP8 their publisher
    warp is told so by the consumers)."""
    w = _w("balanced_tiny_" + kv, 4, 1, 128, 16, kv, "bf16", (3, 70), seed=34)
    inst = wl.instance(w)
    batch = DecodeBatch(inst)
    q, tables, lens, out = _run_step(batch, algo="mma")
    ref, _ = oracle_reference(w, inst.k_scale, inst.v_scale, 0, q, tables, lens.tolist(), [0, 1])
    compare(out, ref, TOL[kv], "balanced tiny " + kv)
    assert batch.pool.errors() == 0
