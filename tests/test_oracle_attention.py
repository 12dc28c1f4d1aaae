"""Pins for the oracle's slot mapping, append and paged attention.

The oracle pipeline (slot mapping -> append -> gather + fp64 softmax
attention) is compared with things that do not share its code: contiguous,
unpaged attention written with torch's own fp64 softmax/matmul; torch's FP8
cast for the dequantised reference; closed-form special cases; invariants the
paging must not break; and the pages' printed numbers.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_194_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _small(name="small", G=4, Hkv=2, D=128, bs=16, kv="bf16", ind="bf16", lens=(1, 5, 16, 17, 40, 100),
           dist="normal", seed=11):
    return wl.Workload(name, seed, len(lens), G * Hkv, Hkv, D, bs, kv, ind, 1.0 / math.sqrt(D),
                       lens="fixed", fixed_lens=tuple(lens), dist=dist)


def _fill_oracle(inst, layer=0):
    """Oracle pool holding every token of every sequence of `inst`."""
    w = inst.w
    pool = oracle.OraclePool(w.num_layers, inst.num_blocks, w.block_size, w.num_kv_heads,
                             w.head_dim, w.kv_dtype, inst.k_scale, inst.v_scale)
    rows = {}
    for b in range(w.num_seqs):
        L = int(inst.lens[b])
        k, v = wl.seq_kv(w, layer, b, L)
        rows[b] = (k, v)
        if L == 0:
            continue
        slots = oracle.slot_mapping(inst.tables, w.block_size, np.full(L, b), np.arange(L))
        oracle.kv_append(pool, layer, k, v, w.in_dtype, slots)
    return pool, rows


def _dequant_torch(x, kv_dtype, scale):
    """Reference values of stored rows, computed with torch's own casts."""
    if kv_dtype == "fp8":
        inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(scale, dtype=torch.float32)
        return (x.float() * inv).to(torch.float8_e4m3fn).to(torch.float64) * scale
    if kv_dtype == "bf16":
        return x.to(torch.bfloat16).to(torch.float64)
    return x.to(torch.float64)


def _brute(inst, rows, q):
    """Contiguous, unpaged attention in torch fp64 (the scale is the binary32
    value the library's interface carries)."""
    w = inst.w
    B, Hq, D = q.shape
    out = torch.zeros(B, Hq, D, dtype=torch.float64)
    lse = torch.full((B, Hq), -math.inf, dtype=torch.float64)
    for b in range(B):
        k, v = rows[b]
        if k.shape[0] == 0:
            continue
        K = _dequant_torch(k, w.kv_dtype, inst.k_scale)  # [L, Hkv, D]
        V = _dequant_torch(v, w.kv_dtype, inst.v_scale)
        for hq in range(Hq):
            h = hq // w.group
            s = (K[:, h, :] @ q[b, hq].to(torch.float64)) * float(np.float32(w.scale))
            out[b, hq] = torch.softmax(s, 0) @ V[:, h, :]
            lse[b, hq] = torch.logsumexp(s, 0)
    return out.numpy(), lse.numpy()


CASES = [
    _small("bf16_g4", kv="bf16"),
    _small("fp8_g4", kv="fp8", bs=32),
    _small("f32_g2", G=2, Hkv=3, D=64, bs=16, kv="f32", ind="f32", dist="uniform"),
    _small("bf16_g8_bs64", G=8, Hkv=1, D=64, bs=64, lens=(63, 64, 65, 200)),
    _small("f32_to_bf16", kv="bf16", ind="f32", lens=(3, 33)),
    _small("f32_to_fp8", kv="fp8", ind="f32", lens=(7, 70), bs=16),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_oracle_matches_contiguous_bruteforce(w):
    inst = wl.instance(w)
    pool, rows = _fill_oracle(inst)
    q = wl.query(w)
    out, lse = oracle.paged_attention(q, w.in_dtype, pool, 0, inst.tables, inst.lens, w.scale)
    ref, ref_lse = _brute(inst, rows, q)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_tiny_workload_matches_bruteforce():
    w = wl.WORKLOADS["tiny"]
    inst = wl.instance(w)
    pool, rows = _fill_oracle(inst)
    q = wl.query(w)
    out, lse = oracle.paged_attention(q, "f32", pool, 0, inst.tables, inst.lens, w.scale)
    ref, ref_lse = _brute(inst, rows, q)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_weights_sum_to_one():
    # with every V row equal to 1 the output is the sum of the weights
    w = _small(kv="bf16")
    inst = wl.instance(w)
    pool, _ = _fill_oracle(inst)
    pool.v[...] = np.uint16(0x3F80)  # bf16 1.0
    out, _ = oracle.paged_attention(wl.query(w), "bf16", pool, 0, inst.tables, inst.lens, w.scale)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-14)


def test_single_token_returns_its_value_row():
    w = _small(lens=(1, 1, 1), kv="bf16")
    inst = wl.instance(w)
    pool, rows = _fill_oracle(inst)
    out, _ = oracle.paged_attention(wl.query(w), "bf16", pool, 0, inst.tables, inst.lens, w.scale)
    for b in range(3):
        v = rows[b][1].to(torch.float64)[0]  # [Hkv, D]
        for hq in range(w.num_q_heads):
            assert np.array_equal(out[b, hq], v[hq // w.group].numpy())


@pytest.mark.parametrize("mode", ["zero_q", "zero_scale"])
def test_uniform_weights_give_mean(mode):
    w = _small(kv="bf16", lens=(9, 31))
    inst = wl.instance(w)
    pool, rows = _fill_oracle(inst)
    q = wl.query(w)
    scale = w.scale
    if mode == "zero_q":
        q = torch.zeros_like(q)
    else:
        scale = 0.0
    out, lse = oracle.paged_attention(q, "bf16", pool, 0, inst.tables, inst.lens, scale)
    for b in range(2):
        mean = rows[b][1].to(torch.float64).mean(0)  # [Hkv, D]
        for hq in range(w.num_q_heads):
            np.testing.assert_allclose(out[b, hq], mean[hq // w.group].numpy(), rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse[b], math.log(int(inst.lens[b])), rtol=1e-14)


def test_block_permutation_invariance():
    w = _small(kv="bf16", lens=(17, 50, 64))
    inst = wl.instance(w)
    pool, _ = _fill_oracle(inst)
    q = wl.query(w)
    out, lse = oracle.paged_attention(q, "bf16", pool, 0, inst.tables, inst.lens, w.scale)
    perm = torch.randperm(inst.num_blocks, generator=torch.Generator().manual_seed(3)).numpy()
    pool2 = oracle.OraclePool(1, inst.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, "bf16")
    pool2.k[:, perm] = pool.k
    pool2.v[:, perm] = pool.v
    t = inst.tables.numpy()
    t2 = np.where(t >= 0, perm[np.maximum(t, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.paged_attention(q, "bf16", pool2, 0, t2, inst.lens, w.scale)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def test_windows_recombine_to_full():
    w = _small(kv="fp8", lens=(1, 100, 64, 250), bs=16)
    inst = wl.instance(w)
    pool, _ = _fill_oracle(inst)
    q = wl.query(w)
    full, full_lse = oracle.paged_attention(q, "bf16", pool, 0, inst.tables, inst.lens, w.scale)
    S = 48
    parts = [oracle.paged_attention(q, "bf16", pool, 0, inst.tables, inst.lens, w.scale,
                                    window=(s, s + S)) for s in range(0, 256, S)]
    for b in range(w.num_seqs):
        for hq in range(w.num_q_heads):
            o = np.stack([p[0][b, hq] for p in parts])
            l = np.array([p[1][b, hq] for p in parts])
            comb, comb_lse = oracle.lse_combine(o, l)
            np.testing.assert_allclose(comb, full[b, hq], rtol=1e-12, atol=1e-13)
            assert abs(comb_lse - full_lse[b, hq]) < 1e-12


def test_empty_sequence_and_empty_combine():
    w = _small(kv="bf16", lens=(0, 5))
    inst = wl.instance(w)
    pool, _ = _fill_oracle(inst)
    out, lse = oracle.paged_attention(wl.query(w), "bf16", pool, 0, inst.tables, inst.lens, w.scale)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0])) and np.all(np.isfinite(lse[1]))
    comb, cl = oracle.lse_combine(np.ones((3, 4)), np.full(3, -np.inf))
    assert np.all(comb == 0) and cl == -np.inf


def test_bad_block_id_is_reported():
    w = _small(kv="bf16", lens=(20,))
    inst = wl.instance(w)
    pool, _ = _fill_oracle(inst)
    bad = inst.tables.clone()
    bad[0, 1] = inst.num_blocks  # one past the pool
    with pytest.raises(IndexError):
        oracle.paged_attention(wl.query(w), "bf16", pool, 0, bad, inst.lens, w.scale)


def test_append_bytes_and_skip_slot():
    # f32 -> bf16 append rounds like torch; slot -1 writes nothing; other
    # slots keep their sentinel fill.
    w = _small(kv="bf16", ind="f32", lens=(5,))
    pool = oracle.OraclePool(1, 4, 16, 2, 128, "bf16", fill=0xAB)
    k, v = wl.seq_kv(w, 0, 0, 5)
    slots = np.array([3, -1, 16, 17, 63], dtype=np.int64)
    oracle.kv_append(pool, 0, k, v, "f32", slots)
    ref = k.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    flat = pool.k.reshape(4, 2, 16, 128)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        assert np.array_equal(flat[s // 16, :, s % 16], ref[t])
    touched = {(int(s) // 16, int(s) % 16) for s in slots if s >= 0}
    for blk in range(4):
        for off in range(16):
            if (blk, off) not in touched:
                assert np.all(flat[blk, :, off] == 0xABAB)


def test_fp8_append_matches_torch_cast():
    w = _small(kv="fp8", lens=(40,))
    inst = wl.instance(w)
    pool, rows = _fill_oracle(inst)
    k = rows[0][0]
    inv = torch.tensor(1.0, dtype=torch.float32) / torch.tensor(inst.k_scale, dtype=torch.float32)
    ref = (k.float() * inv).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    t = inst.tables[0].numpy()
    for p in range(40):
        blk = t[p // w.block_size]
        assert np.array_equal(pool.k[0, blk, :, p % w.block_size], ref[p])


def test_paging_diagram_tables():
    with open(os.path.join(GOLDEN, "paging_diagram.json")) as f:
        g = json.load(f)
    nb = g["num_blocks"]
    names = sorted(g["tables"])
    width = max(len(v) for v in g["tables"].values())
    tables = np.full((len(names), width), -1, dtype=np.int32)
    for i, n in enumerate(names):
        tables[i, :len(g["tables"][n])] = np.array(g["tables"][n]) - 1  # 0-based
    used = sorted(int(x) for x in tables.ravel() if x >= 0)
    free = sorted(int(x) - 1 for x in g["free"])
    assert sorted(used + free) == list(range(nb))  # every block is held or free, once
    bs, D = 4, 8
    lens = [bs * len(g["tables"][n]) for n in names]
    seq_idx = np.concatenate([np.full(L, i) for i, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    slots = oracle.slot_mapping(tables, bs, seq_idx, pos)
    # request A's token 5 lands in its second block (B4 -> id 3) at offset 1
    a = names.index("A")
    i5 = int(np.nonzero((seq_idx == a) & (pos == 5))[0][0])
    assert slots[i5] == 3 * bs + 1
    # the mapping is a bijection onto the held blocks' slots
    assert sorted(slots.tolist()) == sorted(b * bs + o for b in used for o in range(bs))
    # a value written through the mapping is read back through the table
    pool = oracle.OraclePool(1, nb, bs, 1, D, "f32")
    vals = torch.arange(len(pos) * D, dtype=torch.float32).reshape(len(pos), 1, D)
    oracle.kv_append(pool, 0, vals, vals, "f32", slots)
    for t in range(len(pos)):
        blk = tables[seq_idx[t], pos[t] // bs]
        assert np.array_equal(pool.k[0, blk, 0, pos[t] % bs], vals[t, 0].numpy())


def test_pages_closed_forms():
    with open(os.path.join(GOLDEN, "pages_closed_forms.json")) as f:
        g = json.load(f)
    for c in g["kv_bytes_per_token"]["cases"]:
        assert oracle.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"],
                                         c["bytes_per_elem"]) == c["bytes"]
    cap = g["pool_capacity"]
    bf16 = oracle.kv_bytes_per_token(32, 8, 128, 2)
    fp8 = oracle.kv_bytes_per_token(32, 8, 128, 1)
    assert cap["pool_bytes"] == 55 * 2**30
    assert cap["pool_bytes"] // bf16 == cap["bf16_tokens"]
    assert cap["pool_bytes"] // fp8 == cap["fp8_tokens"]
    assert cap["bf16_tokens"] // cap["context"] == cap["bf16_full_context_requests"]
    assert cap["fp8_tokens"] // cap["context"] == cap["fp8_full_context_requests"]
    ex = g["worked_example"]
    assert ex["tokens_per_request"] * bf16 == ex["bytes_per_request"]
    assert ex["bytes_per_request"] / 2**20 == ex["mib_per_request"]
    assert ex["requests"] * ex["bytes_per_request"] == ex["bytes_for_requests"]
    assert round(ex["bytes_for_requests"] / 2**30, 2) == ex["gib_for_requests_approx"]
    # the fp8 workload is the pages' 55 full-context requests
    w = wl.WORKLOADS["fp8"]
    assert w.num_seqs * w.fixed_lens[0] == cap["bf16_tokens"]


# ----------------------------------------------------------- multi-query

@pytest.mark.parametrize("C,G", [(1, 4), (2, 4), (4, 2), (8, 1)])
def test_multi_query_matches_causal_bruteforce(C, G):
    w = _small("mq", G=G, Hkv=2, kv="bf16", lens=(C, C + 1, 17, 64, 100))
    inst = wl.instance(w)
    pool, rows = _fill_oracle(inst)
    q = torch.randn(w.num_seqs, C, w.num_q_heads, w.head_dim,
                    generator=torch.Generator().manual_seed(C)).to(torch.bfloat16)
    out, lse = oracle.paged_attention_mq(q, "bf16", pool, 0, inst.tables, inst.lens, w.scale)
    sc = float(np.float32(w.scale))
    for b in range(w.num_seqs):
        L = int(inst.lens[b])
        K = rows[b][0].to(torch.float64)
        V = rows[b][1].to(torch.float64)
        for c in range(C):
            qpos = L - C + c
            for hq in range(w.num_q_heads):
                h = hq // G
                s = (K[:, h, :] @ q[b, c, hq].to(torch.float64)) * sc
                s[qpos + 1:] = -math.inf  # causal: nothing after the query's own position
                np.testing.assert_allclose(out[b, c, hq], (torch.softmax(s, 0) @ V[:, h, :]).numpy(),
                                           rtol=1e-12, atol=1e-12)
                assert abs(lse[b, c, hq] - float(torch.logsumexp(s, 0))) < 1e-12


def test_multi_query_negative_positions_give_zero_rows():
    """A sequence shorter than C: queries whose position L - C + c is negative
    see no token (a zero row, log-sum-exp -inf); the others see tokens 0 .. L - C + c."""
    C, G = 6, 2
    w = _small("mq_short", G=G, Hkv=2, kv="bf16", lens=(1, 2, 5, 6))
    inst = wl.instance(w)
    pool, rows = _fill_oracle(inst)
    q = torch.randn(w.num_seqs, C, w.num_q_heads, w.head_dim,
                    generator=torch.Generator().manual_seed(12)).to(torch.bfloat16)
    out, lse = oracle.paged_attention_mq(q, "bf16", pool, 0, inst.tables, inst.lens, w.scale)
    sc = float(np.float32(w.scale))
    for b in range(w.num_seqs):
        L = int(inst.lens[b])
        for c in range(C):
            qpos = L - C + c
            for hq in range(w.num_q_heads):
                if qpos < 0:
                    assert np.all(out[b, c, hq] == 0) and lse[b, c, hq] == -math.inf
                    continue
                h = hq // G
                K = rows[b][0].to(torch.float64)[: qpos + 1, h, :]
                V = rows[b][1].to(torch.float64)[: qpos + 1, h, :]
                s = (K @ q[b, c, hq].to(torch.float64)) * sc
                np.testing.assert_allclose(out[b, c, hq], (torch.softmax(s, 0) @ V).numpy(), rtol=1e-12, atol=1e-12)


def test_multi_query_rows_equal_decode_on_prefixes():
    """Query c is exactly decode attention over the first L - C + c + 1 tokens,
    and C = 1 is plain decode."""
    C = 3
    w = _small("mq_prefix", G=4, Hkv=2, kv="fp8", lens=(5, 40, 129))
    inst = wl.instance(w)
    pool, _ = _fill_oracle(inst)
    q = torch.randn(w.num_seqs, C, w.num_q_heads, w.head_dim,
                    generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    out, lse = oracle.paged_attention_mq(q, "bf16", pool, 0, inst.tables, inst.lens, w.scale)
    for c in range(C):
        lens_c = inst.lens - (C - 1 - c)
        ref, ref_lse = oracle.paged_attention(q[:, c].contiguous(), "bf16", pool, 0, inst.tables, lens_c, w.scale)
        assert np.array_equal(out[:, c], ref) and np.array_equal(lse[:, c], ref_lse)
    one, _ = oracle.paged_attention_mq(q[:, -1:].contiguous(), "bf16", pool, 0, inst.tables, inst.lens, w.scale)
    assert np.array_equal(one[:, 0], out[:, -1])
