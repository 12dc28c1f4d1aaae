"""Host-only checks of the C ABI and the block manager (no GPU needed).

The library must load and export every symbol include/pkv.h declares.
Argument validation is exercised only with calls that are rejected before
any launch, so nothing here touches device memory.
"""
import ctypes
import json
import os
import re

import numpy as np
import pytest

import oracle
from paged_kv_cache_194_gb300 import binding as pk
from paged_kv_cache_194_gb300 import workloads as wl
from paged_kv_cache_194_gb300.block_manager import BlockManager, OutOfBlocks

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _header_functions():
    src = open(os.path.join(ROOT, "include", "pkv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", src)
    skip = {"if", "for", "while", "sizeof", "return"}
    return sorted(set(n for n in names if n not in skip))


def test_library_exports_every_declared_symbol():
    L = pk.lib()
    declared = _header_functions()
    assert set(declared) == set(pk.EXPORTS), declared
    for name in declared:
        assert hasattr(L, name), name


def test_status_strings_and_closed_forms():
    L = pk.lib()
    for code in range(6):
        assert L.pkv_status_string(code)
    with open(os.path.join(GOLDEN, "pages_closed_forms.json")) as f:
        g = json.load(f)
    for c in g["kv_bytes_per_token"]["cases"]:
        dt = {2: "bf16", 1: "fp8"}[c["bytes_per_elem"]]
        assert pk.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], dt) == c["bytes"]
    cap = g["pool_capacity"]
    assert cap["pool_bytes"] // pk.kv_bytes_per_token(32, 8, 128, "bf16") == cap["bf16_tokens"]
    assert cap["pool_bytes"] // pk.kv_bytes_per_token(32, 8, 128, "fp8") == cap["fp8_tokens"]


FAKE = 0x10000  # aligned, never dereferenced: every call below is rejected first


def _desc(**kw):
    d = dict(num_layers=1, num_blocks=8, block_size=16, num_kv_heads=2, head_dim=128, kv_dtype=1,
             k_scale=1.0, v_scale=1.0, k_base=FAKE, v_base=FAKE, error_word=None)
    d.update(kw)
    return pk.PoolDesc(**d)


def _create(**kw):
    h = ctypes.c_void_p()
    d = _desc(**kw)
    rc = pk.lib().kv_pool_create(ctypes.byref(d), ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("kw,status", [
    (dict(block_size=8), 2), (dict(head_dim=96), 2), (dict(num_blocks=0), 1),
    (dict(k_base=None), 1), (dict(v_base=FAKE + 4), 1), (dict(kv_dtype=7), 1),
    (dict(kv_dtype=2, k_scale=0.0), 1), (dict(kv_dtype=2, v_scale=float("nan")), 1),
])
def test_pool_descriptor_validation(kw, status):
    rc, h = _create(**kw)
    assert rc == status and not h.value


def test_pool_tensor_bytes():
    d = _desc(num_layers=32, num_blocks=8192, block_size=64, num_kv_heads=8, head_dim=128)
    assert pk.lib().kv_pool_tensor_bytes(ctypes.byref(d)) == 32 * 8192 * 8 * 64 * 128 * 2


def test_rejected_calls_do_not_launch():
    rc, h = _create()
    assert rc == 0 and h.value
    L = pk.lib()
    P = ctypes.c_void_p
    try:
        # append: bad layer, bad dtype, misaligned input, f32 pool rule
        assert L.kv_append(h, 1, P(FAKE), P(FAKE), 1, P(FAKE), 4, None) == 1
        assert L.kv_append(h, 0, P(FAKE), P(FAKE), 2, P(FAKE), 4, None) == 1
        assert L.kv_append(h, 0, P(FAKE + 2), P(FAKE), 1, P(FAKE), 4, None) == 1
        assert L.kv_append(h, 0, P(FAKE), P(FAKE), 1, P(FAKE), 0, None) == 0  # nothing to do
        attn = lambda **k: L.paged_decode_attention(
            P(k.get("q", FAKE)), k.get("qdt", 1), h, k.get("layer", 0), P(FAKE), k.get("mb", 4), P(FAKE),
            k.get("B", 2), k.get("Hq", 8), k.get("maxlen", 64), k.get("scale", 0.1), k.get("split", 0),
            k.get("algo", 0), P(k.get("ws", None)), k.get("wsb", 0), P(FAKE), None)
        assert attn(layer=3) == 1
        assert attn(Hq=7) == 1                  # Hq % Hkv
        assert attn(maxlen=65) == 1             # beyond the table (4 blocks * 16)
        assert attn(qdt=0) == 2                 # q dtype must match a bf16 pool
        assert attn(q=FAKE + 8) == 1            # misaligned q
        assert attn(scale=float("inf")) == 1
        assert attn(algo=9) == 1
        assert attn(split=48) == 1              # not a multiple of 64
        assert attn(B=0) == 0                   # empty batch is a no-op
        # needs a workspace (64 tokens in 64-token splits -> 1 split: none needed);
        # 1024 tokens in 64-token splits need one
        S, NS, ws = pk.ctypes.c_int32(), pk.ctypes.c_int32(), pk.ctypes.c_size_t()
        assert L.paged_decode_plan(h, 2, 8, 1024, 64, ctypes.byref(S), ctypes.byref(NS), ctypes.byref(ws)) == 0
        assert (S.value, NS.value) == (64, 16) and ws.value >= 2 * 8 * 16 * 129 * 4
        assert attn(mb=64, maxlen=1024, split=64) == 3
        assert attn(mb=64, maxlen=1024, split=64, ws=FAKE, wsb=ws.value - 1) == 3
    finally:
        L.kv_pool_destroy(h)


# ------------------------------------------------------------ block manager

def test_block_manager_matches_oracle_slot_mapping():
    rng = np.random.default_rng(0)
    order = rng.permutation(64)
    bm = BlockManager(64, 16, 8, free_order=order)
    lens = [1, 16, 17, 40, 100]
    slots = {}
    for s, L in enumerate(lens):
        bm.add(s)
        slots[s] = bm.grow(s, L)
    bm.check()
    tables = bm.block_tables(range(len(lens))).numpy()
    for s, L in enumerate(lens):
        ref = oracle.slot_mapping(tables, 16, np.full(L, s), np.arange(L))
        assert np.array_equal(slots[s], ref)
    # static workloads: allocation in sequence order = consecutive chunks of the free list
    ch = wl.chunk_tables(__import__("torch").from_numpy(order.astype(np.int32)),
                         __import__("torch").tensor(lens), 16, 8).numpy()
    assert np.array_equal(ch, tables)


def test_block_manager_free_list_conservation_and_pause():
    bm = BlockManager(10, 4, 5)
    bm.add(0)
    bm.add(1)
    bm.grow(0, 9)   # 3 blocks
    bm.grow(1, 12)  # 3 blocks
    assert bm.num_free == 4
    with pytest.raises(OutOfBlocks):
        bm.grow(0, 20)  # would need 5 more blocks, table width 5
    assert bm.lens[0] == 9 and bm.num_free == 4  # unchanged after the refusal
    bm.grow(0, 7)  # 16 tokens -> 4 blocks
    bm.check()
    bm.free_sequence(1)
    assert bm.num_free == 6
    bm.check()
    # waste: at most one partial block per sequence
    held = sum(len(t) for t in bm.tables.values())
    assert held * 4 - sum(bm.lens.values()) < 4 * len(bm.tables)


def test_block_manager_reproduces_paging_diagram():
    with open(os.path.join(GOLDEN, "paging_diagram.json")) as f:
        g = json.load(f)
    # hand out blocks in the order the diagram's requests grew: A1 B2 B3 A4 C5,
    # then a short-lived request takes B6 and finishes, then A7
    bm = BlockManager(9, 1, 9)
    for s in ("A", "B", "C", "D"):
        bm.add(s)
    for s in ("A", "B", "B", "A", "C", "D", "A"):
        bm.grow(s, 1)
    bm.free_sequence("D")
    for name, blocks in g["tables"].items():
        assert [b + 1 for b in bm.tables[name]] == blocks
    assert sorted(b + 1 for b in bm.free) == g["free"]
    bm.check()


def test_prefix_reuse_shares_full_blocks_and_counts_references():
    bm = BlockManager(16, 4, 8)
    prompt = list(range(100, 111))  # 11 tokens: 2 full blocks + 3
    bm.add("a")
    bm.grow("a", len(prompt), token_ids=prompt)
    a_blocks = bm.tables["a"]
    bm.add("b")
    reused = bm.match_prefix("b", prompt + [7, 8])  # same prefix, longer prompt
    assert reused == 8 and bm.tables["b"] == a_blocks[:2]
    assert [bm.ref(x) for x in a_blocks] == [2, 2, 1]
    bm.grow("b", 5, token_ids=prompt[8:] + [7, 8])  # the rest of b's prompt: own blocks
    assert set(bm.tables["b"][2:]).isdisjoint(a_blocks)
    bm.check()
    # a different prompt shares only the blocks whose whole prefix matches
    bm.add("c")
    assert bm.match_prefix("c", prompt[:4] + [0] * 9) == 4
    bm.check()
    bm.free_sequence("a")
    assert [bm.ref(x) for x in a_blocks] == [3 - 1, 1, 0]  # c and b still hold block 0; b holds block 1
    bm.check()


def test_prefix_reuse_never_takes_the_last_prompt_token():
    bm = BlockManager(8, 4, 4)
    ids = [5, 6, 7, 8, 9, 10, 11, 12]  # exactly two full blocks
    bm.add("a")
    bm.grow("a", 8, token_ids=ids)
    bm.add("b")
    assert bm.match_prefix("b", ids) == 4  # the second block holds the last token: recomputed
    bm.check()


def test_freed_blocks_stay_matchable_until_reallocated():
    bm = BlockManager(6, 2, 6)
    ids = [1, 2, 3, 4, 5]
    bm.add("a")
    bm.grow("a", 5, token_ids=ids)  # blocks: [1,2] [3,4] [5]
    cached = bm.tables["a"][:2]
    bm.free_sequence("a")
    assert bm.num_free == 6
    bm.add("b")
    assert bm.match_prefix("b", ids) == 4 and bm.tables["b"] == cached  # revived from the free list
    bm.free_sequence("b")
    # hand out every free block: the cached ones are evicted on reallocation
    bm.add("hog")
    bm.grow("hog", 12)
    bm.free_sequence("hog")
    bm.add("c")
    assert bm.match_prefix("c", ids) == 0
    bm.check()


def test_decode_slots_pause_when_out_of_blocks():
    bm = BlockManager(4, 2, 4)
    for s, n in (("a", 2), ("b", 1), ("c", 4)):
        bm.add(s)
        bm.grow(s, n)
    assert bm.num_free == 0
    slots = bm.decode_slots(["a", "b", "c"])  # a and c need a new block, b has room
    assert slots[0] == -1 and slots[2] == -1 and slots[1] >= 0 and bm.last_paused == 2
    assert bm.lens == {"a": 2, "b": 2, "c": 4}
    bm.free_sequence("b")
    slots = bm.decode_slots(["a", "c"])  # one block freed: a gets it, c still waits
    assert slots[0] >= 0 and slots[1] == -1
    bm.check()


def test_block_manager_random_ops_keep_invariants_and_slots():
    rng = np.random.default_rng(1)
    bs, nb, width = 4, 40, 12
    bm = BlockManager(nb, bs, width, free_order=rng.permutation(nb))
    live, prompts, slot_log = [], {}, {}
    for step in range(400):
        op = rng.integers(0, 5)
        if op == 0 or not live:
            s = "s%d" % step
            bm.add(s)
            live.append(s)
            n = int(rng.integers(1, 20))
            donors = [x for x in live if x in prompts]
            base = prompts[donors[int(rng.integers(0, len(donors)))]][:8] if donors and rng.random() < 0.5 else []
            ids = (base + [int(x) for x in rng.integers(0, 3, n)])[: max(1, n)]
            reused = bm.match_prefix(s, ids)
            try:
                slots = bm.grow(s, len(ids) - reused, token_ids=ids[reused:])
            except OutOfBlocks:
                slots = np.zeros(0, np.int64)
            prompts[s] = ids
            slot_log[s] = {}
            for i, sl in enumerate(slots):
                slot_log[s][reused + i] = int(sl)
        elif op == 1:
            s = live.pop(int(rng.integers(0, len(live))))
            bm.free_sequence(s)
            del slot_log[s]
        elif op == 2:
            s = live[int(rng.integers(0, len(live)))]
            try:
                L = bm.seq_len(s)
                for i, sl in enumerate(bm.grow(s, int(rng.integers(1, 6)))):
                    slot_log[s][L + i] = int(sl)
            except OutOfBlocks:
                pass
        else:
            L0 = {s: bm.seq_len(s) for s in live}
            for s, sl in zip(live, bm.decode_slots(live)):
                if sl >= 0:
                    slot_log[s][L0[s]] = int(sl)
        bm.check()
    # every slot the manager handed out agrees with the oracle's mapping of the final tables
    tables = bm.block_tables(live, width).numpy()
    for i, s in enumerate(live):
        pos = sorted(slot_log[s])
        if pos:
            ref = oracle.slot_mapping(tables, bs, np.full(len(pos), i), np.array(pos))
            assert np.array_equal(ref, [slot_log[s][p] for p in pos])
    # no slot is written by two live sequences (shared blocks are never written again)
    written = [sl for s in live for sl in slot_log[s].values()]
    assert len(written) == len(set(written))
