"""Helpers for GPU-vs-oracle parity tests.

The oracle side never reads anything the CUDA path produced: it regenerates
each sequence's rows from the seeded generators, computes its own slot
mapping from the block tables, appends with its own encoders and attends in
fp64.  Tables and lengths are host inputs shared by both sides.
"""
from __future__ import annotations

import math
from typing import Sequence

import numpy as np
import torch

import oracle
from paged_kv_cache_194_gb300 import workloads as wl

# elementwise |gpu - ref| <= tol + tol * |ref|
TOL = {"bf16": 1e-2, "fp8": 2e-2, "f32": 1e-4}


def oracle_reference(w: wl.Workload, k_scale: float, v_scale: float, layer: int, q: torch.Tensor,
                     tables: torch.Tensor, lens: Sequence[int], seqs: Sequence[int], rows_fn=None):
    """fp64 oracle output for the listed sequences ([len(seqs), Hq, D]).

    Only the blocks of the listed sequences are materialised: their ids are
    relabelled 0..n-1 in table order (the result does not depend on block
    placement).  rows_fn(b, L) -> (k, v) supplies a sequence's rows when they
    do not come from the workload generator."""
    tables = tables.numpy() if isinstance(tables, torch.Tensor) else np.asarray(tables)
    nblk = [(int(lens[b]) + w.block_size - 1) // w.block_size for b in seqs]
    total = max(1, sum(nblk))
    width = max(1, max(nblk))
    sub = np.full((len(seqs), width), -1, dtype=np.int32)
    pos = 0
    for i, (b, n) in enumerate(zip(seqs, nblk)):
        sub[i, :n] = np.arange(pos, pos + n, dtype=np.int32)
        pos += n
    pool = oracle.OraclePool(1, total, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, k_scale, v_scale)
    for i, b in enumerate(seqs):
        L = int(lens[b])
        if L == 0:
            continue
        k, v = rows_fn(b, L) if rows_fn is not None else wl.seq_kv(w, layer, b, L)
        slots = oracle.slot_mapping(sub, w.block_size, np.full(L, i), np.arange(L))
        oracle.kv_append(pool, 0, k, v, w.in_dtype, slots)
    qs = q[list(seqs)]
    sl = np.array([int(lens[b]) for b in seqs], dtype=np.int32)
    out, lse = oracle.paged_attention(qs, w.query_dtype, pool, 0, sub, sl, w.scale)
    return out, lse


def compare(gpu: torch.Tensor, ref: np.ndarray, tol: float, what: str = ""):
    g = gpu.detach().to(torch.float64).cpu().numpy()
    err = np.abs(g - ref)
    bound = tol + tol * np.abs(ref)
    bad = ~(err <= bound)  # NaN counts as a mismatch
    big = np.abs(ref) > 1e-3
    max_abs = float(err.max()) if err.size else 0.0
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d/%d elements outside tol %g (max abs %.3g, max rel %.3g); first %s"
                             % (what, int(bad.sum()), bad.size, tol, max_abs, max_rel, idx.tolist()))
    assert np.isfinite(g).all(), what + ": non-finite output"
    return max_abs, max_rel


def oracle_reference_mq(w: wl.Workload, k_scale: float, v_scale: float, layer: int, q: torch.Tensor,
                        tables, lens: Sequence[int], seqs: Sequence[int]):
    """fp64 oracle for multi-query attention of the listed sequences
    ([len(seqs), C, Hq, D]); rows from the workload generator."""
    tables = tables.numpy() if isinstance(tables, torch.Tensor) else np.asarray(tables)
    nblk = [(int(lens[b]) + w.block_size - 1) // w.block_size for b in seqs]
    total, width = max(1, sum(nblk)), max(1, max(nblk))
    sub = np.full((len(seqs), width), -1, dtype=np.int32)
    pos = 0
    for i, n in enumerate(nblk):
        sub[i, :n] = np.arange(pos, pos + n, dtype=np.int32)
        pos += n
    pool = oracle.OraclePool(1, total, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, k_scale, v_scale)
    for i, b in enumerate(seqs):
        L = int(lens[b])
        if L == 0:
            continue
        k, v = wl.seq_kv(w, layer, b, L)
        oracle.kv_append(pool, 0, k, v, w.in_dtype, oracle.slot_mapping(sub, w.block_size, np.full(L, i), np.arange(L)))
    sl = np.array([int(lens[b]) for b in seqs], dtype=np.int32)
    return oracle.paged_attention_mq(q[list(seqs)], w.query_dtype, pool, 0, sub, sl, w.scale)
