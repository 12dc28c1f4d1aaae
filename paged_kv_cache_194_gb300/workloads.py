"""Seeded synthetic inputs for paged decode attention.

This module is shared by the tests, the benchmark and the callers of the CPU
oracle.  It only draws numbers -- sequence lengths, a shuffled free list of
pool blocks, query/key/value tensors, per-tensor FP8 scales -- and holds none
of the method's arithmetic (no slot mapping, no gather, no attention, no
quantisation).  Everything is drawn from seeded CPU ``torch.Generator``s, so
every process on every machine sees the same inputs.

The five workloads restate the ones the measurements are quoted on:

1. ``tiny``: 4 sequences of lengths {1, 17, 33, 64}; 2 query heads / 1 KV head;
   head_dim 64; 16-token blocks; a 32-block pool; fp32 q/k/v ~ U(-1, 1); block
   tables are consecutive chunks of a seeded shuffle of the pool; scale 1/8.
2. ``llama``: one Llama-3-8B attention layer ("TensorRT-LLM, in depth",
   First principles: 32 layers, 8 KV heads, grouped-query, head_dim 128) with
   32 query heads; 64 sequences of lengths ~ U[128, 4096]; 16-token blocks;
   BF16 q/k/v ~ N(0, 1); scale 1/sqrt(128); tables from a shuffled free list
   whose pool is 1.25x what the batch needs.
3. ``ragged``: an in-flight batch of 256 sequences, lengths lognormal with
   median 1024 (sigma 1 in log space) clipped to [1, 8192]; 32-token blocks;
   otherwise as ``llama``; 8 decode steps each appending one token per
   sequence (new blocks come from the free list).
4. ``fp8``: 55 sequences at 8192 tokens (the pages' "about 55 concurrent
   requests at a full 8,192-token context"); 64-token blocks; K/V stored as
   FP8 E4M3 with per-tensor scales amax/448 taken over the BF16 N(0, 1) data;
   BF16 q.
5. ``long``: 4 sequences at 131072 tokens; 64-token blocks; BF16; 32 layers in
   one pool (8192 blocks per layer); 2048-token splits.

Two multi-query workloads (several queries per sequence, each attending
causally to the positions up to its own):

6. ``specverify``: the ``llama`` batch verifying k = 4 drafted tokens per
   sequence in one pass ("How does TensorRT-LLM work?", "Speculative
   decoding": guess several tokens, let the model check them together).
7. ``prefill``: 16 sequences whose last 256 prompt tokens arrive as one chunk
   over a cached prefix, total lengths ~ U[1024, 8192] ("How does
   TensorRT-LLM work?", "In-flight batching": long prompts are split into
   chunks mixed with decoding); 32-token blocks.

Convention used throughout: ``seq_lens[b]`` is the number of tokens a decode
step attends over, and the last of them (position ``seq_lens[b] - 1``) is the
token that step appends.  A prefill therefore writes positions
``0 .. seq_lens[b] - 2`` first.  With C queries per sequence the step appends
(and queries) the last C positions, ``seq_lens[b] - C .. seq_lens[b] - 1``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str            # pool storage: "f32" | "bf16" | "fp8"
    in_dtype: str            # appended k/v (and q unless q_dtype is set): "f32" | "bf16"
    scale: float
    num_layers: int = 1
    lens: str = "fixed"      # "fixed" | "uniform" | "lognormal"
    fixed_lens: Tuple[int, ...] = ()
    len_lo: int = 1
    len_hi: int = 1
    median: float = 1.0
    sigma: float = 1.0
    dist: str = "normal"     # "normal" | "uniform"  (value distribution of q/k/v)
    pool_blocks: int = 0     # 0: 1.25x the blocks the batch needs over all steps
    split_tokens: int = 0    # 0: let the library choose
    steps: int = 1           # decode steps (each appends one token per sequence)
    q_dtype: str = ""        # query dtype when it differs from in_dtype
    queries: int = 1         # queries per sequence per step (1 = decode)

    @property
    def query_dtype(self) -> str:
        return self.q_dtype or self.in_dtype

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 4, 2, 1, 64, 16, "f32", "f32", 1.0 / 8.0,
                     lens="fixed", fixed_lens=(1, 17, 33, 64), dist="uniform", pool_blocks=32),
    "llama": Workload("llama", 2, 64, 32, 8, 128, 16, "bf16", "bf16", 1.0 / math.sqrt(128.0),
                      lens="uniform", len_lo=128, len_hi=4096),
    "ragged": Workload("ragged", 3, 256, 32, 8, 128, 32, "bf16", "bf16", 1.0 / math.sqrt(128.0),
                       lens="lognormal", median=1024.0, sigma=1.0, len_lo=1, len_hi=8192, steps=8),
    "fp8": Workload("fp8", 4, 55, 32, 8, 128, 64, "fp8", "bf16", 1.0 / math.sqrt(128.0),
                    lens="fixed", fixed_lens=(8192,) * 55),
    "long": Workload("long", 5, 4, 32, 8, 128, 64, "bf16", "bf16", 1.0 / math.sqrt(128.0),
                     num_layers=32, lens="fixed", fixed_lens=(131072,) * 4, pool_blocks=8192,
                     split_tokens=2048),
    "specverify": Workload("specverify", 2, 64, 32, 8, 128, 16, "bf16", "bf16", 1.0 / math.sqrt(128.0),
                           lens="uniform", len_lo=128, len_hi=4096, queries=4),
    "prefill": Workload("prefill", 7, 16, 32, 8, 128, 32, "bf16", "bf16", 1.0 / math.sqrt(128.0),
                        lens="uniform", len_lo=1024, len_hi=8192, queries=256),
}

# workload order as the measurements list them
ORDER = ["tiny", "llama", "ragged", "fp8", "long"]


def _gen(*key: int) -> torch.Generator:
    """A CPU generator seeded from a tuple of small integers."""
    s = 0x9E3779B9
    for k in key:
        s = (s * 1000003 + int(k) + 1) % (2**61 - 1)
    g = torch.Generator(device="cpu")
    g.manual_seed(s)
    return g


def seq_lens(w: Workload) -> torch.Tensor:
    """Lengths attended by the first decode step, int32 [B]."""
    if w.lens == "fixed":
        return torch.tensor(w.fixed_lens, dtype=torch.int32)
    g = _gen(w.seed, 1)
    if w.lens == "uniform":
        return torch.randint(w.len_lo, w.len_hi + 1, (w.num_seqs,), generator=g, dtype=torch.int64).to(torch.int32)
    if w.lens == "lognormal":
        z = torch.randn(w.num_seqs, generator=g, dtype=torch.float64)
        L = torch.round(torch.exp(math.log(w.median) + w.sigma * z))
        return L.clamp(w.len_lo, w.len_hi).to(torch.int32)
    raise ValueError(w.lens)


def blocks_needed(w: Workload, lens: torch.Tensor) -> int:
    """Blocks the batch occupies after all of its decode steps."""
    final = lens.to(torch.int64) + (w.steps - 1)
    return int(((final + w.block_size - 1) // w.block_size).sum())


def num_pool_blocks(w: Workload, lens: torch.Tensor) -> int:
    if w.pool_blocks:
        return w.pool_blocks
    return int(math.ceil(1.25 * blocks_needed(w, lens)))


def free_list(w: Workload, num_blocks: int) -> torch.Tensor:
    """A seeded shuffle of the pool's block ids (int32)."""
    return torch.randperm(num_blocks, generator=_gen(w.seed, 2)).to(torch.int32)


def chunk_tables(order: torch.Tensor, lens: torch.Tensor, block_size: int,
                 max_blocks: Optional[int] = None) -> torch.Tensor:
    """Consecutive chunks of ``order`` as per-sequence block lists, padded
    with -1.  This is how a seeded shuffle of the pool is handed out to the
    sequences of a static workload (an input, not the product's allocator)."""
    nb = [(int(L) + block_size - 1) // block_size for L in lens]
    width = max_blocks if max_blocks is not None else max(1, max(nb))
    t = torch.full((len(nb), width), -1, dtype=torch.int32)
    pos = 0
    for b, n in enumerate(nb):
        t[b, :n] = order[pos:pos + n]
        pos += n
    if pos > order.numel():
        raise ValueError("pool too small for the batch")
    return t


def query(w: Workload, layer: int = 0, step: int = 0) -> torch.Tensor:
    """q [B, Hq, D] (decode) or [B, C, Hq, D] (C = w.queries > 1) in the
    workload's query dtype (CPU)."""
    if w.queries > 1:
        g = _gen(w.seed, 6, layer, step)
        shape = (w.num_seqs, w.queries, w.num_q_heads, w.head_dim)
    else:
        g = _gen(w.seed, 3, layer, step)
        shape = (w.num_seqs, w.num_q_heads, w.head_dim)
    return _draw(w, shape, g, w.query_dtype)


def _draw(w: Workload, shape, g: torch.Generator, dtype: str = "") -> torch.Tensor:
    if w.dist == "uniform":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    else:
        x = torch.randn(shape, generator=g, dtype=torch.float32)
    return x.to(DTYPES[dtype or w.in_dtype])


def seq_kv(w: Workload, layer: int, b: int, n_tokens: int, start: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """K and V rows of sequence b for positions [start, start + n_tokens),
    each [n, Hkv, D] in the input dtype (CPU).  Rows are drawn in chunks of
    256 positions, each chunk from its own generator, so any window can be
    regenerated without drawing the whole sequence."""
    C = 256
    ks, vs = [], []
    first, last = start // C, (start + n_tokens - 1) // C if n_tokens > 0 else start // C - 1
    for c in range(first, last + 1):
        kc = _draw(w, (C, w.num_kv_heads, w.head_dim), _gen(w.seed, 4, layer, b, c))
        vc = _draw(w, (C, w.num_kv_heads, w.head_dim), _gen(w.seed, 5, layer, b, c))
        lo = max(start, c * C) - c * C
        hi = min(start + n_tokens, (c + 1) * C) - c * C
        ks.append(kc[lo:hi])
        vs.append(vc[lo:hi])
    if not ks:
        e = torch.empty((0, w.num_kv_heads, w.head_dim), dtype=DTYPES[w.in_dtype])
        return e, e.clone()
    return torch.cat(ks), torch.cat(vs)


def fp8_scales(w: Workload, lens: torch.Tensor) -> Tuple[float, float]:
    """Per-tensor (k_scale, v_scale) = amax / 448 over all K (resp. V) values
    the workload ever stores, in float32 arithmetic."""
    ka = torch.zeros((), dtype=torch.float32)
    va = torch.zeros((), dtype=torch.float32)
    for layer in range(w.num_layers):
        for b in range(w.num_seqs):
            n = int(lens[b]) + w.steps - 1
            if n <= 0:
                continue
            k, v = seq_kv(w, layer, b, n)
            ka = torch.maximum(ka, k.float().abs().max())
            va = torch.maximum(va, v.float().abs().max())
    four48 = torch.tensor(448.0, dtype=torch.float32)
    return float(ka / four48), float(va / four48)


@dataclass
class Instance:
    """A drawn workload: lengths, pool size, free list and static tables."""
    w: Workload
    lens: torch.Tensor
    num_blocks: int
    order: torch.Tensor
    tables: torch.Tensor          # consecutive chunks of `order` for `lens`
    max_blocks: int
    k_scale: float = 1.0
    v_scale: float = 1.0


def instance(w: Workload, lens: Optional[torch.Tensor] = None, with_scales: bool = True) -> Instance:
    lens = seq_lens(w) if lens is None else lens
    nb = num_pool_blocks(w, lens)
    order = free_list(w, nb)
    final = lens.to(torch.int64) + (w.steps - 1)
    max_blocks = int(((final + w.block_size - 1) // w.block_size).max()) if len(lens) else 1
    max_blocks = max(1, max_blocks)
    tables = chunk_tables(order, lens, w.block_size, max_blocks)
    ks, vs = (1.0, 1.0)
    if w.kv_dtype == "fp8" and with_scales:
        ks, vs = fp8_scales(w, lens)
    return Instance(w, lens, nb, order, tables, max_blocks, ks, vs)
