"""A decode batch resident on the GPU, driven through the library's C ABI.

Lifecycle of one batch (the in-flight decode step of "How does TensorRT-LLM
work?", sections "In-flight batching" and "The full journey of one request",
restricted to the attention layer):

* prefill: the host block manager hands out blocks from the free list and
  returns the slots of positions 0 .. seq_lens[b]-2; ``kv_append`` writes the
  rows there;
* decode step: one more slot per sequence (a new block when the last one is
  full), ``kv_append`` of the step's new K/V row, then
  ``paged_decode_attention`` over seq_lens[b] tokens.
* with C = w.queries > 1 the prefill stops at seq_lens[b] - C and a step
  appends the last C positions of every sequence (drafted tokens to verify,
  or a prompt chunk), then runs ``paged_multi_query_attention``.

Inputs come from ``workloads`` (seeded, synthetic).  Nothing here computes
attention or conversions itself.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import binding as pk
from . import workloads as wl
from .block_manager import BlockManager


class DecodeBatch:
    def __init__(self, inst: wl.Instance, device: str = "cuda", layers: Optional[Sequence[int]] = None,
                 cpu_layers: Optional[Sequence[int]] = None, fill_byte: Optional[int] = None,
                 chunk_tokens: int = 1 << 16):
        """layers: the pool layers to fill (default: all).  cpu_layers: layers
        whose rows are drawn from the seeded CPU generators (the oracle can
        regenerate them); the other filled layers draw N(0, 1) on the device
        from a seeded CUDA generator (used for the 32-layer long-context pool,
        whose CPU draw would take minutes)."""
        w = inst.w
        self.inst, self.w, self.device = inst, w, device
        self.B = w.num_seqs
        self.layers = list(range(w.num_layers)) if layers is None else list(layers)
        self.cpu_layers = set(self.layers if cpu_layers is None else cpu_layers)
        self.pool = pk.KVPool(w.num_layers, inst.num_blocks, w.block_size, w.num_kv_heads, w.head_dim,
                              w.kv_dtype, inst.k_scale, inst.v_scale, device=device, fill=fill_byte)
        self.bm = BlockManager(inst.num_blocks, w.block_size, inst.max_blocks, free_order=inst.order.tolist())
        self.lens = [int(x) for x in inst.lens]
        self.seq_ids = list(range(self.B))
        for b in self.seq_ids:
            self.bm.add(b)
        self.C = max(1, w.queries)
        # prefill slots (positions 0 .. L-C-1), identical for every layer
        self.prefill_slots: Dict[int, np.ndarray] = {}
        for b in self.seq_ids:
            n = max(0, self.lens[b] - self.C)
            self.prefill_slots[b] = self.bm.grow(b, n) if n else np.zeros(0, np.int64)
        self._prefill(chunk_tokens)
        self.step = 0

    # ----------------------------------------------------------- prefill
    def _prefill(self, chunk_tokens: int):
        w = self.w
        in_dt = wl.DTYPES[w.in_dtype]
        for layer in self.layers:
            if layer in self.cpu_layers:
                ks, vs, ss, count = [], [], [], 0
                for b in self.seq_ids:
                    n = len(self.prefill_slots[b])
                    if n == 0:
                        continue
                    k, v = wl.seq_kv(w, layer, b, n)
                    ks.append(k)
                    vs.append(v)
                    ss.append(torch.from_numpy(self.prefill_slots[b]))
                    count += n
                    if count >= chunk_tokens:
                        self._append_cat(layer, ks, vs, ss)
                        ks, vs, ss, count = [], [], [], 0
                if ks:
                    self._append_cat(layer, ks, vs, ss)
            else:
                g = torch.Generator(device=self.device)
                g.manual_seed(1_000_003 * w.seed + layer)
                all_slots = torch.from_numpy(np.concatenate([self.prefill_slots[b] for b in self.seq_ids]))
                for i in range(0, all_slots.numel(), chunk_tokens):
                    sl = all_slots[i:i + chunk_tokens].to(self.device)
                    shape = (sl.numel(), w.num_kv_heads, w.head_dim)
                    k = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32).to(in_dt)
                    v = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32).to(in_dt)
                    pk.kv_append(self.pool, layer, k, v, sl)
        torch.cuda.synchronize()

    def _append_cat(self, layer, ks, vs, ss):
        k = torch.cat(ks).to(self.device)
        v = torch.cat(vs).to(self.device)
        s = torch.cat(ss).to(self.device)
        pk.kv_append(self.pool, layer, k, v, s)

    # -------------------------------------------------------------- step
    def next_token_slots(self) -> np.ndarray:
        """Slots of each sequence's next token (the last of its seq_lens);
        sequences that started empty stay empty and get slot -1.  With C > 1:
        [B * C] slots of positions L-C .. L-1 (-1 where the position is
        negative)."""
        if self.C > 1:
            slots = np.full((self.B, self.C), -1, dtype=np.int64)
            for b in self.seq_ids:
                n = min(self.C, self.lens[b])
                if n > 0:
                    slots[b, self.C - n:] = self.bm.grow(b, n)
            return slots.reshape(-1)
        slots = np.full(self.B, -1, dtype=np.int64)
        active = [b for b in self.seq_ids if self.lens[b] > 0]
        if active:
            slots[active] = self.bm.decode_slots(active)
        return slots

    def step_inputs(self, layer: int, step: int = 0):
        """Host tensors of a decode step: q, k_new, v_new (the rows of
        position seq_lens[b] - 1 + step; zeros for empty sequences).  With
        C > 1: q [B, C, Hq, D] and the rows of positions L-C .. L-1, [B*C, Hkv, D]
        (zeros at negative positions)."""
        w = self.w
        q = wl.query(w, layer, step)
        if self.C > 1:
            ks, vs = [], []
            z = torch.zeros((1, w.num_kv_heads, w.head_dim), dtype=wl.DTYPES[w.in_dtype])
            for b in self.seq_ids:
                L = self.lens[b]
                n = min(self.C, L)
                ks += [z] * (self.C - n)
                vs += [z] * (self.C - n)
                if n > 0:
                    k, v = wl.seq_kv(w, layer, b, n, start=L - n)
                    ks.append(k)
                    vs.append(v)
            return q, torch.cat(ks), torch.cat(vs)
        ks, vs = [], []
        for b in self.seq_ids:
            if self.lens[b] > 0:
                k, v = wl.seq_kv(w, layer, b, 1, start=self.lens[b] + step - 1)
            else:
                k = torch.zeros((1, w.num_kv_heads, w.head_dim), dtype=wl.DTYPES[w.in_dtype])
                v = k
            ks.append(k)
            vs.append(v)
        return q, torch.cat(ks), torch.cat(vs)

    def tables(self) -> torch.Tensor:
        return self.bm.block_tables(self.seq_ids, self.inst.max_blocks)

    def seq_lens(self) -> torch.Tensor:
        return self.bm.seq_lens(self.seq_ids)
