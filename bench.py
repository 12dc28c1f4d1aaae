"""Benchmark: paged decode attention KV GB/s and tokens/s on GB300.

One step = one pass of the decode hot path over the batch: the host block
manager's slot for each sequence's newest token, the append of that token's
K/V row, then attention (split-K + log-sum-exp combine) over seq_lens[b]
tokens.  With the tensor-core design the append runs inside the attention
launch (``paged_decode_append_attention``, one launch per layer-step);
``--unfused`` times ``kv_append`` + ``paged_decode_attention`` instead.  Every step re-appends the same positions, so the bytes
per step are fixed.  Default workload: one Llama-3-8B attention layer, 64
sequences with lengths U[128, 4096], 32 query / 8 KV heads, head_dim 128,
16-token blocks, BF16.  KV per step (~0.56 GB) exceeds the 129 MB L2, so no
flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--algo auto|simt|mma|tc] [--split S] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the only reference this method has).
Multi-GPU (torchrun): every rank runs its own replica of the batch (weak
scaling, no data-path collective); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s and tokens/s (1 GB300) vs HBM roofline"
LAYERS = 32  # Llama-3-8B layers, for the per-output-token figure


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak():
    """bf16 dense tensor peak (TFLOP/s): the measured cuBLAS burst figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def _profile_traffic(kernel_tag: str, src_hash: str):
    """DRAM bytes per launch recorded by an ncu capture in profiles/, if the
    kernel source has not changed since (same sha256)."""
    d = os.path.join(ROOT, "profiles")
    if not os.path.isdir(d):
        return None
    for fn in sorted(os.listdir(d)):
        if not fn.endswith(".md"):
            continue
        txt = open(os.path.join(d, fn)).read()
        m = re.search(r"traffic_bytes_per_launch\[%s\]:\s*([0-9.eE+]+)\s+source_sha256:\s*([0-9a-f]+)"
                      % re.escape(kernel_tag), txt)
        if m and m.group(2) == src_hash:
            return float(m.group(1))
    return None


KERNEL_SOURCES = {"simt": ("decode_simt.cu", "device_common.cuh", "pkv_internal.h"),
                  "mma": ("decode_mma.cuh", "decode_mma.cu", "decode_mma_bf16.cu", "decode_mma_fp8.cu",
                          "device_common.cuh", "pkv_internal.h"),
                  "tc": ("attention_tc.cu", "tc_common.cuh", "device_common.cuh", "pkv_internal.h")}


def kernel_hash(algo: str) -> str:
    """sha256 (first 16 hex digits) of the sources of one kernel design."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_194_gb300", "csrc")
    for fn in KERNEL_SOURCES[algo]:
        h.update(open(os.path.join(csrc, fn), "rb").read())
    return h.hexdigest()[:16]


class Clocks:
    """nvidia-smi sampler (200 ms) for the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "pkv_clocks_%d.csv" % os.getpid())

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def mark(self):
        return time.time()

    def stop(self, t_begin, t_end):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        # rows are ~200 ms apart from t0; keep those inside [t_begin, t_end] (at least one)
        n = len(rows)
        span = max(1e-9, (time.time() - self.t0))
        stamps = [self.t0 + span * (i + 0.5) / n for i in range(n)]
        inside = [r for r, s in zip(rows, stamps) if t_begin <= s <= t_end]
        if not inside:
            best = min(range(n), key=lambda i: abs(stamps[i] - 0.5 * (t_begin + t_end)))
            inside = [rows[best]]
        sm = sorted(float(r[1]) for r in inside if r[1].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None,
                "sm_max_mhz": float(inside[0][2]) if inside[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(inside)}


def query_chunks(C: int, gh: int, algo: str, kv_dtype: str) -> int:
    """Attention launches per call: query chunks of at most 64 rows per KV
    head (tensor-core design) or a power of two of rows the SIMT design holds."""
    if C <= 1 or algo == "tc":
        return 1
    if algo == "mma":
        cq = max(1, 64 // gh)
    else:
        rows = {"f32": 16, "bf16": 8, "fp8": 4}[kv_dtype]
        cq = 1
        while cq * 2 * gh <= rows and cq * 2 <= C:
            cq *= 2
    n, c0 = 0, 0
    while c0 < C:
        c0 += min(cq, C - c0)
        n += 1
    return n


def workload_bytes(w, lens):
    import torch
    kvb = {"f32": 4, "bf16": 2, "fp8": 1}[w.kv_dtype]
    qb = 4 if w.query_dtype == "f32" else 2
    sum_len = int(lens.sum())
    kv = sum_len * w.num_kv_heads * w.head_dim * 2 * kvb
    return sum_len, kv, qb, kvb


def run_ours(args):
    import torch
    import torch.distributed as dist

    from paged_kv_cache_194_gb300 import binding as pk
    from paged_kv_cache_194_gb300 import replicas
    from paged_kv_cache_194_gb300 import workloads as wl
    from paged_kv_cache_194_gb300.decode import DecodeBatch

    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    pk.lib()
    w = replicas.rank_workload(wl.WORKLOADS[args.workload], rank)
    split = w.split_tokens if args.split is None else args.split
    inst = wl.instance(w)
    layers = list(range(w.num_layers))
    # one layer drawn on the CPU (the oracle baseline regenerates it); the
    # rest of a multi-layer pool is drawn on the device
    batch = DecodeBatch(inst, cpu_layers=[0])
    dev = torch.device("cuda", local)
    slots_h = batch.next_token_slots()
    inputs_h = [batch.step_inputs(l) for l in layers]  # (q, k_new, v_new) per layer
    tables_h, lens_h = batch.tables(), batch.seq_lens()
    max_len = int(lens_h.max())
    qs = [x[0].to(dev) for x in inputs_h]
    kns = [x[1].to(dev) for x in inputs_h]
    vns = [x[2].to(dev) for x in inputs_h]
    slots = torch.from_numpy(slots_h).to(dev)
    tables, lens = tables_h.to(dev), lens_h.to(dev)
    out = torch.empty_like(qs[0])
    C = max(1, w.queries)  # queries per sequence (1 = decode)
    if C > 1:
        S, NS, wsb = pk.multi_query_plan(batch.pool, w.num_seqs, C, w.num_q_heads, max_len, split)
    else:
        S, NS, wsb = pk.decode_plan(batch.pool, w.num_seqs, w.num_q_heads, max_len, split)
    algo = (pk.multi_query_algo(batch.pool, C, w.num_q_heads, split, args.algo) if C > 1
            else pk.decode_algo(batch.pool, w.num_q_heads, args.algo))
    fused = (not args.unfused) and C == 1 and algo == "mma" and w.group <= 8
    rows = C * (w.num_q_heads // w.num_kv_heads)  # query rows per KV head
    # (the tcgen05 design balances tiles only when its grid would leave CTA slots idle)
    tc_bal = rows <= 128 and w.num_seqs * w.num_kv_heads < 2 * torch.cuda.get_device_properties(dev).multi_processor_count
    schedule = ("one CTA per 128 query rows" if algo == "tc" and not tc_bal else
                "balanced" if (algo in ("mma", "tc") and split == 0) else "fixed splits")
    work = torch.zeros(max(wsb, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def attend(l):
        if C > 1:
            pk.paged_multi_query_attention(qs[l], batch.pool, l, tables, lens, max_len, w.scale, out=out,
                                           workspace=work, split_tokens=split, algo=args.algo, stream=stream)
        else:
            pk.paged_decode_attention(qs[l], batch.pool, l, tables, lens, max_len, w.scale, out=out, workspace=work,
                                      split_tokens=split, algo=args.algo, stream=stream)

    def fused_step(l):
        pk.paged_decode_append_attention(qs[l], kns[l], vns[l], batch.pool, l, tables, lens, max_len, w.scale,
                                         out=out, workspace=work, split_tokens=split, algo=args.algo, stream=stream)

    def step():
        for l in layers:
            if fused:
                fused_step(l)
            else:
                pk.kv_append(batch.pool, l, kns[l], vns[l], slots, stream)
                attend(l)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if batch.pool.errors():
        raise RuntimeError("device error bits %d" % batch.pool.errors())

    # ---- timed region: K steps, events on the launching stream
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    clocks = Clocks(vis.split(",")[local] if vis else str(local))
    clocks.start()
    time.sleep(0.3)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The fused step is one launch per layer-step: its average launch duration
    # is the timed region over the launches, back to back as a decode loop
    # issues them (an event pair around every launch would put a gap between
    # launches).  The two-launch step brackets each attention call with events.
    att = [] if fused else [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                            for _ in range(args.steps * len(layers))]
    t_begin = time.time()
    ev0.record(stream)
    i = 0
    for _ in range(args.steps):
        for l in layers:
            if fused:
                fused_step(l)
            else:
                pk.kv_append(batch.pool, l, kns[l], vns[l], slots, stream)
                att[i][0].record(stream)
                attend(l)
                att[i][1].record(stream)
            i += 1
    ev1.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    if ws > 1:
        dist.barrier()
    clk = clocks.stop(t_begin, t_end)
    ms_total = replicas.max_over_ranks(ev0.elapsed_time(ev1), dev)
    att_ms = (ms_total / (args.steps * len(layers)) if fused else
              sum(a.elapsed_time(b) for a, b in att) / len(att))
    ms_step = ms_total / args.steps

    sum_len, kv_layer, qb, kvb = workload_bytes(w, inst.lens)
    kv_bytes = kv_layer * len(layers)
    all_kv_bytes = replicas.sum_over_ranks(kv_bytes, dev)
    all_len = replicas.sum_over_ranks(sum_len, dev)
    B, Hq, Hkv, D = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    # algorithmic bytes of one attention call (one layer)
    blocks_read = int(((inst.lens.long() + w.block_size - 1) // w.block_size).sum())
    combine = schedule == "fixed splits" and NS > 1
    part = 0
    if combine:
        nsplit = int(((inst.lens.long() + S - 1) // S).sum())
        part = 2 * nsplit * C * Hq * (D + 1) * 4  # partials written then read
    # algorithmic bytes: every KV byte once, q read and out written once
    att_bytes = kv_layer + B * C * Hq * D * qb * 2 + blocks_read * 4 + B * 4 + part
    if fused:  # the new rows: read in the input dtype, written in the pool's
        att_bytes += B * Hkv * D * 2 * ({"f32": 4, "bf16": 2}[w.in_dtype] + kvb)
    # multiply-adds of QK^T and PV: query c of sequence b sees L_b - C + c + 1 tokens
    Lq = inst.lens.long()
    seen = sum(int(max(0, L - C + c + 1)) for L in Lq.tolist() for c in range(C))
    att_flops = 4 * D * Hq * seen
    value = all_kv_bytes / (ms_step * 1e-3) / 1e9
    achieved = att_bytes / (att_ms * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    traffic = _profile_traffic("%s/%s/%s" % (args.workload, algo, w.kv_dtype), kernel_hash(algo))
    chunks = query_chunks(C, Hq // Hkv, algo, w.kv_dtype)
    launches = args.steps * len(layers) * ((0 if fused else 1) + chunks * (2 if combine else 1))

    # ---- end to end through the public API: pinned host buffers in, result out
    pin = lambda t: t.pin_memory()
    hin = [[pin(t) for t in x] for x in inputs_h]
    hs_, ht_, hl_ = pin(torch.from_numpy(slots_h)), pin(tables_h), pin(lens_h)
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    e2e_steps = max(1, min(args.steps, max(1, 2000 // len(layers))))
    h2d = sum(t.numel() * t.element_size() for x in hin for t in x) + sum(
        t.numel() * t.element_size() for t in ((ht_, hl_) if fused else (hs_, ht_, hl_)))
    d2h = hout.numel() * hout.element_size()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        for l in layers:
            qs[l].copy_(hin[l][0], non_blocking=True)
            kns[l].copy_(hin[l][1], non_blocking=True)
            vns[l].copy_(hin[l][2], non_blocking=True)
        if not fused:  # the fused launch takes each new token's slot from the table
            slots.copy_(hs_, non_blocking=True)
        tables.copy_(ht_, non_blocking=True)
        lens.copy_(hl_, non_blocking=True)
        step()
        hout.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_s = replicas.max_over_ranks((time.perf_counter() - t0) / e2e_steps, dev)
    e2e_value = all_kv_bytes / e2e_s / 1e9

    # the bound: HBM unless the call's flops per algorithmic byte exceed the
    # ridge point of the measured peaks (tensor peak / HBM peak)
    tpeak, tpeak_kind = _tensor_peak()
    tflops = att_flops / (att_ms * 1e-3) / 1e12
    tensor_bound = att_flops / att_bytes > tpeak * 1e12 / (peak * 1e9)
    roof = {"bound": "tensor" if tensor_bound else "hbm",
            "achieved": round(tflops, 2) if tensor_bound else round(achieved, 1),
            "peak": tpeak if tensor_bound else peak, "unit": "TFLOP/s" if tensor_bound else "GB/s",
            "frac": round((tflops / tpeak) if tensor_bound else (achieved / peak), 4),
            "traffic": traffic,
            "kernel": "%s call (%s%s)" % ("paged_decode_append_attention" if fused else
                                          "paged_multi_query_attention" if C > 1 else "paged_decode_attention",
                                          "attention_tc_kernel" if algo == "tc" else "decode_%s_kernel" % algo,
                                          " + combine" if combine else ""),
            "ms_per_launch": round(att_ms, 5), "bytes_per_launch": att_bytes, "flops_per_launch": att_flops,
            "hbm_gbs": round(achieved, 1), "hbm_frac": round(achieved / peak, 4), "tflops": round(tflops, 2),
            "kernel_launches_per_call": chunks * (2 if combine else 1),
            "peak_kind": ("%s (MEASURED_PEAKS.json %s)" % (tpeak_kind if tensor_bound else peak_kind,
                                                          "bf16_tflops" if tensor_bound else "hbm_gbs"))}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.kv_dtype, "data": "synthetic",
        "tokens_per_s": round(all_len * len(layers) / (ms_step * 1e-3), 1),
        "decode_tokens_per_s_32_layers": round(ws * B * C / (ms_step * 1e-3 * LAYERS / len(layers)), 1),
        "config": {"workload": "%s: %d seqs, lens %s, %dq/%dkv heads, head_dim %d, block %d, %s KV%s%s"
                   % (w.name, B, _lens_desc(w), Hq, Hkv, D, w.block_size, w.kv_dtype,
                      ", %d layers per step" % len(layers) if len(layers) > 1 else "",
                      ", %d causal queries per sequence (the last %d positions)" % (C, C) if C > 1 else ""),
                   "queries_per_seq": C,
                   "step": ("append fused into the attention launch" if fused else
                            "kv_append launch + attention launch"),
                   "sum_seq_len": sum_len, "kv_bytes_per_step": kv_bytes,
                   "split_tokens": S if schedule == "fixed splits" else None,
                   "num_splits": NS if schedule == "fixed splits" else None, "schedule": schedule, "algo": algo,
                   "parallelism": "replica per GPU" if ws > 1 else "1 GPU",
                   "l2": "inputs exceed L2 (%.0f MB KV per layer vs 129 MB L2); no flush" % (kv_layer / 1e6)},
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 4), "steps": e2e_steps},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inst, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _lens_desc(w):
    if w.lens == "uniform":
        return "U[%d,%d]" % (w.len_lo, w.len_hi)
    if w.lens == "lognormal":
        return "lognormal(median %g, sigma %g) clipped [%d,%d]" % (w.median, w.sigma, w.len_lo, w.len_hi)
    return "fixed %s" % (w.fixed_lens[0] if len(set(w.fixed_lens)) == 1 else list(w.fixed_lens))


def _oracle_sample(w, inst, seqs):
    import numpy as np
    import oracle
    tables = inst.tables.numpy()
    pool = oracle.OraclePool(1, inst.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype,
                             inst.k_scale, inst.v_scale)
    from paged_kv_cache_194_gb300 import workloads as wl
    for b in seqs:
        L = int(inst.lens[b])
        k, v = wl.seq_kv(w, 0, b, L)
        oracle.kv_append(pool, 0, k, v, w.in_dtype, oracle.slot_mapping(tables, w.block_size, np.full(L, b), np.arange(L)))
    q = wl.query(w)[list(seqs)]
    sub_t = tables[list(seqs)]
    sub_l = inst.lens.numpy()[list(seqs)]
    return pool, q, sub_t, sub_l


def _oracle_attend(w, pool, q, t, l, window=None, threads=0):
    """The oracle's attention for the workload's query shape; returns the
    thread count it used."""
    import oracle
    if w.queries > 1:
        return oracle.paged_attention_mq(q, w.query_dtype, pool, 0, t, l, w.scale, threads=threads,
                                         return_threads=True)[2]
    kw = {} if window is None else {"window": window}
    return oracle.paged_attention(q, w.query_dtype, pool, 0, t, l, w.scale, threads=threads, return_threads=True,
                                  **kw)[2]


def _kv_bytes(w, tokens):
    return tokens * w.num_kv_heads * w.head_dim * 2 * {"f32": 4, "bf16": 2, "fp8": 1}[w.kv_dtype]


def cpu_baseline(w, inst, budget_s=15.0):
    """Time the fp64 oracle's attention over the batch (as it stands, all host
    cores) for about budget_s seconds; report KV GB/s of the sample."""
    import oracle
    seqs = list(range(w.num_seqs))
    pool, q, t, l = _oracle_sample(w, inst, seqs)
    kv_bytes = _kv_bytes(w, int(l.sum()))
    reps, spent, threads = 0, 0.0, 0
    while spent < budget_s and reps < 50:
        t0 = time.perf_counter()
        threads = _oracle_attend(w, pool, q, t, l)
        spent += time.perf_counter() - t0
        reps += 1
    # one thread, on the first sequence only (a few seconds)
    one = [0]
    t0 = time.perf_counter()
    _oracle_attend(w, pool, q[one], t[one], l[one], threads=1)
    one_s = time.perf_counter() - t0
    return {"value": round(reps * kv_bytes / spent / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "value_1_thread": round(_kv_bytes(w, int(l[0])) / one_s / 1e9, 4),
            "sample": "fp64 oracle attention over the whole %s batch (%d seqs, %d tokens), %d repetitions, %.1f s; "
                      "1-thread figure: sequence 0 (%d tokens) once"
                      % (w.name, len(seqs), int(l.sum()), reps, spent, int(l[0]))}


def run_reference(args):
    """The oracle as the reference arm (rank 0 only): each step attends over a
    bounded sample of the batch, sized so that warm-up + steps take about
    --ref-budget seconds."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_194_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    inst = wl.instance(w)
    lens = [int(x) for x in inst.lens]
    # calibrate on sequence 0
    pool, q, t, l = _oracle_sample(w, inst, [0])
    t0 = time.perf_counter()
    _oracle_attend(w, pool, q, t, l)
    per_token = (time.perf_counter() - t0) / max(1, lens[0])
    want = max(16, int(args.ref_budget / (args.steps + args.warmup) / per_token))
    seqs, window, acc = [], 2**31 - 1, 0
    for b, L in enumerate(lens):
        if acc + L > want:
            break
        seqs.append(b)
        acc += L
    if not seqs:
        seqs, window, acc = [0], min(lens[0], want), min(lens[0], want)
        if w.queries > 1:  # no window for multi-query: the whole first sequence
            window, acc = 2**31 - 1, lens[0]
    pool, q, t, l = _oracle_sample(w, inst, seqs)
    kv_bytes = _kv_bytes(w, acc)
    for _ in range(args.warmup):
        _oracle_attend(w, pool, q, t, l, window=(0, window))
    threads = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        threads = _oracle_attend(w, pool, q, t, l, window=(0, window))
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = kv_bytes / dt / 1e9
    sample = ("first %d of %d sequences (%d tokens) of the %s batch per step" % (len(seqs), w.num_seqs, acc, w.name)
              if window == 2**31 - 1 else "first %d tokens of sequence 0 of the %s batch per step" % (acc, w.name))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "%s; sample: %s" % (w.name, sample)},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="llama")
    ap.add_argument("--algo", default="auto", choices=["auto", "simt", "mma", "tc"])
    ap.add_argument("--split", type=int, default=None,
                    help="fixed split size in tokens; 0 = balanced schedule; default: the workload's recipe")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-budget", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unfused", action="store_true", help="time kv_append + attention as two launches")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
