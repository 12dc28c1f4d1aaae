// Paged attention over the KV pool, tensor-core design (BF16 and FP8-E4M3
// pools, head_dim 128), for one or several queries per sequence.
//
// "How does TensorRT-LLM work?", "Custom attention kernels": one kernel does
// the whole attention step and keeps the intermediate scores on chip.
// "Introduction to TensorRT-LLM", figure "TensorRT-LLM Acceleration Stack":
// Flash-Decoding splits the key/value length across CTAs and merges the
// pieces by their log-sum-exp.
//
// Query rows.  A CTA serves one KV head of one sequence and the NQ query rows
// that share it: gh query heads (grouped-query attention) times C queries of
// the sequence, row n = c * gh + g.  C = 1 is decode; C > 1 verifies drafted
// tokens or processes a prompt chunk: the queries sit at the last C positions
// of the visible length L and query c sees positions < L - C + c + 1.  NQ is
// the template bound (1, 2, 4, ..., 64); the real row count may be smaller
// (the rest is zero padding).  Longer query lists are served by several
// launches (the host splits them).
//
// Work is a list of tiles (64 tokens for BF16, 128 for FP8) of (sequence, KV
// head) pairs.  Two schedules share the same producer and consumer code:
//  * balanced (the default): a persistent grid of 2 CTAs per SM (1 for the
//    64-row bound); CTA c takes
//    the contiguous tile range [c*T/P, (c+1)*T/P) of the flattened list
//    (T tiles, P CTAs), so every CTA streams the same number of KV bytes
//    whatever the length mix.  A (sequence, KV head) whose tiles straddle
//    CTAs leaves one fp32 partial per CTA; the CTA that finishes that pair
//    last (an atomic counter in the workspace, no waiting) merges the
//    partials by their log-sum-exp and writes the output.
//  * fixed splits (when the caller names a split size): one CTA per
//    (split, KV head, sequence); partials go to the combine kernel.
// CTA = 4 consumer warps + 1 producer warp (+ 1 publisher warp: balanced, FP8).
//  * Producer: one lane walks the block table and issues, per stage, one TMA
//    tile load (cp.async.bulk.tensor, 128-byte swizzle) per block of K and of
//    V: for BF16 a 3D box {64 columns, bs rows, 2 halves} fetches a block's
//    whole 256-byte rows at once (two 2D boxes if the driver refuses that
//    descriptor).  At the first tile of a segment it also bulk-copies the
//    query rows into the stage.  A full mbarrier counts the bytes, an empty
//    mbarrier (4 arrivals) frees the stage; a per-stage TileInfo tells the
//    consumers what the stage holds and marks the CTA's last tile.
//    Every KV byte crosses HBM once per launch; all query rows share it.
//  * Consumers: a grid of kWT token groups x kWC column groups of warps.  Up
//    to 8 query rows (decode) the 4 warps split the tokens of a stage and each
//    holds all columns; beyond 8 they split the columns (8 per n-tile, 1 or 2
//    n-tiles per warp) and read the same tokens.  Per 16-token m-tile:
//      S^T[16 tok x 8] = K[16 x 128] . Q^T[128 x 8]   8 x mma.m16n8k16 per n-tile
//      (tokens fill M; query rows fill N)
//      online softmax on the fragment (3 shuffles per max, exp2 with the
//      scale*log2(e) folded in), P packed to 16 bits and transposed in
//      registers with movmatrix into the B operand of
//      O^T[128 x 8] += V^T[128 x 16 tok] . P^T[16 tok x 8]  8 x mma per n-tile
//      (V^T through ldmatrix.trans for BF16).  The K and V fragments loaded
//      for an m-tile serve every n-tile of the warp.
//  * FP8 pools: E4M3 converts exactly to f16 in registers and the mma runs
//    f16 x f16 -> f32.  K is read with ldmatrix and the head_dim order is
//    permuted consistently in K and Q (a dot product does not depend on the
//    order of its terms); V^T pairs two tokens' bytes with one byte_perm.
//    Q is converted from BF16 to f16 (exact for |q| in [2^-14, 65504]).
//  * At a segment's end the token groups' (m, l, O) are merged through shared
//    memory and the CTA writes the final rows or its fp32 partials.  When a
//    dedicated merge area would cost the second CTA per SM, the merge uses the
//    buffer of the segment's last stage, which is released only afterwards.
//  * Publisher (balanced schedule, FP8 pools): at a segment's end the consumers only put
//    their (m, l, O) into the segment's last stage and post a message; the
//    publisher warp writes the rows or the partial, frees the stage, counts
//    the piece and merges when it is the last.  A partial must be visible
//    GPU-wide before it is counted, and that release waits behind the SM's
//    copies in flight (microseconds mid-stream), so the consumers do not wait
//    for it: they go on with the next segment.
// Rows past the sequence end inside a loaded block are masked in S and zeroed
// in V (uninitialised pool bytes could hold NaN patterns, and 0 * NaN = NaN).
// Every mbarrier wait is bounded; on expiry the CTA flags PKV_ERRBIT_TIMEOUT,
// drains its in-flight copies (bounded) and skips its output.
#pragma once

#include <cuda.h>

#include "device_common.cuh"

namespace pkv {

// Per-dtype translation units.
cudaError_t launch_decode_mma_bf16(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                   cudaStream_t stream);
cudaError_t launch_decode_mma_fp8(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t stream);

namespace {

constexpr int kCWarps = 4;
// The balanced schedule over an FP8 pool adds a publisher warp (see
// publisher()): there the consumers set the pace, and it takes the segment
// ends off them.  Over BF16 the stream of copies sets the pace; three stages in
// flight already cover the consumers' segment ends, and the publisher's
// mid-stream release fence cost more than it saved (measured).
template <int DT, bool kBal>
constexpr bool kPubOf = kBal && DT == PKV_FP8_E4M3;
// consumers + producer (+ publisher)
template <bool kPub>
constexpr int kThreadsOf = (kCWarps + (kPub ? 2 : 1)) * 32;
constexpr int kBoxRowBytes = 128;          // one swizzled TMA row
constexpr int kD = 128;                    // head_dim served by this design
constexpr uint32_t kSpinLimit = 1u << 22;  // try_wait polls before a wait gives up
constexpr size_t kTwoCtaSmem = 115712;     // dynamic shared memory per CTA that still lets 2 CTAs share an SM
constexpr size_t kOneCtaSmem = 232448;     // the per-CTA maximum

template <int DT>
struct MmaCfg;
template <>
struct MmaCfg<PKV_BF16> {
    static constexpr int kHalves = 2;  // 128 columns = two 64-column (128-byte) halves
    static constexpr int kMT = 1;      // 16-token m-tiles per consume step
};
template <>
struct MmaCfg<PKV_FP8_E4M3> {
    static constexpr int kHalves = 1;  // 128 one-byte columns = one 128-byte row
    static constexpr int kMT = 2;      // two independent m-tiles per step: half the bytes per token need more ILP
};

// What one pipeline stage holds.
struct TileInfo {
    int b, h;       // sequence, KV head
    int L;          // the sequence's visible length
    int tok0, n;    // first token of the tile, valid tokens in it (1..kTT)
    int flags;      // kSeg* / kEnd bits
    int pieces;     // CTAs that share this (sequence, KV head)
    int c_first;    // the first of them
    int s_first;    // partial slot that first CTA uses
};
constexpr int kSegFirst = 1;  // first tile of a segment (load q, reset state)
constexpr int kSegLast = 2;   // last tile of a segment (merge and emit)
constexpr int kSegWhole = 4;  // the segment is the whole sequence
constexpr int kCtaFirst = 8;  // the segment holds the CTA's first tile
constexpr int kEnd = 16;      // no tiles at all (a CTA that owns none)
constexpr int kLenRegs = 8;   // sequence lengths per producer lane held in registers by the balanced cut
constexpr int kCtaLast = 32;  // the CTA's last tile

// Shared memory of one CTA:
//   stages: [kStages][K, V][block of the tile][half][bs rows][128 B]
//     A block's two halves (head_dim 0-63 and 64-127 for BF16) are bs*128
//     bytes apart; both start on 1024-byte boundaries (bs >= 16), so the
//     128-byte swizzle phase of a row is its row index within the block, mod 8.
//   q slots [kStages][NQ][128] BF16, tile info [kStages],
//   merge m, l [kWT][NQ] + one flag word,
//   with a publisher: merge m, l [kStages][kWT][NQ] (of a segment ending in that stage),
//   merge O [kWT][NQ][128] fp32 (dedicated, or in the segment's last stage;
//     always the stage with a publisher, which reads it while the consumers
//     go on),
//   barriers full[kStages], empty[kStages], consumer sync, abort word,
//   with a publisher: message barriers [kStages], message ring [kStages], progress word.
template <int DT, int NQ, int HP = 1, bool kPub = false>
struct Layout {
    static constexpr int kHalves = MmaCfg<DT>::kHalves;
    static constexpr int kMT = MmaCfg<DT>::kMT;
    static constexpr int kTT = 16 * kCWarps * kMT / HP;  // tokens per stage (of each of the HP KV heads)
    // warp grid: HP head groups x kWC column groups x kWT token groups
    static constexpr int kNQH = NQ / HP;  // column bound per KV head
    static constexpr int kWC = kNQH <= 8 ? 1 : (kNQH / 8 < kCWarps / HP ? kNQH / 8 : kCWarps / HP);
    static constexpr int kWT = kCWarps / (HP * kWC);
    static constexpr int kNT = kNQH <= 8 ? 1 : kNQH / (8 * kWC);  // n-tiles (8 columns) per warp
    static constexpr int kRowsPerWarp = kTT / kWT;
    // A warp's rows of a stage are consumed kCallMT m-tiles at a time: their
    // QK chains interleave and share one softmax reduction.
    static constexpr int kCallMT = (kRowsPerWarp / 16) < 4 ? (kRowsPerWarp / 16) : 4;
    static constexpr int kCalls = kRowsPerWarp / (16 * kCallMT);
    // Up to 32 rows: 2 CTAs per SM (the register cap is then 168 per thread).
    // 64 rows need two n-tiles of accumulators per warp: 1 CTA per SM with
    // twice the stages keeps as many bytes in flight.
    static constexpr int kMinBlocks = NQ <= 32 ? 2 : 1;
    static constexpr size_t kBudget = kMinBlocks == 2 ? kTwoCtaSmem : kOneCtaSmem;
    static constexpr int kStages = NQ <= 16 ? 3 : (kMinBlocks == 2 ? 2 : 4);
    static constexpr int kTensorBytes = kHalves * kTT * HP * kBoxRowBytes;
    static constexpr int kStageBytes = 2 * kTensorBytes;
    static constexpr int kQBytes = NQ * kD * 2;
    static constexpr size_t kQOff = static_cast<size_t>(kStages) * kStageBytes;
    static constexpr size_t kInfoOff = kQOff + static_cast<size_t>(kStages) * kQBytes;
    static constexpr size_t kMlOff = kInfoOff + static_cast<size_t>(kStages) * sizeof(TileInfo);
    static constexpr size_t kMlBytes = (static_cast<size_t>(kWT) * NQ * 2 + 4) * 4;
    static constexpr size_t kStageMlOff = (kMlOff + kMlBytes + 15) / 16 * 16;
    static constexpr size_t kStageMlBytes = kPub ? static_cast<size_t>(kWT) * NQ * 2 * 4 : 0;
    static constexpr size_t kMergeOBytes = static_cast<size_t>(kWT) * NQ * kD * 4;
    // barriers + abort word (+ message barriers, ring and progress word)
    static constexpr size_t kCtl = (2 * kStages + 1) * 8 + 16 + (kPub ? kStages * 8 + (kStages + 1) * 4 : 0);
    static constexpr size_t kBase = (kStageMlOff + kStages * kStageMlBytes + 15) / 16 * 16;
    static constexpr bool kMergeInStage = kPub || kBase + kMergeOBytes + kCtl + 1024 > kBudget;
    static constexpr size_t kMergeOff = kBase;  // dedicated merge O (unused when kMergeInStage)
    static constexpr size_t kBarOff = kBase + (kMergeInStage ? 0 : kMergeOBytes);
    static constexpr size_t kBytes = kBarOff + kCtl;
    static constexpr size_t kAlloc = kBytes + 1024;  // + alignment slack
    static_assert(kMergeOBytes <= static_cast<size_t>(kStageBytes), "the merge area must fit in a stage");
    static_assert(kNT * 8 * kWC * HP >= NQ && kCalls * kCallMT * 16 == kRowsPerWarp, "warp grid must cover the rows");
    static_assert(HP == 1 || (HP == 2 && NQ <= 8), "KV-head pairs serve decode only");
    static_assert(kAlloc <= kBudget, "shared memory budget");
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
// n arrivals at once (the publisher frees a stage for the 4 consumer warps)
__device__ __forceinline__ void mbar_arrive_n(uint32_t bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(n) : "memory");
}
// Bounded wait for the phase with the given parity to complete: at most
// `polls` polls (0: give up without looking).  A pipeline wait passes the
// CTA's abort word: it also gives up once another warp has raised it, so one
// expired wait ends the whole CTA's pipeline promptly.  The drain waits that
// guard copies still in flight pass none and keep their full bound.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t polls = kSpinLimit,
                                          const volatile int* abort = nullptr) {
    for (uint32_t i = 0; i < polls; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if (abort && (i & 255u) == 255u && *abort) return false;
    }
    return false;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ int cta_linear() {
    return static_cast<int>(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z));
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
// Two 16x16 E4M3 matrices, transposed: lanes 0-15 give the 16-byte rows of
// the first, lanes 16-31 those of the second; lane (g, t) = (lane / 4,
// lane % 4) receives bytes g and g + 8 of rows 4t .. 4t + 3 of each -- the
// A fragment of mma m16n8k32 for a source stored k-major (rows = k).
__device__ __forceinline__ void ldsm_x2_t_b8(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
template <int kImm = 0>
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1+%2];\n" : "=r"(v) : "r"(addr), "n"(kImm) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

template <int DT>
__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    if constexpr (DT == PKV_BF16) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};\n"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// Two floats -> packed 16-bit pair (low = lo) in the mma operand type.
template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (DT == PKV_BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// FP8 pools run both products on the E4M3 tensor-core path, with no
// per-element conversion of the cache: mma m16n8k32 takes E4M3 operands and
// accumulates in fp32.  K and V enter as stored; the query and the
// probabilities, which the method keeps at higher precision, enter as two
// E4M3 terms each, hi = e4m3(x) and lo = e4m3(x - hi), whose two MMAs
// accumulate into one result (hi + lo carries about 8 significant bits,
// as many as BF16).
__device__ __forceinline__ void mma_e4m3(float* c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// f16x2 x -> two E4M3x2 terms (element order kept, low element in the low
// byte): hi = e4m3_rn(x), lo = e4m3_rn(x - hi).  x - hi is exact in f16 (hi
// is x rounded to 4 significant bits, within a factor 2 of it).
__device__ __forceinline__ void split_e4m3x2(uint32_t x, uint32_t& hi, uint32_t& lo) {
    __half2_raw xr;
    xr.x = static_cast<unsigned short>(x & 0xFFFFu);
    xr.y = static_cast<unsigned short>(x >> 16);
    const __nv_fp8x2_storage_t h = __nv_cvt_halfraw2_to_fp8x2(xr, __NV_SATFINITE, __NV_E4M3);
    const __half2_raw hb = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
    __half2 xv, hv;
    *reinterpret_cast<__half2_raw*>(&xv) = xr;
    *reinterpret_cast<__half2_raw*>(&hv) = hb;
    const __half2 r = __hsub2(xv, hv);
    const __nv_fp8x2_storage_t l =
        __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&r), __NV_SATFINITE, __NV_E4M3);
    hi = static_cast<uint32_t>(h);
    lo = static_cast<uint32_t>(l);
}
// Probabilities enter the E4M3 MMA scaled by 2^kFp8PLog2 (they are <= 1;
// E4M3 holds up to 448).
constexpr float kFp8PLog2 = 8.f;

// Byte offset of 16-byte chunk `chunk` of row `lr` inside a 128B-swizzled run
// of rows whose first row sits on a 1024-byte boundary (and is a multiple of 8
// rows into the run).
__device__ __forceinline__ uint32_t swz(int lr, int chunk) {
    return static_cast<uint32_t>(lr * kBoxRowBytes + ((chunk ^ (lr & 7)) << 4));
}

// Head-dim index held by O^T accumulator row `m` (0..15) of m-tile `mt`.
template <int DT>
__device__ __forceinline__ int o_dim(int mt, int m) {
    return mt * 16 + m;
}

// ---------------------------------------------------------------- consumers
// State of one warp's NT n-tiles; lane (r, q) = (lane / 4, lane % 4) holds
// columns 2q and 2q+1 of each n-tile.
template <int NT>
struct Acc {
    float m[NT][2];        // running max (log2 domain) per column
    float l[NT][2];        // lane-partial running sums
    float o[8][NT][4];     // O^T accumulator fragments (8 m-tiles of head_dim)
    uint32_t bq[8][NT][2]; // Q^T as the mma B operand, per 16-wide k-step
    float qk[NT][2];       // score scale (log2 domain) of this lane's two columns
};

// FP8 pools: each query row enters the E4M3 MMA scaled by a power of two,
// 2^-e, chosen so that the row's largest |q| lands in [2^7, 2^8): a BF16
// query of any magnitude then fits E4M3 (largest finite 448) and its f16
// staging copy exactly, and small entries keep the E4M3 range below it;
// 2^e is folded back into that row's score scale.
__device__ __forceinline__ int q_row_exponent(float amax) {
    if (!(amax > 0.f)) return 0;  // zero (or NaN) row
    const int ex = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFFu) - 127;  // floor(log2) for normal amax
    const int e = ex - 7;
    return e < -110 ? -110 : (e > 110 ? 110 : e);  // keeps 2^e and 2^-e normal binary32
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// Start a segment: clear the state and build the Q^T fragments of columns
// [col0, col0 + 8*NT) from the stage's query rows qs[NQ][128] (BF16, shared
// memory); columns >= col_end are zero padding.  qk: the score scale
// (scale * k_scale * log2 e).
template <int DT, int NT>
__device__ __forceinline__ void acc_begin(Acc<NT>& s, const __nv_bfloat16* qs, int lane, int col0, int col_end,
                                          float qk) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        s.m[j][0] = s.m[j][1] = -INFINITY;
        s.l[j][0] = s.l[j][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) s.o[mt][j][0] = s.o[mt][j][1] = s.o[mt][j][2] = s.o[mt][j][3] = 0.f;
    }
    const int r = lane >> 2, q = lane & 3;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int n = col0 + 8 * j + r;
        if constexpr (DT == PKV_BF16) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                if (n >= col_end) {
                    s.bq[ks][j][0] = s.bq[ks][j][1] = 0u;
                    continue;
                }
                const uint32_t* w = reinterpret_cast<const uint32_t*>(qs + n * kD + ks * 16 + 2 * q);
                s.bq[ks][j][0] = w[0];
                s.bq[ks][j][1] = w[4];  // +8 elements
            }
            s.qk[j][0] = s.qk[j][1] = qk;
        } else {
            // E4M3 B fragments of m16n8k32: k32 step kp, register h holds
            // head dims 32 kp + 16 h + 4q .. +3 of row n (K's A fragments come
            // from ldmatrix in natural order).  bq[2 kp] = hi terms, bq[2 kp + 1] = lo.
            // the row's largest |q|: this lane's 32 values, then the row's 4 lanes
            float amax = 0.f;
            if (n < col_end) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const __nv_bfloat16* p = qs + n * kD + ks * 16 + 4 * q;
#pragma unroll
                    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(__bfloat162float(p[i])));
                }
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
            const int e = q_row_exponent(amax);
            const float f = pow2f(-e);
#pragma unroll
            for (int kp = 0; kp < 4; ++kp) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t hi = 0u, lo = 0u;
                    if (n < col_end) {
                        const __nv_bfloat16* p = qs + n * kD + 32 * kp + 16 * h + 4 * q;
                        uint32_t h01, l01, h23, l23;
                        split_e4m3x2(pack2<DT>(__bfloat162float(p[0]) * f, __bfloat162float(p[1]) * f), h01, l01);
                        split_e4m3x2(pack2<DT>(__bfloat162float(p[2]) * f, __bfloat162float(p[3]) * f), h23, l23);
                        hi = h01 | (h23 << 16);
                        lo = l01 | (l23 << 16);
                    }
                    s.bq[2 * kp][j][h] = hi;
                    s.bq[2 * kp + 1][j][h] = lo;
                }
            }
            // this lane's columns 2q, 2q+1 are the rows held by lanes 8q and 8q+4
            const float qrow = qk * pow2f(e);
            s.qk[j][0] = __shfl_sync(0xFFFFFFFFu, qrow, 8 * q);
            s.qk[j][1] = __shfl_sync(0xFFFFFFFFu, qrow, 8 * q + 4);
        }
    }
}

// Per-lane byte offsets (relative to the warp's first row in a tensor of a
// stage) of the shared-memory fragments a consumer lane reads every tile;
// they depend only on the lane, so they are computed once.
struct LaneOffsets {
    uint32_t k[4];  // K ldmatrix rows: chunk pair i (BF16: + half * half_stride)
    uint32_t v[4];  // BF16: V ldmatrix.trans, chunk pair i; FP8: v[0] = byte offset of this lane's V row, v[1] = its swizzle phase
};

template <int DT>
__device__ __forceinline__ LaneOffsets lane_offsets(int lane) {
    LaneOffsets o;
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;  // K: row (of the warp's 16) this lane addresses
#pragma unroll
    for (int i = 0; i < 4; ++i) o.k[i] = swz(lrow, 2 * i + (lane >> 4));
    if constexpr (DT == PKV_BF16) {
        const int trow = (lane & 7) + ((lane >> 4) & 1) * 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) o.v[i] = swz(trow, 2 * i + ((lane >> 3) & 1));
    } else {
        // V rows for ldsm_x2_t_b8: source row i (= k-slot i) of an m-tile is
        // token 2(i/4) + (i%4 & 1) + 8 (i%4 >> 1), the order P's B fragments
        // use (see consume_tile); lanes 16-31 address the second m-tile.
        const int i = lane & 15, row = 2 * (i >> 2) + (i & 1) + 8 * ((i & 3) >> 1);
        o.v[0] = static_cast<uint32_t>(row * kBoxRowBytes);
        o.v[1] = static_cast<uint32_t>(row & 7);
        o.v[2] = o.v[3] = 0;
    }
    return o;
}

// One consume step: this warp's MT m-tiles of 16 rows, [row0, row0 + 16*MT)
// (n valid rows in the stage), against its NT n-tiles.  wb[i]: byte offset of
// m-tile i's first row in a tensor of the stage; half_stride: bytes between a
// block's two 64-column halves.  The m-tiles' S chains are interleaved and
// share one softmax update.  lim[j][0/1]: rows of the tile visible to this
// lane's two columns of n-tile j (all <= n; equal to n for decode).
template <int DT, int MT, int NT>
__device__ __forceinline__ void consume_tile(Acc<NT>& s, uint8_t* kst, uint8_t* vst, int n, int row0, int lane,
                                             const uint32_t (&wb)[MT], uint32_t half_stride,
                                             const LaneOffsets& lo, const int (&lim)[NT][2]) {
    constexpr int kHalves = MmaCfg<DT>::kHalves;
    if (row0 >= n) return;
    const int r = lane >> 2;
    if (n < row0 + 16 * MT) {  // zero these V rows past the end (other column groups write the same zeros)
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            if (row0 + 16 * i >= n) continue;  // a fully empty m-tile is skipped below
            for (int e = lane; e < 16 * kHalves * 8; e += 32) {
                const int lr = e / (kHalves * 8);
                const int rest = e % (kHalves * 8);
                if (row0 + 16 * i + lr >= n)
                    *reinterpret_cast<uint4*>(vst + wb[i] + (rest >> 3) * half_stride + lr * kBoxRowBytes +
                                              (rest & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async();
        __syncwarp();
    }
    bool live[MT];
#pragma unroll
    for (int i = 0; i < MT; ++i) live[i] = row0 + 16 * i < n;
    // ---- S^T = K Q^T, m-tiles interleaved; one K fragment feeds every n-tile
    float sc[MT][NT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j) sc[i][j][0] = sc[i][j][1] = sc[i][j][2] = sc[i][j][3] = 0.f;
    const uint32_t kb = smem_u32(kst);
    if constexpr (DT == PKV_BF16) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                if (!live[i]) continue;
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kb + wb[i] + (ks >> 2) * half_stride + lo.k[ks & 3], a0, a1, a2, a3);
#pragma unroll
                for (int j = 0; j < NT; ++j) mma16816<DT>(sc[i][j], a0, a1, a2, a3, s.bq[ks][j][0], s.bq[ks][j][1]);
            }
        }
    } else {
        // one ldmatrix.x4 = the E4M3 A fragment of a k32 step (bytes 32 kp ..
        // 32 kp + 31 of 16 token rows); hi and lo query terms accumulate apart
        // (two independent chains) and are summed after the last step
        // four independent accumulator chains per m-tile: hi / lo terms x
        // head-dim halves (each two k32 steps long)
        float sl[MT][NT][4], sc2[MT][NT][4], sl2[MT][NT][4];
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) sl[i][j][c] = sc2[i][j][c] = sl2[i][j][c] = 0.f;
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                if (!live[i]) continue;
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kb + wb[i] + lo.k[kp], r0, r1, r2, r3);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    mma_e4m3(kp < 2 ? sc[i][j] : sc2[i][j], r0, r1, r2, r3, s.bq[2 * kp][j][0], s.bq[2 * kp][j][1]);
                    mma_e4m3(kp < 2 ? sl[i][j] : sl2[i][j], r0, r1, r2, r3, s.bq[2 * kp + 1][j][0],
                             s.bq[2 * kp + 1][j][1]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < MT; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int c = 0; c < 4; ++c) sc[i][j][c] = (sc[i][j][c] + sl[i][j][c]) + (sc2[i][j][c] + sl2[i][j][c]);
    }
    // FP8: probabilities (and with them l and O) carry a factor 2^kPLog2, so
    // that they fill E4M3's range (they are <= 1 before it; E4M3 holds up to
    // 448); it cancels in O / l and is taken out of each log-sum-exp.
    constexpr float kPLog2 = DT == PKV_FP8_E4M3 ? kFp8PLog2 : 0.f;
    // ---- online softmax (log2 domain) over the step's 16*MT rows, per column
    float sv[MT][NT][4];
    float x[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) x[j][0] = x[j][1] = -INFINITY;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        const int ra = row0 + 16 * i + r, rb = ra + 8;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            sv[i][j][0] = ra < lim[j][0] ? sc[i][j][0] * s.qk[j][0] : -INFINITY;
            sv[i][j][1] = ra < lim[j][1] ? sc[i][j][1] * s.qk[j][1] : -INFINITY;
            sv[i][j][2] = rb < lim[j][0] ? sc[i][j][2] * s.qk[j][0] : -INFINITY;
            sv[i][j][3] = rb < lim[j][1] ? sc[i][j][3] * s.qk[j][1] : -INFINITY;
            x[j][0] = fmaxf(x[j][0], fmaxf(sv[i][j][0], sv[i][j][2]));
            x[j][1] = fmaxf(x[j][1], fmaxf(sv[i][j][1], sv[i][j][3]));
        }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            x[j][0] = fmaxf(x[j][0], __shfl_xor_sync(0xFFFFFFFFu, x[j][0], off));
            x[j][1] = fmaxf(x[j][1], __shfl_xor_sync(0xFFFFFFFFu, x[j][1], off));
        }
    }
    // a column that has seen no token yet keeps max -inf; b = its exponent base
    float nm[NT][2], bb[NT][2];
    bool moved = false;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            nm[j][h] = fmaxf(s.m[j][h], x[j][h]);
            bb[j][h] = nm[j][h] == -INFINITY ? 0.f : nm[j][h];
            moved = moved || nm[j][h] != s.m[j][h];
        }
    }
    float p[MT][NT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            p[i][j][0] = exp2f(sv[i][j][0] - bb[j][0] + kPLog2);
            p[i][j][1] = exp2f(sv[i][j][1] - bb[j][1] + kPLog2);
            p[i][j][2] = exp2f(sv[i][j][2] - bb[j][0] + kPLog2);
            p[i][j][3] = exp2f(sv[i][j][3] - bb[j][1] + kPLog2);
        }
    }
    // rescale only when some running max moved (the factor is exactly 1
    // otherwise); against b, a column still without tokens gets 0, not 2^NaN
    if (__any_sync(0xFFFFFFFFu, moved)) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float al0 = exp2f(s.m[j][0] - bb[j][0]), al1 = exp2f(s.m[j][1] - bb[j][1]);
            s.l[j][0] *= al0;
            s.l[j][1] *= al1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                s.o[mt][j][0] *= al0;
                s.o[mt][j][1] *= al1;
                s.o[mt][j][2] *= al0;
                s.o[mt][j][3] *= al1;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            s.l[j][0] += p[i][j][0] + p[i][j][2];
            s.l[j][1] += p[i][j][1] + p[i][j][3];
        }
        s.m[j][0] = nm[j][0];
        s.m[j][1] = nm[j][1];
    }
    // ---- O^T += V^T P^T; one V fragment feeds every n-tile
    const uint32_t vb0 = smem_u32(vst);
    if constexpr (DT == PKV_BF16) {
        uint32_t pb[MT][NT][2];
#pragma unroll
        for (int i = 0; i < MT; ++i) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                pb[i][j][0] = movmatrix_t(pack2<DT>(p[i][j][0], p[i][j][1]));  // tokens 0-7 of m-tile i
                pb[i][j][1] = movmatrix_t(pack2<DT>(p[i][j][2], p[i][j][3]));  // tokens 8-15
            }
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                if (!live[i]) continue;
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vb0 + wb[i] + (mt >> 2) * half_stride + lo.v[mt & 3], a0, a1, a2, a3);
#pragma unroll
                for (int j = 0; j < NT; ++j) mma16816<DT>(s.o[mt][j], a0, a1, a2, a3, pb[i][j][0], pb[i][j][1]);
            }
        }
    } else {
        static_assert(MT % 2 == 0, "an E4M3 k32 step spans two 16-token m-tiles");
        // k-slot order within a 16-token m-tile: slots 4q .. 4q+3 hold tokens
        // 2q, 2q+1, 2q+8, 2q+9 (the same order in P and in V, so every product
        // pairs the right token); a k32 step covers m-tiles (i, i+1).
        // P^T (scaled by 2^8) as hi / lo E4M3 B fragments per m-tile
        uint32_t ph[MT][NT], pl[MT][NT];
#pragma unroll
        for (int i = 0; i < MT; ++i) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                uint32_t t0 = movmatrix_t(pack2<DT>(p[i][j][0], p[i][j][1]));  // (column r; tokens 2q, 2q+1)
                uint32_t t1 = movmatrix_t(pack2<DT>(p[i][j][2], p[i][j][3]));  // (column r; tokens 2q+8, 2q+9)
                uint32_t hi0, lo0, hi1, lo1;
                split_e4m3x2(t0, hi0, lo0);
                split_e4m3x2(t1, hi1, lo1);
                ph[i][j] = hi0 | (hi1 << 16);
                pl[i][j] = lo0 | (lo1 << 16);
            }
        }
        // V^T A fragments straight from the staged rows: one transposing
        // ldmatrix per 16 head dims (O^T m-tile c) and k32 step; the source rows
        // follow the k-slot order above (lo.v[0]); a dead second m-tile's
        // stale rows are replaced by zeros.
#pragma unroll
        for (int i0 = 0; i0 < MT; i0 += 2) {
            if (!live[i0]) continue;
            const uint32_t vrow = vb0 + (lane < 16 ? wb[i0] : wb[i0 + 1]) + lo.v[0];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t a0, a1, a2, a3;
                ldsm_x2_t_b8(vrow + ((static_cast<uint32_t>(c) ^ lo.v[1]) << 4), a0, a1, a2, a3);
                if (!live[i0 + 1]) a2 = a3 = 0u;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    mma_e4m3(s.o[c][j], a0, a1, a2, a3, ph[i0][j], ph[i0 + 1][j]);
                    mma_e4m3(s.o[c][j], a0, a1, a2, a3, pl[i0][j], pl[i0 + 1][j]);
                }
            }
        }
    }
}

// Merge area: O [token group][NQ][128], m and l [token group][NQ], a flag word.
template <int NQ, int WT>
struct Merge {
    float* o;
    float* m;
    float* l;
    volatile int* flag;
    __device__ Merge(uint8_t* o_base, uint8_t* ml_base) {
        o = reinterpret_cast<float*>(o_base);
        m = reinterpret_cast<float*>(ml_base);
        l = m + WT * NQ;
        flag = reinterpret_cast<volatile int*>(l + WT * NQ);
    }
};

// Publish this warp's (m, l, O) for its columns [col0, min(col0 + 8*NT, col_end)) as token group wt.
template <int DT, int NQ, int WT, int NT>
__device__ __forceinline__ void merge_put(const Acc<NT>& s, const Merge<NQ, WT>& mg, int wt, int col0, int col_end,
                                          int lane) {
    const int cend = col_end < NQ ? col_end : NQ;
    const int r = lane >> 2, q = lane & 3;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        float l0 = s.l[j][0], l1 = s.l[j][1];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
            l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
        }
        const int n0 = col0 + 8 * j + 2 * q, n1 = n0 + 1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            if (n0 < cend) {
                mg.o[(wt * NQ + n0) * kD + o_dim<DT>(mt, r)] = s.o[mt][j][0];
                mg.o[(wt * NQ + n0) * kD + o_dim<DT>(mt, r + 8)] = s.o[mt][j][2];
            }
            if (n1 < cend) {
                mg.o[(wt * NQ + n1) * kD + o_dim<DT>(mt, r)] = s.o[mt][j][1];
                mg.o[(wt * NQ + n1) * kD + o_dim<DT>(mt, r + 8)] = s.o[mt][j][3];
            }
        }
        if (lane < 4) {
            if (n0 < cend) {
                mg.m[wt * NQ + n0] = s.m[j][0];
                mg.l[wt * NQ + n0] = l0;
            }
            if (n1 < cend) {
                mg.m[wt * NQ + n1] = s.m[j][1];
                mg.l[wt * NQ + n1] = l1;
            }
        }
    }
}

// Merged (sum O, max m, sum l) of column n at head-dim index d.
template <int NQ, int WT>
__device__ __forceinline__ void merge_get(const Merge<NQ, WT>& mg, int n, int d, float& acc, float& M, float& lsum) {
    M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WT; ++w) M = fmaxf(M, mg.m[w * NQ + n]);
    acc = 0.f;
    lsum = 0.f;
    if (M == -INFINITY) return;  // no token for this query in the segment
#pragma unroll
    for (int w = 0; w < WT; ++w) {
        const float f = exp2f(mg.m[w * NQ + n] - M);  // token groups without rows: 2^-inf = 0
        acc += f * mg.o[(w * NQ + n) * kD + d];
        lsum += f * mg.l[w * NQ + n];
    }
}

// Output row of column n of (sequence b, KV head unit h): query q_first +
// n / gh, head h * gh + n % gh; for a KV-head pair (decode) unit h is heads
// 2h, 2h+1 and column n is query head 2h * gh + n.
template <int HP = 1>
__device__ __forceinline__ size_t out_row(const DecodeArgs& a, int b, int h, int n, int gh) {
    if constexpr (HP == 1)
        return (static_cast<size_t>(b) * a.q_total + a.q_first + n / gh) * a.num_q_heads +
               static_cast<size_t>(h) * gh + n % gh;
    else
        return (static_cast<size_t>(b) * a.q_total + a.q_first) * a.num_q_heads + static_cast<size_t>(HP * h) * gh + n;
}

// Fused append (decode), done by the producer warp: the rows [K, V] x [HP
// heads] x [chunks] of a unit's newest token, lane `lane` owning output chunks
// lane + 32 j.  prefetch() issues the input loads when a segment that ends
// the unit starts; write() encodes them exactly as kv_append does and stores
// them at the position's slot just before the TMA copy of that block, with a
// proxy fence so that the copy reads the new bytes.
template <int DT, int HP>
struct NewRows {
    static constexpr int kPoolBytes = DT == PKV_BF16 ? 2 : 1;
    static constexpr int kPer = 16 / kPoolBytes;          // pool elements per 16-byte chunk
    static constexpr int kChunksRow = kD / kPer;          // 16 (BF16) or 8 (FP8) chunks per row
    static constexpr int kTotal = 2 * HP * kChunksRow;    // K and V rows of the HP heads
    static constexpr int kOut = (kTotal + 31) / 32;       // output chunks per lane
    static constexpr int kInMax = DT == PKV_BF16 ? 2 : 4; // 16-byte input chunks per output chunk (f32 input)
    uint4 x[kOut][kInMax];

    __device__ __forceinline__ void prefetch(const DecodeArgs& a, int b, int h, int lane) {
        const bool f32 = a.new_dtype == PKV_F32;
        const int nin = f32 ? kInMax : kInMax / 2;
#pragma unroll
        for (int j = 0; j < kOut; ++j) {
            const int oc = lane + 32 * j;
            if (oc >= kTotal) continue;
            const int tensor = oc / (HP * kChunksRow), head = (oc / kChunksRow) % HP, c = oc % kChunksRow;
            const uint4* src = reinterpret_cast<const uint4*>(
                (tensor ? a.new_v : a.new_k) +
                ((static_cast<size_t>(b) * a.num_kv_heads + HP * h + head) * kD + c * kPer) * (f32 ? 4 : 2));
#pragma unroll
            for (int i = 0; i < kInMax; ++i)
                if (i < nin) x[j][i] = __ldg(src + i);
        }
    }

    __device__ __forceinline__ void write(const DecodeArgs& a, int h, int blk, int row, int lane) {
        const bool f32 = a.new_dtype == PKV_F32;
#pragma unroll
        for (int j = 0; j < kOut; ++j) {
            const int oc = lane + 32 * j;
            if (oc >= kTotal) continue;
            const int tensor = oc / (HP * kChunksRow), head = (oc / kChunksRow) % HP, c = oc % kChunksRow;
            const float inv = tensor ? a.v_inv_scale : a.k_inv_scale;
            const uint4 w = f32 ? AppendChunk<DT, PKV_F32>::convert(x[j], inv)
                                : AppendChunk<DT, PKV_BF16>::convert(x[j], inv);
            uint8_t* dst = (tensor ? a.v_layer_w : a.k_layer_w) +
                           ((static_cast<size_t>(blk) * a.num_kv_heads + HP * h + head) * a.block_size + row) * kD *
                               kPoolBytes +
                           c * 16;
            *reinterpret_cast<uint4*>(dst) = w;
        }
        asm volatile("fence.proxy.async.global;\n" ::: "memory");
    }
};

// ---------------------------------------------------------------- producer
// The pool block ids of tile ti, one per lane (lane k: block k of the tile;
// -1 past the tile).  The producer loads them before it waits for a free
// stage, so the block table's latency overlaps that wait.
__device__ __forceinline__ int tile_blocks(const DecodeArgs& a, const int32_t* table, const TileInfo& ti, int lane) {
    const int bs = a.block_size;
    const int nblk = (ti.n + bs - 1) / bs;  // <= 32 (a tile holds at most 128 tokens)
    const int j = ti.tok0 / bs + lane;
    return (lane < nblk && j < a.max_blocks) ? __ldg(table + j) : -1;
}

// Stage s <- tile ti: tile info, the query rows at a segment's first tile,
// and one TMA box per KV block (K and V).  All 32 producer lanes call it
// (lane k holds block k's id, from tile_blocks); lane 0 issues.
template <int DT, int NQ, int HP, bool kPub>
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                            uint8_t* smem, uint64_t* full, int s, const TileInfo& ti, int myblk,
                                            int lane, int gh, NewRows<DT, HP>& nr, bool append) {
    using Lt = Layout<DT, NQ, HP, kPub>;
    const int bs = a.block_size;
    uint8_t* kst = smem + s * Lt::kStageBytes;
    uint8_t* vst = kst + Lt::kTensorBytes;
    const uint32_t fb = smem_u32(&full[s]);
    const int nblk = (ti.n + bs - 1) / bs;
    const bool need_q = (ti.flags & kSegFirst) != 0;
    if (lane == 0) {
        reinterpret_cast<TileInfo*>(smem + Lt::kInfoOff)[s] = ti;
        const uint32_t qbytes = static_cast<uint32_t>(a.num_queries * gh * kD * 2);
        mbar_expect_tx(fb, static_cast<uint32_t>(nblk * HP * bs * kBoxRowBytes * Lt::kHalves * 2) +
                               (need_q ? static_cast<uint32_t>(HP) * qbytes : 0u));
        if (need_q) {
            if constexpr (HP == 1) {  // query rows n = c * gh + g: one copy of gh contiguous rows per query
                for (int c = 0; c < a.num_queries; ++c) {
                    const __nv_bfloat16* qsrc =
                        static_cast<const __nv_bfloat16*>(a.q) + out_row(a, ti.b, ti.h, c * gh, gh) * kD;
                    bulk_load(smem_u32(smem + Lt::kQOff + s * Lt::kQBytes + c * gh * kD * 2), qsrc,
                              static_cast<uint32_t>(gh * kD * 2), fb);
                }
            } else {  // a pair's HP * gh query heads are contiguous
                const __nv_bfloat16* qsrc = static_cast<const __nv_bfloat16*>(a.q) + out_row<HP>(a, ti.b, ti.h, 0, gh) * kD;
                bulk_load(smem_u32(smem + Lt::kQOff + s * Lt::kQBytes), qsrc, HP * qbytes, fb);
            }
        }
    }
    const int64_t layer_blk0 = static_cast<int64_t>(a.layer) * a.num_blocks;
    if (append) {  // the block holding the unit's newest position takes its new row before the copies
        const int blk = __shfl_sync(0xFFFFFFFFu, myblk, nblk - 1);
        if (static_cast<unsigned>(blk) < static_cast<unsigned>(a.num_blocks)) nr.write(a, ti.h, blk, (ti.L - 1) % bs, lane);
    }
    __syncwarp();  // (and the expected bytes are posted before any copy lands)
    // One copy instruction for the whole stage: lane l copies box l of the
    // (block, K or V, half) list.  Issuing a copy costs a few hundred cycles,
    // about the same for one lane or several, so one lane issuing them in
    // turn held the ring back.  A box holds the block's rows of the HP
    // adjacent KV heads; with 3D boxes, both 128-byte halves of every row.
    constexpr int kBoxes = 1;  // per block and tensor with 3D boxes
    const int bpb = (Lt::kHalves == 2 && a.tma_3d) ? kBoxes : Lt::kHalves;
    const int k = lane / (2 * bpb), r = lane % (2 * bpb), tv = r / bpb, hf = r % bpb;
    int blk = __shfl_sync(0xFFFFFFFFu, myblk, k & 31);
    if (k < nblk) {  // nblk * 2 * bpb <= 32: a tile holds at most 128 tokens, blocks hold 16 or more
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.num_blocks)) {
            if (a.err) atomicOr(a.err, PKV_ERRBIT_BLOCK_ID);
            blk = 0;  // read an in-bounds block; the flag marks the output invalid
        }
        const int y = static_cast<int>(((layer_blk0 + blk) * a.num_kv_heads + HP * ti.h) * bs);
        const uint32_t off = k * Lt::kHalves * HP * bs * kBoxRowBytes;
        uint8_t* dst = tv ? vst : kst;
        const CUtensorMap* map = tv ? tmv : tmk;
        if (Lt::kHalves == 2 && a.tma_3d) {
            tma_load_3d(smem_u32(dst + off), map, 0, y, 0, fb);
        } else {  // (never with HP = 2: the host requires 3D boxes)
            tma_load_2d(smem_u32(dst + off + hf * HP * bs * kBoxRowBytes), map, hf * 64, y, fb);
        }
    }
}

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Tiles of sequence b (kTT tokens each), 0 past the batch.
template <int kTT>
__device__ __forceinline__ int seq_tiles(const DecodeArgs& a, int b) {
    return b < a.num_seqs ? (visible_len(a, b, false) + kTT - 1) / kTT : 0;
}

// Publisher warp (balanced schedule, FP8 pools).  Message i is the i-th segment end of
// the CTA: its stage holds the token groups' O, the stage's m/l slot their
// m and l, and info[stage] the segment.  Messages are taken in order; each
// keeps its stage until the publisher frees it, so at most kStages are
// outstanding and a ring of kStages slots cannot be overrun.  Lane l owns
// head-dim entries 4l..4l+3 of every row.
template <int DT, int NQ, int HP>
__device__ __forceinline__ void publisher(const DecodeArgs& a, uint8_t* smem, uint64_t* empty, uint64_t* msg_full,
                                          const volatile int* msg_ring, const volatile int* progress,
                                          volatile int* abort_flag, int lane, int gh, int nq) {
    using Lt = Layout<DT, NQ, HP, true>;
    constexpr int kStages = Lt::kStages;
    constexpr int kWT = Lt::kWT;
    constexpr float kLseBias = DT == PKV_FP8_E4M3 ? kFp8PLog2 : 0.f;
    const float vscale = a.v_scale;
    const TileInfo* info = reinterpret_cast<const TileInfo*>(smem + Lt::kInfoOff);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    struct Piece {
        int b, h, pieces, c_first, s_first;
    };
    // every piece is published: out = sum_j 2^(lse_j - M) o_j / sum_j 2^(lse_j - M),
    // accumulated piece by piece with the running maximum M
    auto merge = [&](const Piece& pc) {
        for (int n0 = 0; n0 < nq; n0 += 4) {
            float4 acc[4];
            float Mx[4], z[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                Mx[u] = -INFINITY;
                z[u] = 0.f;
            }
#pragma unroll 2
            for (int j = 0; j < pc.pieces; ++j) {
                const size_t pb = (static_cast<size_t>(pc.c_first + j) * 2 + (j == 0 ? pc.s_first : 0)) * NQ;
                float lj[4];
                float4 oj[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int n = n0 + u < nq ? n0 + u : n0;
                    lj[u] = __ldcg(a.bal_lse + pb + n);
                    oj[u] = __ldcg(reinterpret_cast<const float4*>(a.bal_o + (pb + n) * kD) + lane);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (lj[u] == -INFINITY) continue;  // a piece with no token for this query
                    const float Mn = fmaxf(Mx[u], lj[u]);
                    const float c = exp2f(Mx[u] - Mn), w = exp2f(lj[u] - Mn);
                    acc[u].x = fmaf(w, oj[u].x, acc[u].x * c);
                    acc[u].y = fmaf(w, oj[u].y, acc[u].y * c);
                    acc[u].z = fmaf(w, oj[u].z, acc[u].z * c);
                    acc[u].w = fmaf(w, oj[u].w, acc[u].w * c);
                    z[u] = fmaf(z[u], c, w);
                    Mx[u] = Mn;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int n = n0 + u;
                if (n >= nq) break;
                const float iz = z[u] > 0.f ? 1.f / z[u] : 0.f;
                const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[u].x * iz, acc[u].y * iz);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[u].z * iz, acc[u].w * iz);
                uint2 pk;
                pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                reinterpret_cast<uint2*>(out + out_row<HP>(a, pc.b, pc.h, n, gh) * kD)[lane] = pk;
            }
        }
        if (lane == 0) a.counters[static_cast<size_t>(pc.b) * a.num_kv_heads + pc.h] = 0;  // ready for the next call
    };
    for (long long i = 0;; ++i) {
        const int r = static_cast<int>(i % kStages);
        // The wait may span a whole segment: rounds of bounded polls, another
        // round only while the consumers keep taking tiles.
        bool got = false;
        for (int seen = *progress;;) {
            if (mbar_wait(smem_u32(&msg_full[r]), static_cast<uint32_t>((i / kStages) & 1), kSpinLimit, abort_flag)) {
                got = true;
                break;
            }
            const int now = *progress;
            if (*abort_flag || now == seen) break;
            seen = now;
        }
        if (!got) {
            if (lane == 0 && !*abort_flag) {
                *abort_flag = 1;
                if (a.err) atomicOr(a.err, PKV_ERRBIT_TIMEOUT);
            }
            return;
        }
        const int s = msg_ring[r];
        if (s < 0) return;  // a CTA without tiles
        const TileInfo ti = info[s];
        const float* mo = reinterpret_cast<const float*>(smem + static_cast<size_t>(s) * Lt::kStageBytes);
        const float* mm = reinterpret_cast<const float*>(smem + Lt::kStageMlOff + s * Lt::kStageMlBytes);
        const float* ml = mm + kWT * NQ;
        const bool whole = (ti.flags & kSegWhole) != 0;
        const size_t pbase = (static_cast<size_t>(blockIdx.x) * 2 + ((ti.flags & kCtaFirst) ? 0 : 1)) * NQ;
        // the segment's rows: sum the token groups' O, scaled to the largest m
#pragma unroll 4
        for (int n = 0; n < nq; ++n) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWT; ++w) M = fmaxf(M, mm[w * NQ + n]);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            float l = 0.f;
            if (M != -INFINITY) {  // else no token for this query in the segment
#pragma unroll
                for (int w = 0; w < kWT; ++w) {
                    const float f = exp2f(mm[w * NQ + n] - M);  // token groups without rows: 2^-inf = 0
                    const float4 o = reinterpret_cast<const float4*>(mo + (w * NQ + n) * kD)[lane];
                    v.x += f * o.x;
                    v.y += f * o.y;
                    v.z += f * o.z;
                    v.w += f * o.w;
                    l += f * ml[w * NQ + n];
                }
            }
            const float sc = l > 0.f ? vscale / l : 0.f;
            if (whole) {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x * sc, v.y * sc);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z * sc, v.w * sc);
                uint2 pk;
                pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                reinterpret_cast<uint2*>(out + out_row<HP>(a, ti.b, ti.h, n, gh) * kD)[lane] = pk;
            } else {
                reinterpret_cast<float4*>(a.bal_o + (pbase + n) * kD)[lane] =
                    make_float4(v.x * sc, v.y * sc, v.z * sc, v.w * sc);
                if (lane == 0) a.bal_lse[pbase + n] = l > 0.f ? M + log2f(l) - kLseBias : -INFINITY;
            }
        }
        // the merge area is read: the producer may refill the stage
        __syncwarp();
        if (lane == 0) mbar_arrive_n(smem_u32(&empty[s]), kCWarps);
        if (!whole) {
            // Count the piece: one GPU-scope acq_rel atomic after the warp's
            // writes (ordered before it by the __syncwarp above); the last
            // piece's lanes read the others' writes after it.
            int last = 0;
            if (lane == 0)
                last = (atom_add_acq_rel(a.counters + static_cast<size_t>(ti.b) * a.num_kv_heads + ti.h, 1) ==
                        ti.pieces - 1)
                           ? 1
                           : 0;
            __syncwarp();
            if (__shfl_sync(0xFFFFFFFFu, last, 0)) merge(Piece{ti.b, ti.h, ti.pieces, ti.c_first, ti.s_first});
        }
        if (ti.flags & kCtaLast) return;
    }
}

// kBal: balanced persistent schedule (grid = P CTAs); otherwise one CTA per
// (split, KV head, sequence) with grid (num_splits, num_kv_heads, num_seqs).
template <int DT, int NQ, bool kBal, int HP>
__global__ void __launch_bounds__(kThreadsOf<kPubOf<DT, kBal>>, Layout<DT, NQ, HP, kPubOf<DT, kBal>>::kMinBlocks)
decode_mma_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
    constexpr bool kPub = kPubOf<DT, kBal>;
    using Lt = Layout<DT, NQ, HP, kPub>;
    constexpr int kStages = Lt::kStages;
    constexpr int kHalves = Lt::kHalves;
    constexpr int kTT = Lt::kTT;
    constexpr int kWC = Lt::kWC;
    constexpr int kWT = Lt::kWT;
    constexpr int kNT = Lt::kNT;
    constexpr int kCallMT = Lt::kCallMT;
    constexpr int kCalls = Lt::kCalls;
    constexpr bool kInStage = Lt::kMergeInStage;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lt::kBarOff);
    uint64_t* empty = full + kStages;
    uint64_t* csync_bar = empty + kStages;  // the 4 consumer warps meet here at segment ends
    volatile int* abort_flag = reinterpret_cast<volatile int*>(csync_bar + 1);
    // publisher: message i (a segment end) is the stage msg_ring[i % kStages], posted on msg_full[i % kStages]
    uint64_t* msg_full = csync_bar + 3;
    volatile int* msg_ring = reinterpret_cast<volatile int*>(msg_full + kStages);
    volatile int* progress = msg_ring + kStages;  // tiles the consumers have taken
    const TileInfo* info = reinterpret_cast<const TileInfo*>(smem + Lt::kInfoOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gh = a.num_q_heads / a.num_kv_heads;  // query heads per KV head
    const int nq = HP * a.num_queries * gh;         // real query rows (<= NQ)
    const int Hu = a.num_kv_heads / HP;             // KV-head units per sequence

    // Launched as a programmatic dependent of the previous kernel in the
    // stream (the append, or the previous decode step): nothing is read
    // before that grid has finished.  The next kernel may be scheduled at
    // once: it too waits before it reads anything, so its CTAs take over SMs
    // as ours leave.
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    asm volatile("griddepcontrol.wait;\n" ::: "memory");

    // fixed schedule: this CTA's one segment
    int fb_ = 0, fh_ = 0, fsplit = 0, t_begin = 0, t_end = 0, fL = 0;
    if constexpr (!kBal) {
        fsplit = blockIdx.x;
        fh_ = blockIdx.y;
        fb_ = blockIdx.z;
        const int L = visible_len(a, fb_, fsplit == 0 && fh_ == 0 && threadIdx.x == 0);
        fL = L;
        t_begin = fsplit * a.split_tokens;
        t_end = min(L, t_begin + a.split_tokens);
        if (t_begin >= t_end) {
            if (a.num_splits == 1) {  // nothing visible: zero output rows
                for (int i = threadIdx.x; i < nq * kD; i += kThreadsOf<kPub>)
                    static_cast<__nv_bfloat16*>(a.out)[out_row<HP>(a, fb_, fh_, i / kD, gh) * kD + i % kD] =
                        __float2bfloat16_rn(0.f);
            }
            return;
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kCWarps);
        }
        mbar_init(smem_u32(csync_bar), kCWarps);
        *abort_flag = 0;
        if constexpr (kPub) {
            for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&msg_full[s]), kCWarps);
            *progress = 0;
        }
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    if (warp == kCWarps) {
        // ------------------------------------------------------------ producer
        long long k = 0;  // stages issued
        bool ok = true;
        auto acquire = [&](long long kk) -> int {  // stage for the kk-th issue, after it is free
            const int s = static_cast<int>(kk % kStages);
            if (kk >= kStages && ok)
                ok = mbar_wait(smem_u32(&empty[s]), static_cast<uint32_t>(((kk / kStages) - 1) & 1), kSpinLimit,
                               abort_flag);
            if (*abort_flag) ok = false;
            return s;
        };
        if constexpr (kBal) {
            const int B = a.num_seqs, Hkv = Hu;
            // The tiles of sequences lane, lane + 32, ... (batches up to 256):
            // one round of independent loads for both passes below, instead
            // of a dependent load per 32 sequences and pass.
            int ntl[kLenRegs];
#pragma unroll
            for (int i = 0; i < kLenRegs; ++i) ntl[i] = seq_tiles<kTT>(a, 32 * i + lane);
            auto tiles32 = [&](int b0) {  // the tiles of sequence b0 + lane
                int v = 0;
#pragma unroll
                for (int i = 0; i < kLenRegs; ++i)
                    if (b0 == 32 * i) v = ntl[i];
                return b0 < 32 * kLenRegs ? v : seq_tiles<kTT>(a, b0 + lane);
            };
            long long T = 0;
#pragma unroll 4
            for (int b0 = 0; b0 < B; b0 += 32) T += warp_sum_ll(tiles32(b0));
            T *= Hkv;
            // CTA c < P owns tiles [c*T/P, (c+1)*T/P); P <= T keeps every range non-empty
            const long long P = T < static_cast<long long>(gridDim.x) ? T : static_cast<long long>(gridDim.x);
            const long long c = blockIdx.x;
            const long long g0 = c < P ? c * T / P : T, g1 = c < P ? (c + 1) * T / P : T;
            if (g0 < g1) {
                // locate tile g0: sequence b, and cum = tiles before b (x Hkv)
                long long cum = 0;
                int b = 0;
                for (int b0 = 0; b0 < B; b0 += 32) {
                    const long long u = static_cast<long long>(tiles32(b0)) * Hkv;
                    long long incl = u;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                        if (lane >= o) incl += t;
                    }
                    const long long tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
                    if (g0 < cum + tot) {
                        const unsigned m = __ballot_sync(0xFFFFFFFFu, cum + incl > g0);
                        const int l = __ffs(m) - 1;
                        cum += __shfl_sync(0xFFFFFFFFu, incl - u, l);
                        b = b0 + l;
                        break;
                    }
                    cum += tot;
                }
                int L = visible_len(a, b, false);
                int nt = (L + kTT - 1) / kTT;
                const long long off = g0 - cum;
                int h = static_cast<int>(off / nt), t = static_cast<int>(off % nt);
                const int32_t* table = a.tables + static_cast<size_t>(b) * a.max_blocks;
                auto owner = [&](long long g) { return ((g + 1) * P - 1) / T; };
                TileInfo ti;
                NewRows<DT, HP> nr;
                bool app = false;  // this CTA appends the current unit's newest token
                for (long long g = g0; g < g1 && ok; ++g, ++k) {
                    const long long pstart = cum + static_cast<long long>(h) * nt, pend = pstart + nt;
                    if (g == g0 || t == 0) {  // a new segment: who shares this (sequence, KV head)
                        if constexpr (NQ <= 8) {  // fused append: the segment holds the unit's last tile
                            app = a.new_k != nullptr && pend <= g1 && a.lens[b] == L;
                            if (app) nr.prefetch(a, b, h, lane);
                        }
                        const long long cf = owner(pstart);
                        ti.b = b;
                        ti.h = h;
                        ti.c_first = static_cast<int>(cf);
                        ti.pieces = static_cast<int>(owner(pend - 1) - cf + 1);
                        ti.s_first = (cf * T / P < pstart) ? 1 : 0;
                    }
                    ti.L = L;
                    ti.tok0 = t * kTT;
                    ti.n = min(kTT, L - ti.tok0);
                    ti.flags = ((g == g0 || t == 0) ? kSegFirst : 0) | ((g == g1 - 1 || t == nt - 1) ? kSegLast : 0) |
                               ((pstart >= g0 && pend <= g1) ? kSegWhole : 0) | (pstart <= g0 ? kCtaFirst : 0) |
                               (g == g1 - 1 ? kCtaLast : 0);
                    const int myblk = tile_blocks(a, table, ti, lane);
                    const int s = acquire(k);
                    if (!ok) break;
                    issue_stage<DT, NQ, HP, kPub>(a, &tmk, &tmv, smem, full, s, ti, myblk, lane, gh, nr, app && t == nt - 1);
                    if (++t == nt) {  // next (sequence, KV head)
                        t = 0;
                        if (++h == Hkv) {
                            h = 0;
                            cum += static_cast<long long>(nt) * Hkv;
                            ++b;
                            while (b < B) {
                                L = visible_len(a, b, false);
                                if (L > 0) break;
                                ++b;
                            }
                            if (b < B) {
                                nt = (L + kTT - 1) / kTT;
                                table = a.tables + static_cast<size_t>(b) * a.max_blocks;
                            }
                        }
                    }
                }
            }
        } else {
            const int32_t* table = a.tables + static_cast<size_t>(fb_) * a.max_blocks;
            const int ntiles = (t_end - t_begin + kTT - 1) / kTT;
            NewRows<DT, HP> nr;
            bool app = false;
            if constexpr (NQ <= 8) {  // fused append: this split holds the newest position
                app = a.new_k != nullptr && t_end == fL && a.lens[fb_] == fL;
                if (app) nr.prefetch(a, fb_, fh_, lane);
            }
            for (int t = 0; t < ntiles && ok; ++t, ++k) {
                TileInfo ti;
                ti.b = fb_;
                ti.h = fh_;
                ti.L = fL;
                ti.tok0 = t_begin + t * kTT;
                ti.n = min(kTT, t_end - ti.tok0);
                ti.flags = (t == 0 ? kSegFirst : 0) | (t == ntiles - 1 ? kSegLast | kCtaLast : 0) |
                           (a.num_splits == 1 ? kSegWhole : 0) | kCtaFirst;
                ti.pieces = 1;
                ti.c_first = 0;
                ti.s_first = 0;
                const int myblk = tile_blocks(a, table, ti, lane);
                const int s = acquire(k);
                if (!ok) break;
                issue_stage<DT, NQ, HP, kPub>(a, &tmk, &tmv, smem, full, s, ti, myblk, lane, gh, nr, app && t == ntiles - 1);
            }
        }
        if (ok && k == 0) {  // a CTA without tiles: tell the consumers
            if (lane == 0) {
                TileInfo* ti = reinterpret_cast<TileInfo*>(smem + Lt::kInfoOff);
                ti->flags = kEnd;
                mbar_arrive(smem_u32(&full[0]));
            }
            k = 1;
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            if (a.err) atomicOr(a.err, PKV_ERRBIT_TIMEOUT);
        }
        // drain: every issued copy has landed before the CTA may exit
        if (lane == 0) {
            for (long long kk = k - 1; kk >= 0 && kk >= k - kStages; --kk)
                (void)mbar_wait(smem_u32(&full[kk % kStages]), static_cast<uint32_t>((kk / kStages) & 1));
        }
        return;
    }
    if constexpr (kPub) {
        if (warp == kCWarps + 1) {
            publisher<DT, NQ, HP>(a, smem, empty, msg_full, msg_ring, progress, abort_flag, lane, gh, nq);
            return;
        }
    }

    // ---------------------------------------------------------------- consumers
    // warp = (KV head hp of the unit, column group wc, token group wt)
    const int hp = warp / (kCWarps / HP), wi = warp % (kCWarps / HP);
    const int wc = wi % kWC, wt = wi / kWC;
    // this warp's query columns [col0, col_end) and first token of a stage
    const int col0 = HP == 1 ? wc * kNT * 8 : hp * gh;
    const int col_end = HP == 1 ? nq : col0 + gh;
    const int rbase = wt * Lt::kRowsPerWarp;
    const float qk = a.qk_scale_log2;
    // (O and l carry the same probability scale, which cancels in O / l)
    const float vscale = a.v_scale;
    // log-sum-exp of a piece: max + log2(l), less the probability scale
    constexpr float kLseBias = DT == PKV_FP8_E4M3 ? kFp8PLog2 : 0.f;
    const int bsz = a.block_size;
    const uint32_t half_stride = static_cast<uint32_t>(HP * bsz * kBoxRowBytes);
    // m-tile i of call k: rows rbase+16(k*kCallMT+i).. = block row/bs of the tile, rows row%bs.. of it
    uint32_t wb[kCalls][kCallMT];
#pragma unroll
    for (int st = 0; st < kCalls; ++st)
#pragma unroll
        for (int i = 0; i < kCallMT; ++i) {
            const int row = rbase + 16 * (st * kCallMT + i);  // token of the tile; head hp's rows follow head 0's
            wb[st][i] = static_cast<uint32_t>((row / bsz) * kHalves * HP * bsz * kBoxRowBytes +
                                              (hp * bsz + row % bsz) * kBoxRowBytes);
        }
    // causal offset of this lane's columns: query c sees positions < L - C + c + 1
    // (padding columns see the whole tile; decode: offset 0)
    int coff[kNT][2];
#pragma unroll
    for (int j = 0; j < kNT; ++j)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int n = col0 + 8 * j + 2 * (lane & 3) + hh;
            coff[j][hh] = (HP == 1 && n < nq) ? n / gh + 1 - a.num_queries : 0;
        }
    const int d = threadIdx.x;  // 128 consumer threads = 128 head-dim entries
    const LaneOffsets lane_off = lane_offsets<DT>(lane);
    Acc<kNT> acc;
    bool aborted = false;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    // Bounded meeting point of the 4 consumer warps (an mbarrier, so that a
    // warp that gave up on a wait cannot leave the others blocked forever).
    uint32_t cphase = 0;
    auto csync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(csync_bar));
        const bool okw = mbar_wait(smem_u32(csync_bar), cphase, kSpinLimit, abort_flag);
        cphase ^= 1u;
        __syncwarp();
        if (!okw) {
            aborted = true;
            if (lane == 0) {
                *abort_flag = 1;
                if (a.err) atomicOr(a.err, PKV_ERRBIT_TIMEOUT);
            }
        }
        return okw;
    };
    auto release = [&](int s) {
        // generic merge writes before the next TMA fill (with a publisher, a
        // stage with merge writes is freed by it, after that fence)
        if constexpr (kInStage && !kPub) fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    };
    long long nmsg = 0;  // messages posted to the publisher
    auto post = [&](int s) {  // message nmsg: stage s (-1: no tiles)
        const int r = static_cast<int>(nmsg % kStages);
        if (threadIdx.x == 0) msg_ring[r] = s;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&msg_full[r]));
        ++nmsg;
    };

    if constexpr (kBal) {
        // zero the rows of sequences with nothing visible (and report bad
        // lengths once), while the first tiles are in flight
        const int per_seq = a.num_queries * a.num_q_heads;
        for (int b = blockIdx.x; b < a.num_seqs; b += gridDim.x) {
            if (visible_len(a, b, threadIdx.x == 0) == 0) {
                __nv_bfloat16* o = out + (static_cast<size_t>(b) * a.q_total + a.q_first) * a.num_q_heads * kD;
                for (int i = threadIdx.x; i < per_seq * kD; i += kCWarps * 32) o[i] = __float2bfloat16_rn(0.f);
            }
        }
    }
    // test hook: this CTA's first stage wait may be cut short (an expired wait on demand)
    const bool short_first = a.test_wait_on != 0 && (a.test_wait_cta < 0 || a.test_wait_cta == cta_linear());
    for (long long k = 0;; ++k) {
        const int s = static_cast<int>(k % kStages);
        const uint32_t polls = (k == 0 && short_first) ? a.test_wait_polls : kSpinLimit;
        if (!mbar_wait(smem_u32(&full[s]), static_cast<uint32_t>((k / kStages) & 1), polls, abort_flag)) {
            aborted = true;
            if (lane == 0) {
                *abort_flag = 1;
                if (a.err) atomicOr(a.err, PKV_ERRBIT_TIMEOUT);
            }
            break;
        }
        const TileInfo ti = info[s];
        if (ti.flags & kEnd) {
            if constexpr (kPub) post(-1);
            break;
        }
        if constexpr (kPub)
            if (threadIdx.x == 0) *progress = static_cast<int>(k);
        uint8_t* kst = smem + s * Lt::kStageBytes;
        if (ti.flags & kSegFirst)
            acc_begin<DT, kNT>(acc, reinterpret_cast<const __nv_bfloat16*>(smem + Lt::kQOff + s * Lt::kQBytes), lane,
                               col0, col_end, qk);
        int lim[kNT][2];
#pragma unroll
        for (int j = 0; j < kNT; ++j) {
            lim[j][0] = min(ti.n, ti.L + coff[j][0] - ti.tok0);
            lim[j][1] = min(ti.n, ti.L + coff[j][1] - ti.tok0);
        }
#pragma unroll
        for (int st = 0; st < kCalls; ++st)
            consume_tile<DT, kCallMT, kNT>(acc, kst, kst + Lt::kTensorBytes, ti.n, rbase + 16 * kCallMT * st, lane,
                                           wb[st], half_stride, lane_off, lim);
        const bool seg_last = (ti.flags & kSegLast) != 0;
        if (!kInStage || !seg_last) release(s);
        if (!seg_last) continue;

        // ---- segment end: merge the token groups, emit
        if constexpr (kInStage) {  // the stage becomes the merge area once every warp is done reading it
            if (!csync()) break;
        }
        if constexpr (kPub) {  // hand the merge area to the publisher and go on
            const Merge<NQ, kWT> mg(kst, smem + Lt::kStageMlOff + s * Lt::kStageMlBytes);
            merge_put<DT, NQ, kWT, kNT>(acc, mg, wt, col0, col_end, lane);
            fence_proxy_async();  // generic merge writes before the stage's next TMA fill
            post(s);
            if (ti.flags & kCtaLast) break;
            continue;
        }
        const Merge<NQ, kWT> mg(kInStage ? kst : smem + Lt::kMergeOff, smem + Lt::kMlOff);
        merge_put<DT, NQ, kWT, kNT>(acc, mg, wt, col0, col_end, lane);
        if (!csync()) break;
        if (ti.flags & kSegWhole) {
#pragma unroll 4
            for (int n = 0; n < nq; ++n) {
                float v, M, l;
                merge_get<NQ, kWT>(mg, n, d, v, M, l);
                out[out_row<HP>(a, ti.b, ti.h, n, gh) * kD + d] =
                    __float2bfloat16_rn(l > 0.f ? v * (vscale / l) : 0.f);
            }
        } else if constexpr (!kBal) {
#pragma unroll 4
            for (int n = 0; n < nq; ++n) {
                float v, M, l;
                merge_get<NQ, kWT>(mg, n, d, v, M, l);
                // partial rows of this launch: (sequence, query, head)
                const size_t prow = HP == 1 ? (static_cast<size_t>(ti.b) * a.num_queries + n / gh) * a.num_q_heads +
                                                  static_cast<size_t>(ti.h) * gh + n % gh
                                            : static_cast<size_t>(ti.b) * a.num_q_heads + static_cast<size_t>(HP * ti.h) * gh + n;
                a.o_part[(prow * a.num_splits + fsplit) * kD + d] = l > 0.f ? v * (vscale / l) : 0.f;
                if (d == 0) a.lse_part[prow * a.num_splits + fsplit] = l > 0.f ? M + log2f(l) - kLseBias : -INFINITY;
            }
        } else {
            // partial of a (sequence, KV head) shared with other CTAs
            const int slot = (ti.flags & kCtaFirst) ? 0 : 1;
            const size_t pbase = (static_cast<size_t>(blockIdx.x) * 2 + slot) * NQ;
#pragma unroll 4
            for (int n = 0; n < nq; ++n) {
                float v, M, l;
                merge_get<NQ, kWT>(mg, n, d, v, M, l);
                a.bal_o[(pbase + n) * kD + d] = l > 0.f ? v * (vscale / l) : 0.f;
                if (d == 0) a.bal_lse[pbase + n] = l > 0.f ? M + log2f(l) - kLseBias : -INFINITY;
            }
            if constexpr (kInStage) release(s);
            // Publish: after the consumer barrier one GPU-scope acq_rel atomic by
            // thread 0 orders every consumer's partial writes before the count,
            // and (for the last arriver) the other pieces' writes before our reads.
            if (!csync()) break;
            int* counter = a.counters + static_cast<size_t>(ti.b) * a.num_kv_heads + ti.h;
            if (threadIdx.x == 0) *mg.flag = (atom_add_acq_rel(counter, 1) == ti.pieces - 1) ? 1 : 0;
            if (!csync()) break;
            if (*mg.flag) {  // every other piece is published: merge them all
                // pass 1: per row, the largest log-sum-exp M and 1/z, z = sum_j 2^(lse_j - M)
                float* fm = mg.m;  // the merge m/l area is free again: [NQ] M, [NQ] 1/z
                float* fz = mg.m + NQ;
                if (threadIdx.x < nq) {
                    const int n = threadIdx.x;
                    float M = -INFINITY, z = 0.f;
                    for (int j0 = 0; j0 < ti.pieces; j0 += 4) {
                        float l4[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int j = j0 + u;
                            l4[u] = j < ti.pieces
                                        ? __ldcg(a.bal_lse + (static_cast<size_t>(ti.c_first + j) * 2 +
                                                              (j == 0 ? ti.s_first : 0)) * NQ + n)
                                        : -INFINITY;
                        }
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (l4[u] == -INFINITY) continue;  // a piece with no token for this query
                            const float Mn = fmaxf(M, l4[u]);
                            z = z * exp2f(M - Mn) + exp2f(l4[u] - Mn);
                            M = Mn;
                        }
                    }
                    fm[n] = M;
                    fz[n] = z > 0.f ? 1.f / z : 0.f;
                }
                if (!csync()) break;
                // pass 2: thread t owns 4-float chunks t, t+128, ... of the rows
                // (32 chunks per row); one round of independent loads per piece
                constexpr int kC = (NQ * (kD / 4) + kCWarps * 32 - 1) / (kCWarps * 32);
                float4 acc4[kC];
#pragma unroll
                for (int c = 0; c < kC; ++c) acc4[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int j = 0; j < ti.pieces; ++j) {
                    const size_t pb = (static_cast<size_t>(ti.c_first + j) * 2 + (j == 0 ? ti.s_first : 0)) * NQ;
#pragma unroll
                    for (int c = 0; c < kC; ++c) {
                        const int idx = threadIdx.x + c * kCWarps * 32, n = idx >> 5, d4 = idx & 31;
                        if (n >= nq) continue;
                        const float lj = __ldcg(a.bal_lse + pb + n);
                        const float4 o4 = __ldcg(reinterpret_cast<const float4*>(a.bal_o + (pb + n) * kD) + d4);
                        const float w = lj == -INFINITY ? 0.f : exp2f(lj - fm[n]) * fz[n];
                        acc4[c].x = fmaf(w, o4.x, acc4[c].x);
                        acc4[c].y = fmaf(w, o4.y, acc4[c].y);
                        acc4[c].z = fmaf(w, o4.z, acc4[c].z);
                        acc4[c].w = fmaf(w, o4.w, acc4[c].w);
                    }
                }
#pragma unroll
                for (int c = 0; c < kC; ++c) {
                    const int idx = threadIdx.x + c * kCWarps * 32, n = idx >> 5, d4 = idx & 31;
                    if (n >= nq) continue;
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc4[c].x, acc4[c].y);
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc4[c].z, acc4[c].w);
                    uint2 pk;
                    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
                    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
                    *reinterpret_cast<uint2*>(out + out_row<HP>(a, ti.b, ti.h, n, gh) * kD + 4 * d4) = pk;
                }
                if (threadIdx.x == 0) *counter = 0;  // ready for the next call
                // pass 2 read M and 1/z from the merge m/l area: a warp that
                // runs ahead must not put its next segment there before every
                // warp is through (nothing follows the CTA's last segment)
                if (!(ti.flags & kCtaLast) && !csync()) break;
            }
            // otherwise every consumer read the merge area before the second
            // barrier, so the next segment may overwrite it without another
            if (ti.flags & kCtaLast) break;
            continue;
        }
        if constexpr (kInStage) {
            release(s);  // the next segment merges in another stage, or in this one once refilled
        } else {
            if (!csync()) break;  // the dedicated merge area is reused by the next segment
        }
        if (ti.flags & kCtaLast) break;
    }
}

template <int DT, int NQ, bool kBal, int HP = 1>
cudaError_t launch_nq(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    constexpr bool kPub = kPubOf<DT, kBal>;
    using Lt = Layout<DT, NQ, HP, kPub>;
    constexpr size_t smem = Lt::kAlloc;
    auto kern = decode_mma_kernel<DT, NQ, kBal, HP>;
    static int configured_mask = 0;
    static int ctas_per_sm[32] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 31) return cudaErrorNotSupported;
    if (!(configured_mask & (1 << dev))) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        // ask for the largest shared-memory carveout so that two CTAs fit per SM
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        int occ = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreadsOf<kPub>, smem);
        if (e != cudaSuccess) return e;
        ctas_per_sm[dev] = occ > 0 ? occ : 1;
        configured_mask |= 1 << dev;
    }
    dim3 grid;
    if constexpr (kBal) {
        const int P = num_sms() * ctas_per_sm[dev];
        grid = dim3(P < a.bal_max_ctas ? P : a.bal_max_ctas);
    } else {
        grid = dim3(a.num_splits, a.num_kv_heads / HP, a.num_seqs);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreadsOf<kPub>);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the previous kernel drains
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, a);
}

// Smallest template row bound that holds this launch's query rows.
template <int DT, bool kBal>
cudaError_t launch_rows(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    const int rows = a.num_queries * (a.num_q_heads / a.num_kv_heads);
    if constexpr (DT == PKV_BF16) {
        if (a.heads_per_cta == 2) {  // a KV-head pair: 2 * rows columns
            if (a.num_queries != 1 || a.num_kv_heads % 2 != 0) return cudaErrorNotSupported;
            if (rows <= 1) return launch_nq<DT, 2, kBal, 2>(a, tk, tv, stream);
            if (rows <= 2) return launch_nq<DT, 4, kBal, 2>(a, tk, tv, stream);
            if (rows <= 4) return launch_nq<DT, 8, kBal, 2>(a, tk, tv, stream);
            return cudaErrorNotSupported;
        }
    }
    if (a.heads_per_cta != 1) return cudaErrorNotSupported;
    if (rows <= 1) return launch_nq<DT, 1, kBal>(a, tk, tv, stream);
    if (rows <= 2) return launch_nq<DT, 2, kBal>(a, tk, tv, stream);
    if (rows <= 4) return launch_nq<DT, 4, kBal>(a, tk, tv, stream);
    if (rows <= 8) return launch_nq<DT, 8, kBal>(a, tk, tv, stream);
    if (rows <= 16) return launch_nq<DT, 16, kBal>(a, tk, tv, stream);
    if (rows <= 32) return launch_nq<DT, 32, kBal>(a, tk, tv, stream);
    if (rows <= 64) return launch_nq<DT, 64, kBal>(a, tk, tv, stream);
    return cudaErrorNotSupported;
}

template <int DT>
cudaError_t launch_dt(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    return a.bal_max_ctas > 0 ? launch_rows<DT, true>(a, tk, tv, stream) : launch_rows<DT, false>(a, tk, tv, stream);
}

}  // namespace
}  // namespace pkv
