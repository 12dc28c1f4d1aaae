// Paged decode attention, tensor-core design (BF16 and FP8-E4M3 pools,
// head_dim 128).  The B operand holds the NQ = C * G query rows of one KV head:
// G query heads (grouped-query attention) times C queries per sequence (C = 1
// for decode; C > 1 verifies drafted tokens or processes a prompt chunk: the
// last C tokens of the sequence, each attending causally), NQ in {1, 2, 4, 8}.
//
// "How does TensorRT-LLM work?", "Custom attention kernels": one kernel does
// the whole attention step and keeps the intermediate scores on chip.
// "Introduction to TensorRT-LLM", figure "TensorRT-LLM Acceleration Stack":
// Flash-Decoding splits the key/value length across CTAs and merges the
// pieces by their log-sum-exp.
//
// Work is a list of 64-token tiles of (sequence, KV head) pairs.  Two
// schedules share the same producer and consumer code:
//  * balanced (the default): a persistent grid of 2 CTAs per SM; CTA c takes
//    the contiguous tile range [c*T/P, (c+1)*T/P) of the flattened list
//    (T tiles, P CTAs), so every CTA streams the same number of KV bytes
//    whatever the length mix.  A (sequence, KV head) whose tiles straddle
//    CTAs leaves one fp32 partial per CTA; the CTA that finishes that pair
//    last (an atomic counter in the workspace, no waiting) merges the
//    partials by their log-sum-exp and writes the output.
//  * fixed splits (when the caller names a split size): one CTA per
//    (split, KV head, sequence); partials go to the combine kernel.
// CTA = 4 consumer warps + 1 producer warp.
//  * Producer: one lane walks the block table and issues, per 64-token stage,
//    one TMA tile load (cp.async.bulk.tensor, 128-byte swizzle) per block of
//    K and of V: for BF16 a 3D box {64 columns, bs rows, 2 halves} fetches a
//    block's whole 256-byte rows at once (two 2D boxes if the driver refuses
//    that descriptor).  At the first tile of a segment it also bulk-copies the
//    G query rows into the stage.  A full mbarrier counts the bytes, an empty
//    mbarrier (4 arrivals) frees the stage; a per-stage TileInfo tells the
//    consumers what the stage holds and marks the CTA's last tile.
//    Every KV byte crosses HBM once; the G query heads of a KV head share it.
//  * Consumer warp w owns tokens [16w, 16w+16) of each stage:
//      S^T[16 tok x 8] = K[16 x 128] . Q^T[128 x 8]   8 x mma.m16n8k16
//      (tokens fill M; the G query heads fill N, padded to 8)
//      online softmax on the fragment (3 shuffles per max, exp2 with the
//      scale*log2(e) folded in), P packed to 16 bits and transposed in
//      registers with movmatrix into the B operand of
//      O^T[128 x 8] += V^T[128 x 16 tok] . P^T[16 tok x 8]  8 x mma
//      (V^T through ldmatrix.trans for BF16).
//  * FP8 pools: E4M3 converts exactly to f16 in registers and the mma runs
//    f16 x f16 -> f32.  K is read with ldmatrix and the head_dim order is
//    permuted consistently in K and Q (a dot product does not depend on the
//    order of its terms); V^T pairs two tokens' bytes with one byte_perm.
//    Q is converted from BF16 to f16 (exact for |q| in [2^-14, 65504]).
//  * At a segment's end the 4 warps' (m, l, O) are merged through shared
//    memory and the CTA writes the final row or its fp32 partial.
// Rows past the sequence end inside a loaded block are masked in S and zeroed
// in V (uninitialised pool bytes could hold NaN patterns, and 0 * NaN = NaN).
// Every mbarrier wait is bounded; on expiry the CTA flags PKV_ERRBIT_TIMEOUT,
// drains its in-flight copies (bounded) and skips its output.
#include <cuda.h>

#include "device_common.cuh"

namespace pkv {
namespace {

constexpr int kCWarps = 4;
constexpr int kMmaThreads = (kCWarps + 1) * 32;
constexpr int kBoxRowBytes = 128;          // one swizzled TMA row
constexpr int kD = 128;                    // head_dim served by this design
constexpr uint32_t kSpinLimit = 1u << 22;  // try_wait polls before a wait gives up

template <int DT>
struct MmaCfg;
template <>
struct MmaCfg<PKV_BF16> {
    static constexpr int kHalves = 2;  // 128 columns = two 64-column (128-byte) halves
    static constexpr int kStages = 3;
    static constexpr int kMT = 1;      // 16-token m-tiles per consumer warp per stage
};
template <>
struct MmaCfg<PKV_FP8_E4M3> {
    static constexpr int kHalves = 1;  // 128 one-byte columns = one 128-byte row
    static constexpr int kStages = 3;
    static constexpr int kMT = 2;      // two independent m-tiles per warp: half the bytes per token need more ILP
};

// What one pipeline stage holds.
struct TileInfo {
    int b, h;       // sequence, KV head
    int L;          // the sequence's length
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
constexpr int kCtaLast = 32;  // the CTA's last tile

// Shared memory of one CTA (a stage holds kTT = 64 * kMT tokens):
//   stages: [kStages][K, V][block of the tile][half][bs rows][128 B]
//     A block's two halves (head_dim 0-63 and 64-127 for BF16) are bs*128
//     bytes apart; both start on 1024-byte boundaries (bs >= 16), so the
//     128-byte swizzle phase of a row is its row index within the block, mod 8.
//   q slots [kStages][G][128] BF16, tile info [kStages],
//   merge area [warp][G][128] O + [warp][G] m, l, + one flag word,
//   barriers full[kStages], empty[kStages], consumer sync, abort word.
template <int DT, int G>
struct Layout {
    static constexpr int kHalves = MmaCfg<DT>::kHalves;
    static constexpr int kStages = MmaCfg<DT>::kStages;
    static constexpr int kMT = MmaCfg<DT>::kMT;
    static constexpr int kTT = 16 * kCWarps * kMT;  // tokens per stage
    static constexpr int kTensorBytes = kHalves * kTT * kBoxRowBytes;
    static constexpr int kStageBytes = 2 * kTensorBytes;
    static constexpr int kQBytes = G * kD * 2;
    static constexpr size_t kQOff = static_cast<size_t>(kStages) * kStageBytes;
    static constexpr size_t kInfoOff = kQOff + static_cast<size_t>(kStages) * kQBytes;
    static constexpr size_t kMergeOff = kInfoOff + static_cast<size_t>(kStages) * sizeof(TileInfo);
    static constexpr size_t kMergeBytes = (static_cast<size_t>(kCWarps) * G * (kD + 2) + 4) * 4;
    static constexpr size_t kBarOff = (kMergeOff + kMergeBytes + 15) / 16 * 16;
    static constexpr size_t kBytes = kBarOff + (2 * kStages + 1) * 8 + 16;
    static constexpr size_t kAlloc = kBytes + 1024;  // + alignment slack
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
// Bounded wait for the phase with the given parity to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
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
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
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

// Two E4M3 codes (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
    __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two & 0xFFFFu), __NV_E4M3);
    return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

// Byte offset of 16-byte chunk `chunk` of row `lr` inside a 128B-swizzled run
// of rows whose first row sits on a 1024-byte boundary (and is a multiple of 8
// rows into the run).
__device__ __forceinline__ uint32_t swz(int lr, int chunk) {
    return static_cast<uint32_t>(lr * kBoxRowBytes + ((chunk ^ (lr & 7)) << 4));
}

// Head-dim index held by O^T accumulator row `m` (0..15) of m-tile `mt`.
template <int DT>
__device__ __forceinline__ int o_dim(int mt, int m) {
    if constexpr (DT == PKV_BF16) {
        return mt * 16 + m;
    } else {  // m-tiles (2j, 2j+1) rows (r, r+8) -> 32j + 4r + {0,1,2,3}
        const int j = mt >> 1, r = m & 7;
        return 32 * j + 4 * r + ((mt & 1) << 1) + (m >> 3);
    }
}

// ---------------------------------------------------------------- consumers
template <int DT>
struct Acc {
    float m0, m1, l0, l1;  // running max (log2 domain) and lane-partial sums, heads 2q and 2q+1
    float o[8][4];         // O^T accumulator fragments
    uint32_t bq[8][2];     // Q^T as the mma B operand
};

// Start a segment: clear the state and build the Q^T fragments from the
// stage's query rows qs[G][128] (BF16, shared memory).
template <int DT, int G>
__device__ __forceinline__ void acc_begin(Acc<DT>& s, const __nv_bfloat16* qs, int lane) {
    s.m0 = s.m1 = -INFINITY;
    s.l0 = s.l1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) s.o[mt][0] = s.o[mt][1] = s.o[mt][2] = s.o[mt][3] = 0.f;
    const int r = lane >> 2, q = lane & 3;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
        if (r >= G) {
            s.bq[ks][0] = s.bq[ks][1] = 0u;
            continue;
        }
        if constexpr (DT == PKV_BF16) {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(qs + r * kD + ks * 16 + 2 * q);
            s.bq[ks][0] = w[0];
            s.bq[ks][1] = w[4];  // +8 elements
        } else {  // head_dim order permuted like K's: chunk ks, bytes 4q..4q+3
            const __nv_bfloat16* p = qs + r * kD + ks * 16 + 4 * q;
            s.bq[ks][0] = pack2<DT>(__bfloat162float(p[0]), __bfloat162float(p[1]));
            s.bq[ks][1] = pack2<DT>(__bfloat162float(p[2]), __bfloat162float(p[3]));
        }
    }
}

// Per-lane byte offsets (relative to the warp's first row in a tensor of a
// stage) of the shared-memory fragments a consumer lane reads every tile;
// they depend only on the lane, so they are computed once.
struct LaneOffsets {
    uint32_t k[4];  // K ldmatrix rows: chunk pair i (BF16: + half * half_stride)
    uint32_t v[8];  // BF16: V ldmatrix.trans, chunk pair i (4 used); FP8: V bytes, (j, row ta / ta+1)
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
#pragma unroll
        for (int i = 4; i < 8; ++i) o.v[i] = 0;
    } else {
        const int r = lane >> 2, q = lane & 3;
        const uint32_t inner = static_cast<uint32_t>((r & 3) * 4);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            o.v[2 * j] = swz(2 * q, 2 * j + (r >> 2)) + inner;
            o.v[2 * j + 1] = swz(2 * q + 1, 2 * j + (r >> 2)) + inner;
        }
    }
    return o;
}

// One stage for this warp's MT m-tiles of 16 rows, [row0, row0 + 16*MT)
// (n valid rows in the stage).  wb[i]: byte offset of m-tile i's first row in
// a tensor of the stage; half_stride: bytes between a block's two 64-column
// halves.  The m-tiles' S chains are interleaved and share one softmax update.
// lim0 / lim1: rows of the tile visible to this lane's two query columns
// (2q, 2q+1); both <= n, and equal to n for single-query decode.
template <int DT, int MT>
__device__ __forceinline__ void consume_tile(Acc<DT>& s, uint8_t* kst, uint8_t* vst, int n, int row0, int lane,
                                             const uint32_t (&wb)[MT], uint32_t half_stride, float qk,
                                             const LaneOffsets& lo, int lim0, int lim1) {
    constexpr int kHalves = MmaCfg<DT>::kHalves;
    if (row0 >= n) return;
    const int r = lane >> 2;
    if (n < row0 + 16 * MT) {  // zero this warp's V rows past the end
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
    // ---- S^T = K Q^T, m-tiles interleaved
    float sc[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
    const uint32_t kb = smem_u32(kst);
    if constexpr (DT == PKV_BF16) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                if (!live[i]) continue;
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kb + wb[i] + (ks >> 2) * half_stride + lo.k[ks & 3], a0, a1, a2, a3);
                mma16816<DT>(sc[i], a0, a1, a2, a3, s.bq[ks][0], s.bq[ks][1]);
            }
        }
    } else {
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {  // two k-steps (chunks 2kp, 2kp+1) per ldmatrix.x4
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                if (!live[i]) continue;
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kb + wb[i] + lo.k[kp], r0, r1, r2, r3);
                mma16816<DT>(sc[i], e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                             e4m3x2_to_f16x2(r1 >> 16), s.bq[2 * kp][0], s.bq[2 * kp][1]);
                mma16816<DT>(sc[i], e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                             e4m3x2_to_f16x2(r3 >> 16), s.bq[2 * kp + 1][0], s.bq[2 * kp + 1][1]);
            }
        }
    }
    // ---- online softmax (log2 domain) over the warp's 16*MT rows
    float sv[MT][4];
    float x0 = -INFINITY, x1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        const int ra = row0 + 16 * i + r, rb = ra + 8;
        sv[i][0] = ra < lim0 ? sc[i][0] * qk : -INFINITY;
        sv[i][1] = ra < lim1 ? sc[i][1] * qk : -INFINITY;
        sv[i][2] = rb < lim0 ? sc[i][2] * qk : -INFINITY;
        sv[i][3] = rb < lim1 ? sc[i][3] * qk : -INFINITY;
        x0 = fmaxf(x0, fmaxf(sv[i][0], sv[i][2]));
        x1 = fmaxf(x1, fmaxf(sv[i][1], sv[i][3]));
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        x0 = fmaxf(x0, __shfl_xor_sync(0xFFFFFFFFu, x0, off));
        x1 = fmaxf(x1, __shfl_xor_sync(0xFFFFFFFFu, x1, off));
    }
    const float n0 = fmaxf(s.m0, x0), n1 = fmaxf(s.m1, x1);
    // a column that has seen no token yet keeps max -inf and weights 0
    const float b0 = n0 == -INFINITY ? 0.f : n0, b1 = n1 == -INFINITY ? 0.f : n1;
    float p[MT][4];
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        p[i][0] = exp2f(sv[i][0] - b0);
        p[i][1] = exp2f(sv[i][1] - b1);
        p[i][2] = exp2f(sv[i][2] - b0);
        p[i][3] = exp2f(sv[i][3] - b1);
    }
    // rescale only when some head's running max moved (the factor is exactly 1 otherwise)
    if (__any_sync(0xFFFFFFFFu, n0 != s.m0 || n1 != s.m1)) {
        // against b0/b1: a column still without tokens (both maxima -inf) gets 0, not 2^NaN
        const float al0 = exp2f(s.m0 - b0), al1 = exp2f(s.m1 - b1);
        s.l0 *= al0;
        s.l1 *= al1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            s.o[mt][0] *= al0;
            s.o[mt][1] *= al1;
            s.o[mt][2] *= al0;
            s.o[mt][3] *= al1;
        }
    }
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        s.l0 += p[i][0] + p[i][2];
        s.l1 += p[i][1] + p[i][3];
    }
    s.m0 = n0;
    s.m1 = n1;
    uint32_t pb[MT][2];
#pragma unroll
    for (int i = 0; i < MT; ++i) {
        pb[i][0] = movmatrix_t(pack2<DT>(p[i][0], p[i][1]));  // tokens 0-7 of m-tile i
        pb[i][1] = movmatrix_t(pack2<DT>(p[i][2], p[i][3]));  // tokens 8-15
    }
    // ---- O^T += V^T P^T
    const uint32_t vb0 = smem_u32(vst);
    if constexpr (DT == PKV_BF16) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                if (!live[i]) continue;
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vb0 + wb[i] + (mt >> 2) * half_stride + lo.v[mt & 3], a0, a1, a2, a3);
                mma16816<DT>(s.o[mt], a0, a1, a2, a3, pb[i][0], pb[i][1]);
            }
        }
    } else {
        // rows ta, ta+1 (ta = 2q) at offsets v[2j], v[2j+1]; rows ta+8, ta+9 are 8 rows (1024 B) further
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                if (!live[i]) continue;
                const uint32_t vb_ = vb0 + wb[i];
                const uint32_t w0 = lds32(vb_ + lo.v[2 * j]);
                const uint32_t w1 = lds32(vb_ + lo.v[2 * j + 1]);
                const uint32_t w8 = lds32<8 * kBoxRowBytes>(vb_ + lo.v[2 * j]);
                const uint32_t w9 = lds32<8 * kBoxRowBytes>(vb_ + lo.v[2 * j + 1]);
                const uint32_t x01 = __byte_perm(w0, w1, 0x5140), x23 = __byte_perm(w0, w1, 0x7362);
                const uint32_t y01 = __byte_perm(w8, w9, 0x5140), y23 = __byte_perm(w8, w9, 0x7362);
                mma16816<DT>(s.o[2 * j], e4m3x2_to_f16x2(x01), e4m3x2_to_f16x2(x01 >> 16), e4m3x2_to_f16x2(y01),
                             e4m3x2_to_f16x2(y01 >> 16), pb[i][0], pb[i][1]);
                mma16816<DT>(s.o[2 * j + 1], e4m3x2_to_f16x2(x23), e4m3x2_to_f16x2(x23 >> 16),
                             e4m3x2_to_f16x2(y23), e4m3x2_to_f16x2(y23 >> 16), pb[i][0], pb[i][1]);
            }
        }
    }
}

// Merge area: O [warp][G][128], m [warp][G], l [warp][G], one flag word.
template <int G>
struct Merge {
    float* o;
    float* m;
    float* l;
    volatile int* flag;
    __device__ explicit Merge(uint8_t* base) {
        o = reinterpret_cast<float*>(base);
        m = o + kCWarps * G * kD;
        l = m + kCWarps * G;
        flag = reinterpret_cast<volatile int*>(l + kCWarps * G);
    }
};

// Publish this warp's (m, l, O) for the G real heads.
template <int DT, int G>
__device__ __forceinline__ void merge_put(const Acc<DT>& s, const Merge<G>& mg, int warp, int lane) {
    const int r = lane >> 2, q = lane & 3;
    float l0 = s.l0, l1 = s.l1;
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
    }
    const int h0 = 2 * q, h1 = 2 * q + 1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        if (h0 < G) {
            mg.o[(warp * G + h0) * kD + o_dim<DT>(mt, r)] = s.o[mt][0];
            mg.o[(warp * G + h0) * kD + o_dim<DT>(mt, r + 8)] = s.o[mt][2];
        }
        if (h1 < G) {
            mg.o[(warp * G + h1) * kD + o_dim<DT>(mt, r)] = s.o[mt][1];
            mg.o[(warp * G + h1) * kD + o_dim<DT>(mt, r + 8)] = s.o[mt][3];
        }
    }
    if (lane < 4) {
        if (h0 < G) {
            mg.m[warp * G + h0] = s.m0;
            mg.l[warp * G + h0] = l0;
        }
        if (h1 < G) {
            mg.m[warp * G + h1] = s.m1;
            mg.l[warp * G + h1] = l1;
        }
    }
}

// Merged (sum O, max m, sum l) of head g at head-dim index d.
template <int G>
__device__ __forceinline__ void merge_get(const Merge<G>& mg, int g, int d, float& acc, float& M, float& lsum) {
    M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCWarps; ++w) M = fmaxf(M, mg.m[w * G + g]);
    acc = 0.f;
    lsum = 0.f;
    if (M == -INFINITY) return;  // no token for this query in the segment
#pragma unroll
    for (int w = 0; w < kCWarps; ++w) {
        const float f = exp2f(mg.m[w * G + g] - M);  // warps without rows: 2^-inf = 0
        acc += f * mg.o[(w * G + g) * kD + d];
        lsum += f * mg.l[w * G + g];
    }
}

// ---------------------------------------------------------------- producer
// Stage s <- tile ti: tile info, the query rows at a segment's first tile,
// and one TMA box per KV block (K and V).  All 32 producer lanes call it
// (they share the block-table window); lane 0 issues.
template <int DT, int G>
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, const CUtensorMap* tmk, const CUtensorMap* tmv,
                                            uint8_t* smem, uint64_t* full, int s, const TileInfo& ti,
                                            const int32_t* table, int& cache, int& cache_base, int lane) {
    using Lt = Layout<DT, G>;
    const int bs = a.block_size;
    uint8_t* kst = smem + s * Lt::kStageBytes;
    uint8_t* vst = kst + Lt::kTensorBytes;
    const uint32_t fb = smem_u32(&full[s]);
    const int nblk = (ti.n + bs - 1) / bs;
    const bool need_q = (ti.flags & kSegFirst) != 0;
    if (lane == 0) {
        reinterpret_cast<TileInfo*>(smem + Lt::kInfoOff)[s] = ti;
        mbar_expect_tx(fb, static_cast<uint32_t>(nblk * bs * kBoxRowBytes * Lt::kHalves * 2 +
                                                 (need_q ? Lt::kQBytes : 0)));
        if (need_q) {  // query rows n = c * gh + g: C copies of gh contiguous rows
            const int C = a.num_queries, gh = G / C;
            for (int c = 0; c < C; ++c) {
                const __nv_bfloat16* qsrc =
                    static_cast<const __nv_bfloat16*>(a.q) +
                    ((static_cast<size_t>(ti.b) * C + c) * a.num_q_heads + static_cast<size_t>(ti.h) * gh) * kD;
                bulk_load(smem_u32(smem + Lt::kQOff + s * Lt::kQBytes + c * gh * kD * 2), qsrc,
                          static_cast<uint32_t>(gh * kD * 2), fb);
            }
        }
    }
    const int64_t layer_blk0 = static_cast<int64_t>(a.layer) * a.num_blocks;
    for (int k = 0; k < nblk; ++k) {
        const int j = ti.tok0 / bs + k;  // block index within the sequence
        if (cache_base < 0 || j - cache_base >= 32 || j < cache_base) {
            cache_base = j & ~31;
            const int idx = cache_base + lane;
            cache = idx < a.max_blocks ? table[idx] : -1;
        }
        int blk = __shfl_sync(0xFFFFFFFFu, cache, j - cache_base);
        if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.num_blocks)) {
            if (lane == 0 && a.err) atomicOr(a.err, PKV_ERRBIT_BLOCK_ID);
            blk = 0;  // read an in-bounds block; the flag marks the output invalid
        }
        if (lane == 0) {
            const int y = static_cast<int>(((layer_blk0 + blk) * a.num_kv_heads + ti.h) * bs);
            const uint32_t off = k * Lt::kHalves * bs * kBoxRowBytes;
            if (Lt::kHalves == 2 && a.tma_3d) {  // one box: both 128-byte halves of every row
                tma_load_3d(smem_u32(kst + off), tmk, 0, y, 0, fb);
                tma_load_3d(smem_u32(vst + off), tmv, 0, y, 0, fb);
            } else {
                for (int hf = 0; hf < Lt::kHalves; ++hf) {
                    const uint32_t o2 = off + hf * bs * kBoxRowBytes;
                    tma_load_2d(smem_u32(kst + o2), tmk, hf * 64, y, fb);
                    tma_load_2d(smem_u32(vst + o2), tmv, hf * 64, y, fb);
                }
            }
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
    return b < a.num_seqs ? (clamped_len(a, b, false) + kTT - 1) / kTT : 0;
}

// kBal: balanced persistent schedule (grid = P CTAs); otherwise one CTA per
// (split, KV head, sequence) with grid (num_splits, num_kv_heads, num_seqs).
template <int DT, int G, bool kBal>
__global__ void __launch_bounds__(kMmaThreads, 2)
decode_mma_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
    using Lt = Layout<DT, G>;
    constexpr int kStages = Lt::kStages;
    constexpr int kHalves = Lt::kHalves;
    constexpr int kMT = Lt::kMT;
    constexpr int kTT = Lt::kTT;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Lt::kBarOff);
    uint64_t* empty = full + kStages;
    uint64_t* csync_bar = empty + kStages;  // the 4 consumer warps meet here at segment ends
    volatile int* abort_flag = reinterpret_cast<volatile int*>(csync_bar + 1);
    const TileInfo* info = reinterpret_cast<const TileInfo*>(smem + Lt::kInfoOff);
    const Merge<G> mg(smem + Lt::kMergeOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Launched as a programmatic dependent of the previous kernel in the
    // stream (the append): nothing is read before that grid has finished.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");

    // fixed schedule: this CTA's one segment
    int fb_ = 0, fh_ = 0, fsplit = 0, t_begin = 0, t_end = 0, fL = 0;
    if constexpr (!kBal) {
        fsplit = blockIdx.x;
        fh_ = blockIdx.y;
        fb_ = blockIdx.z;
        const int L = clamped_len(a, fb_, fsplit == 0 && fh_ == 0 && threadIdx.x == 0);
        fL = L;
        t_begin = fsplit * a.split_tokens;
        t_end = min(L, t_begin + a.split_tokens);
        if (t_begin >= t_end) {
            if (a.num_splits == 1) {  // empty sequence: zero output rows
                const int C = a.num_queries, gh = G / C;
                for (int i = threadIdx.x; i < G * kD; i += kMmaThreads) {
                    const int nq = i / kD, c = nq / gh, g = nq % gh;
                    static_cast<__nv_bfloat16*>(a.out)[((static_cast<size_t>(fb_) * C + c) * a.num_q_heads +
                                                        fh_ * gh + g) * kD + i % kD] = __float2bfloat16_rn(0.f);
                }
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
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    if (warp == kCWarps) {
        // ------------------------------------------------------------ producer
        int cache = -1, cache_base = -1;
        long long k = 0;  // stages issued
        bool ok = true;
        auto acquire = [&](long long kk) -> int {  // stage for the kk-th issue, after it is free
            const int s = static_cast<int>(kk % kStages);
            if (kk >= kStages && ok) ok = mbar_wait(smem_u32(&empty[s]), static_cast<uint32_t>(((kk / kStages) - 1) & 1));
            if (*abort_flag) ok = false;
            return s;
        };
        if constexpr (kBal) {
            const int B = a.num_seqs, Hkv = a.num_kv_heads;
            long long T = 0;
#pragma unroll 4
            for (int b0 = 0; b0 < B; b0 += 32) T += warp_sum_ll(seq_tiles<kTT>(a, b0 + lane));
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
                    const long long u = static_cast<long long>(seq_tiles<kTT>(a, b0 + lane)) * Hkv;
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
                int L = clamped_len(a, b, false);
                int nt = (L + kTT - 1) / kTT;
                const long long off = g0 - cum;
                int h = static_cast<int>(off / nt), t = static_cast<int>(off % nt);
                const int32_t* table = a.tables + static_cast<size_t>(b) * a.max_blocks;
                auto owner = [&](long long g) { return ((g + 1) * P - 1) / T; };
                TileInfo ti;
                for (long long g = g0; g < g1 && ok; ++g, ++k) {
                    const int s = acquire(k);
                    if (!ok) break;
                    const long long pstart = cum + static_cast<long long>(h) * nt, pend = pstart + nt;
                    if (g == g0 || t == 0) {  // a new segment: who shares this (sequence, KV head)
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
                    issue_stage<DT, G>(a, &tmk, &tmv, smem, full, s, ti, table, cache, cache_base, lane);
                    if (++t == nt) {  // next (sequence, KV head)
                        t = 0;
                        if (++h == Hkv) {
                            h = 0;
                            cum += static_cast<long long>(nt) * Hkv;
                            ++b;
                            while (b < B) {
                                L = clamped_len(a, b, false);
                                if (L > 0) break;
                                ++b;
                            }
                            if (b < B) {
                                nt = (L + kTT - 1) / kTT;
                                table = a.tables + static_cast<size_t>(b) * a.max_blocks;
                                cache_base = -1;
                            }
                        }
                    }
                }
            }
        } else {
            const int32_t* table = a.tables + static_cast<size_t>(fb_) * a.max_blocks;
            const int ntiles = (t_end - t_begin + kTT - 1) / kTT;
            for (int t = 0; t < ntiles && ok; ++t, ++k) {
                const int s = acquire(k);
                if (!ok) break;
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
                issue_stage<DT, G>(a, &tmk, &tmv, smem, full, s, ti, table, cache, cache_base, lane);
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

    // ---------------------------------------------------------------- consumers
    const int row0 = warp * 16 * kMT;
    const float qk = a.qk_scale_log2;
    const int bsz = a.block_size;
    const uint32_t half_stride = static_cast<uint32_t>(bsz * kBoxRowBytes);
    // this warp's m-tile i: rows row0+16i.. = block (row0+16i)/bs of the tile, rows (row0+16i)%bs.. of it
    uint32_t wb[kMT];
#pragma unroll
    for (int i = 0; i < kMT; ++i)
        wb[i] = static_cast<uint32_t>(((row0 + 16 * i) / bsz) * kHalves * bsz * kBoxRowBytes +
                                      ((row0 + 16 * i) % bsz) * kBoxRowBytes);
    const int d = threadIdx.x;  // 128 consumer threads = 128 head-dim entries
    const LaneOffsets lane_off = lane_offsets<DT>(lane);
    Acc<DT> acc;
    bool aborted = false;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
    // Bounded meeting point of the 4 consumer warps (an mbarrier, so that a
    // warp that gave up on a wait cannot leave the others blocked forever).
    uint32_t cphase = 0;
    auto csync = [&]() -> bool {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(csync_bar));
        const bool okw = mbar_wait(smem_u32(csync_bar), cphase);
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

    for (long long k = 0;; ++k) {
        const int s = static_cast<int>(k % kStages);
        if (!mbar_wait(smem_u32(&full[s]), static_cast<uint32_t>((k / kStages) & 1))) {
            aborted = true;
            if (lane == 0) {
                *abort_flag = 1;
                if (a.err) atomicOr(a.err, PKV_ERRBIT_TIMEOUT);
            }
            break;
        }
        const TileInfo ti = info[s];
        if (ti.flags & kEnd) break;
        uint8_t* kst = smem + s * Lt::kStageBytes;
        if (ti.flags & kSegFirst)
            acc_begin<DT, G>(acc, reinterpret_cast<const __nv_bfloat16*>(smem + Lt::kQOff + s * Lt::kQBytes), lane);
        // causal limit of this lane's columns (2q, 2q+1): query c sees positions < L - C + c + 1
        int lim0 = ti.n, lim1 = ti.n;
        if (a.num_queries > 1) {
            const int gh = G / a.num_queries, q2 = (lane & 3) * 2;
            if (q2 < G) lim0 = min(ti.n, ti.L - a.num_queries + q2 / gh + 1 - ti.tok0);
            if (q2 + 1 < G) lim1 = min(ti.n, ti.L - a.num_queries + (q2 + 1) / gh + 1 - ti.tok0);
        }
        consume_tile<DT, kMT>(acc, kst, kst + Lt::kTensorBytes, ti.n, row0, lane, wb, half_stride, qk, lane_off,
                              lim0, lim1);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
        if (!(ti.flags & kSegLast)) continue;

        // ---- segment end: merge the 4 warps, emit
        merge_put<DT, G>(acc, mg, warp, lane);
        if (!csync()) break;
        // output row of query column g: (sequence, query c, head h*gh + g % gh)
        const int Cq = a.num_queries, gh = G / Cq;
        auto qrow = [&](int g) -> size_t {
            return (static_cast<size_t>(ti.b) * Cq + g / gh) * a.num_q_heads + static_cast<size_t>(ti.h) * gh + g % gh;
        };
        if (ti.flags & kSegWhole) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v, M, l;
                merge_get<G>(mg, g, d, v, M, l);
                out[qrow(g) * kD + d] = __float2bfloat16_rn(l > 0.f ? v * (a.v_scale / l) : 0.f);
            }
        } else if constexpr (!kBal) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v, M, l;
                merge_get<G>(mg, g, d, v, M, l);
                a.o_part[(qrow(g) * a.num_splits + fsplit) * kD + d] = l > 0.f ? v * (a.v_scale / l) : 0.f;
                if (d == 0) a.lse_part[qrow(g) * a.num_splits + fsplit] = l > 0.f ? M + log2f(l) : -INFINITY;
            }
        } else {
            // partial of a (sequence, KV head) shared with other CTAs
            const int slot = (ti.flags & kCtaFirst) ? 0 : 1;
            const size_t pbase = (static_cast<size_t>(blockIdx.x) * 2 + slot) * G;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float v, M, l;
                merge_get<G>(mg, g, d, v, M, l);
                a.bal_o[(pbase + g) * kD + d] = l > 0.f ? v * (a.v_scale / l) : 0.f;
                if (d == 0) a.bal_lse[pbase + g] = l > 0.f ? M + log2f(l) : -INFINITY;
            }
            // Publish: after the consumer barrier one GPU-scope acq_rel atomic by
            // thread 0 orders every consumer's partial writes before the count,
            // and (for the last arriver) the other pieces' writes before our reads.
            if (!csync()) break;
            int* counter = a.counters + static_cast<size_t>(ti.b) * a.num_kv_heads + ti.h;
            if (threadIdx.x == 0) *mg.flag = (atom_add_acq_rel(counter, 1) == ti.pieces - 1) ? 1 : 0;
            if (!csync()) break;
            if (*mg.flag) {  // every other piece is published: merge them all in one pass
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float M = -INFINITY, v = 0.f, z = 0.f;
#pragma unroll 4
                    for (int j = 0; j < ti.pieces; ++j) {
                        const size_t pj = (static_cast<size_t>(ti.c_first + j) * 2 + (j == 0 ? ti.s_first : 0)) * G + g;
                        const float lj = __ldcg(a.bal_lse + pj), oj = __ldcg(a.bal_o + pj * kD + d);
                        if (lj == -INFINITY) continue;  // a piece with no token for this query
                        const float Mn = fmaxf(M, lj);
                        const float c = exp2f(M - Mn), w = exp2f(lj - Mn);
                        v = fmaf(v, c, w * oj);
                        z = fmaf(z, c, w);
                        M = Mn;
                    }
                    out[qrow(g) * kD + d] = __float2bfloat16_rn(z > 0.f ? v / z : 0.f);
                }
                if (threadIdx.x == 0) *counter = 0;  // ready for the next call
            }
            // every consumer read the merge area before the second barrier, so
            // the next segment may overwrite it without another barrier
            if (ti.flags & kCtaLast) break;
            continue;
        }
        if (!csync()) break;  // the merge area is reused by the next segment
        if (ti.flags & kCtaLast) break;
    }
    if (aborted || *abort_flag) return;
    if constexpr (kBal) {  // zero the rows of empty sequences (and report bad lengths once)
        for (int b = blockIdx.x; b < a.num_seqs; b += gridDim.x) {
            if (clamped_len(a, b, threadIdx.x == 0) == 0) {
                __nv_bfloat16* o = out + static_cast<size_t>(b) * a.num_queries * a.num_q_heads * kD;
                for (int i = threadIdx.x; i < a.num_queries * a.num_q_heads * kD; i += kCWarps * 32)
                    o[i] = __float2bfloat16_rn(0.f);
            }
        }
    }
}

template <int DT, int G, bool kBal>
cudaError_t launch_g(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    using Lt = Layout<DT, G>;
    constexpr size_t smem = Lt::kAlloc;
    auto kern = decode_mma_kernel<DT, G, kBal>;
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
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kMmaThreads, smem);
        if (e != cudaSuccess) return e;
        ctas_per_sm[dev] = occ > 0 ? occ : 1;
        configured_mask |= 1 << dev;
    }
    dim3 grid;
    if constexpr (kBal) {
        const int P = num_sms() * ctas_per_sm[dev];
        grid = dim3(P < a.bal_max_ctas ? P : a.bal_max_ctas);
    } else {
        grid = dim3(a.num_splits, a.num_kv_heads, a.num_seqs);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start while the previous kernel drains
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tk, tv, a);
}

template <int DT, bool kBal>
cudaError_t launch_dt(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    switch (a.num_queries * (a.num_q_heads / a.num_kv_heads)) {
        case 1: return launch_g<DT, 1, kBal>(a, tk, tv, stream);
        case 2: return launch_g<DT, 2, kBal>(a, tk, tv, stream);
        case 4: return launch_g<DT, 4, kBal>(a, tk, tv, stream);
        case 8: return launch_g<DT, 8, kBal>(a, tk, tv, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool decode_mma_supported(pkv_dtype kv, int head_dim, int group, int block_size) {
    if (kv != PKV_BF16 && kv != PKV_FP8_E4M3) return false;
    if (head_dim != kD) return false;
    if (group != 1 && group != 2 && group != 4 && group != 8) return false;
    return block_size == 16 || block_size == 32 || block_size == 64;
}

cudaError_t launch_decode_mma(pkv_dtype kv, const DecodeArgs& a, const void* tmap_k, const void* tmap_v,
                              cudaStream_t stream) {
    const CUtensorMap& tk = *static_cast<const CUtensorMap*>(tmap_k);
    const CUtensorMap& tv = *static_cast<const CUtensorMap*>(tmap_v);
    const bool bal = a.bal_max_ctas > 0;
    if (kv == PKV_BF16)
        return bal ? launch_dt<PKV_BF16, true>(a, tk, tv, stream) : launch_dt<PKV_BF16, false>(a, tk, tv, stream);
    if (kv == PKV_FP8_E4M3)
        return bal ? launch_dt<PKV_FP8_E4M3, true>(a, tk, tv, stream)
                   : launch_dt<PKV_FP8_E4M3, false>(a, tk, tv, stream);
    return cudaErrorNotSupported;
}

}  // namespace pkv
