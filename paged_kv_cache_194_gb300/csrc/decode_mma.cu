// Paged decode attention, tensor-core design (BF16 and FP8-E4M3 pools,
// head_dim 128, query group G in {1, 2, 4, 8}).
//
// "How does TensorRT-LLM work?", "Custom attention kernels": one kernel does
// the whole attention step and keeps the intermediate scores on chip.
// "Introduction to TensorRT-LLM", figure "TensorRT-LLM Acceleration Stack":
// Flash-Decoding splits the key/value length across CTAs; the log-sum-exp
// merge of the splits runs in the combine kernel.
//
// CTA = one (split, KV head, sequence); 4 consumer warps + 1 producer warp.
//  * Producer: one lane walks the block table and issues, per 64-token stage,
//    one TMA tile load (cp.async.bulk.tensor, 128-byte swizzle) per block of
//    K and of V into the stage: for BF16 a 3D box {64 columns, bs rows,
//    2 halves} fetches the block's whole 256-byte rows at once (two 2D boxes
//    if the driver refuses that descriptor); a full mbarrier counts the
//    bytes, an empty mbarrier (4 arrivals) frees the stage.
//    Every KV byte crosses HBM once; the G query heads of the KV head share it.
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
//  * The 4 warps' (m, l, O) are merged through shared memory at the end; the
//    CTA writes the final row (one split) or fp32 partials + log2-sum-exp.
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
constexpr int kTT = kTileTokens;           // tokens per stage (16 per consumer warp)
constexpr int kBoxRowBytes = 128;          // one swizzled TMA row
constexpr uint32_t kSpinLimit = 1u << 22;  // try_wait polls before a wait gives up

template <int DT>
struct MmaCfg;
template <>
struct MmaCfg<PKV_BF16> {
    static constexpr int kHalves = 2;  // 128 columns = two 64-column (128-byte) boxes
    static constexpr int kStages = 3;
};
template <>
struct MmaCfg<PKV_FP8_E4M3> {
    static constexpr int kHalves = 1;  // 128 one-byte columns = one 128-byte box
    static constexpr int kStages = 5;
};

// Stage layout of one tensor (K or V): [block of the tile][half][bs rows][128 B].
// A block's two halves (head_dim 0-63 and 64-127 for BF16) are bs*128 bytes
// apart; both start on 1024-byte boundaries (bs >= 16), so the 128-byte
// swizzle phase of a row is its row index within the block, mod 8.
constexpr int kHalfBytes = kTT * kBoxRowBytes;  // 8 KB: 64 rows x 128 B
template <int DT>
constexpr int tensor_stage_bytes() { return MmaCfg<DT>::kHalves * kHalfBytes; }
template <int DT>
constexpr int stage_bytes() { return 2 * tensor_stage_bytes<DT>(); }

constexpr int kMergeStride = 128 + 4;  // padded d stride of the merge buffer
constexpr int kMergeBytes = (kCWarps * 8 * kMergeStride + 2 * kCWarps * 8) * 4;

template <int DT>
constexpr size_t body_bytes() {
    const size_t st = static_cast<size_t>(MmaCfg<DT>::kStages) * stage_bytes<DT>();
    return st > kMergeBytes ? st : kMergeBytes;
}
template <int DT>
constexpr size_t mma_smem_bytes() {
    return 1024 /* alignment slack */ + body_bytes<DT>() + 2 * MmaCfg<DT>::kStages * 8 + 16;
}

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
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kCWarps * 32) : "memory"); }

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
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
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

template <int DT, int G>
__global__ void __launch_bounds__(kMmaThreads, 2)
decode_mma_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
    using C = MmaCfg<DT>;
    constexpr int kStages = C::kStages;
    constexpr int kHalves = C::kHalves;
    constexpr int kTB = tensor_stage_bytes<DT>();
    constexpr int kSB = stage_bytes<DT>();

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + body_bytes<DT>());
    uint64_t* empty = full + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int L = clamped_len(a, b, split == 0 && h == 0 && threadIdx.x == 0);
    const int t_begin = split * a.split_tokens;
    const int t_end = min(L, t_begin + a.split_tokens);
    const bool direct = a.num_splits == 1;
    const int hq0 = h * G;
    constexpr int D = 128;

    if (t_begin >= t_end) {
        if (direct) {
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) + (static_cast<size_t>(b) * a.num_q_heads + hq0) * D;
            for (int i = threadIdx.x; i < G * D; i += kMmaThreads) o[i] = __float2bfloat16_rn(0.f);
        }
        return;
    }
    const int num_tiles = (t_end - t_begin + kTT - 1) / kTT;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kCWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    __syncthreads();

    if (warp == kCWarps) {
        // ------------------------------------------------------------ producer
        const int bs = a.block_size;
        const int32_t* table = a.tables + static_cast<size_t>(b) * a.max_blocks;
        const int64_t layer_blk0 = static_cast<int64_t>(a.layer) * a.num_blocks;
        int cache = -1, cache_base = -1;
        int issued = 0;
        bool ok = true;
        for (int tile = 0; tile < num_tiles && ok; ++tile) {
            const int s = tile % kStages;
            if (tile >= kStages) {
                ok = mbar_wait(smem_u32(&empty[s]), ((tile / kStages) - 1) & 1);
                if (!ok) break;
            }
            if (*abort_flag) {
                ok = false;
                break;
            }
            const int tok0 = t_begin + tile * kTT;
            const int n = min(kTT, t_end - tok0);
            const int nblk = (n + bs - 1) / bs;
            if (lane == 0) mbar_expect_tx(smem_u32(&full[s]), static_cast<uint32_t>(nblk * bs * kBoxRowBytes * kHalves * 2));
            uint8_t* kst = smem + s * kSB;
            uint8_t* vst = kst + kTB;
            for (int k = 0; k < nblk; ++k) {
                const int j = tok0 / bs + k;  // block index within the sequence
                if (cache_base < 0 || j - cache_base >= 32) {
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
                    const int y = static_cast<int>(((layer_blk0 + blk) * a.num_kv_heads + h) * bs);
                    const uint32_t off = k * kHalves * bs * kBoxRowBytes;
                    if (kHalves == 2 && a.tma_3d) {  // one box: both 128-byte halves of every row
                        tma_load_3d(smem_u32(kst + off), &tmk, 0, y, 0, smem_u32(&full[s]));
                        tma_load_3d(smem_u32(vst + off), &tmv, 0, y, 0, smem_u32(&full[s]));
                    } else {
                        for (int hf = 0; hf < kHalves; ++hf) {
                            const uint32_t o2 = off + hf * bs * kBoxRowBytes;
                            tma_load_2d(smem_u32(kst + o2), &tmk, hf * 64, y, smem_u32(&full[s]));
                            tma_load_2d(smem_u32(vst + o2), &tmv, hf * 64, y, smem_u32(&full[s]));
                        }
                    }
                }
            }
            ++issued;
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            if (a.err) atomicOr(a.err, PKV_ERRBIT_TIMEOUT);
        }
        // drain: every issued copy has landed before the CTA may exit
        if (lane == 0) {
            for (int t = issued - 1; t >= 0 && t >= issued - kStages; --t)
                (void)mbar_wait(smem_u32(&full[t % kStages]), (t / kStages) & 1);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int r = lane >> 2, q = lane & 3;  // fragment row / column-pair index
    // Q^T as the B operand, one k-step of 16 head-dim entries per register pair.
    uint32_t bq[8][2];
    {
        const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(a.q) +
                                    (static_cast<size_t>(b) * a.num_q_heads + hq0 + (r < G ? r : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            if (r >= G) {
                bq[ks][0] = bq[ks][1] = 0u;
                continue;
            }
            if constexpr (DT == PKV_BF16) {
                const uint32_t* w = reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * q);
                bq[ks][0] = w[0];
                bq[ks][1] = w[4];  // +8 elements
            } else {
                const __nv_bfloat16* p = qrow + ks * 16 + 4 * q;
                bq[ks][0] = pack2<DT>(__bfloat162float(p[0]), __bfloat162float(p[1]));
                bq[ks][1] = pack2<DT>(__bfloat162float(p[2]), __bfloat162float(p[3]));
            }
        }
    }
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2q, 2q+1
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    const int row0 = warp * 16;
    const float qk = a.qk_scale_log2;
    const int bsz = a.block_size;
    const uint32_t half_stride = static_cast<uint32_t>(bsz * kBoxRowBytes);
    // this warp's 16 rows: block row0/bs of the tile, rows row0%bs.. of it
    const uint32_t warp_base = static_cast<uint32_t>((row0 / bsz) * kHalves * bsz * kBoxRowBytes +
                                                     (row0 % bsz) * kBoxRowBytes);
    bool aborted = false;

    for (int tile = 0; tile < num_tiles; ++tile) {
        const int s = tile % kStages;
        if (!mbar_wait(smem_u32(&full[s]), (tile / kStages) & 1)) {
            aborted = true;
            if (lane == 0) {
                *abort_flag = 1;
                if (a.err) atomicOr(a.err, PKV_ERRBIT_TIMEOUT);
            }
            break;
        }
        const int n = min(kTT, t_end - (t_begin + tile * kTT));
        uint8_t* kst = smem + s * kSB;
        uint8_t* vst = kst + kTB;
        if (row0 < n) {
            if (n < row0 + 16) {  // zero this warp's V rows past the end
                for (int i = lane; i < 16 * kHalves * 8; i += 32) {
                    const int lr = i / (kHalves * 8);
                    const int rest = i % (kHalves * 8);
                    if (row0 + lr >= n)
                        *reinterpret_cast<uint4*>(vst + warp_base + (rest >> 3) * half_stride + lr * kBoxRowBytes +
                                                  (rest & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async();
                __syncwarp();
            }
            // ---- S^T = K Q^T
            float sc[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t kb = smem_u32(kst) + warp_base;
            const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;  // row (of the warp's 16) this lane addresses
            if constexpr (DT == PKV_BF16) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const int chunk = 2 * (ks & 3) + (lane >> 4);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(kb + (ks >> 2) * half_stride + swz(lrow, chunk), a0, a1, a2, a3);
                    mma16816<DT>(sc, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
                }
            } else {
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {  // two k-steps (chunks 2kp, 2kp+1) per ldmatrix.x4
                    const int chunk = 2 * kp + (lane >> 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(kb + swz(lrow, chunk), r0, r1, r2, r3);
                    mma16816<DT>(sc, e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                                 e4m3x2_to_f16x2(r1 >> 16), bq[2 * kp][0], bq[2 * kp][1]);
                    mma16816<DT>(sc, e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                                 e4m3x2_to_f16x2(r3 >> 16), bq[2 * kp + 1][0], bq[2 * kp + 1][1]);
                }
            }
            // ---- online softmax (log2 domain); rows row0+r and row0+r+8
            const bool va = row0 + r < n, vb = row0 + r + 8 < n;
            const float s0 = va ? sc[0] * qk : -INFINITY;
            const float s1 = va ? sc[1] * qk : -INFINITY;
            const float s2 = vb ? sc[2] * qk : -INFINITY;
            const float s3 = vb ? sc[3] * qk : -INFINITY;
            float x0 = fmaxf(s0, s2), x1 = fmaxf(s1, s3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(0xFFFFFFFFu, x0, off));
                x1 = fmaxf(x1, __shfl_xor_sync(0xFFFFFFFFu, x1, off));
            }
            const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
            const float al0 = exp2f(m0 - n0), al1 = exp2f(m1 - n1);
            const float p0 = exp2f(s0 - n0), p1 = exp2f(s1 - n1);
            const float p2 = exp2f(s2 - n0), p3 = exp2f(s3 - n1);
            l0 = l0 * al0 + (p0 + p2);
            l1 = l1 * al1 + (p1 + p3);
            m0 = n0;
            m1 = n1;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                o[mt][0] *= al0;
                o[mt][1] *= al1;
                o[mt][2] *= al0;
                o[mt][3] *= al1;
            }
            const uint32_t pb0 = movmatrix_t(pack2<DT>(p0, p1));  // tokens 0-7 of the warp's 16
            const uint32_t pb1 = movmatrix_t(pack2<DT>(p2, p3));  // tokens 8-15
            // ---- O^T += V^T P^T
            const uint32_t vb_ = smem_u32(vst) + warp_base;
            if constexpr (DT == PKV_BF16) {
                const int trow = (lane & 7) + ((lane >> 4) & 1) * 8;
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    const int chunk = 2 * (mt & 3) + ((lane >> 3) & 1);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(vb_ + (mt >> 2) * half_stride + swz(trow, chunk), a0, a1, a2, a3);
                    mma16816<DT>(o[mt], a0, a1, a2, a3, pb0, pb1);
                }
            } else {
                const int ta = 2 * q;  // the warp's rows ta, ta+1, ta+8, ta+9
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int chunk = 2 * j + (r >> 2);
                    const uint32_t inner = static_cast<uint32_t>((r & 3) * 4);
                    const uint32_t w0 = lds32(vb_ + swz(ta, chunk) + inner);
                    const uint32_t w1 = lds32(vb_ + swz(ta + 1, chunk) + inner);
                    const uint32_t w8 = lds32(vb_ + swz(ta + 8, chunk) + inner);
                    const uint32_t w9 = lds32(vb_ + swz(ta + 9, chunk) + inner);
                    const uint32_t x01 = __byte_perm(w0, w1, 0x5140), x23 = __byte_perm(w0, w1, 0x7362);
                    const uint32_t y01 = __byte_perm(w8, w9, 0x5140), y23 = __byte_perm(w8, w9, 0x7362);
                    mma16816<DT>(o[2 * j], e4m3x2_to_f16x2(x01), e4m3x2_to_f16x2(x01 >> 16), e4m3x2_to_f16x2(y01),
                                 e4m3x2_to_f16x2(y01 >> 16), pb0, pb1);
                    mma16816<DT>(o[2 * j + 1], e4m3x2_to_f16x2(x23), e4m3x2_to_f16x2(x23 >> 16),
                                 e4m3x2_to_f16x2(y23), e4m3x2_to_f16x2(y23 >> 16), pb0, pb1);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }

    // ---- merge the 4 warps' partial (m, l, O) through shared memory
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
    }
    consumer_sync();  // every consumer is done with the stages
    float* mo = reinterpret_cast<float*>(smem);          // [warp][head 8][kMergeStride]
    float* mm = mo + kCWarps * 8 * kMergeStride;         // [warp][head 8]
    float* ml = mm + kCWarps * 8;                        // [warp][head 8]
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        float* base = mo + (warp * 8 + 2 * q) * kMergeStride;
        base[o_dim<DT>(mt, r)] = o[mt][0];
        base[kMergeStride + o_dim<DT>(mt, r)] = o[mt][1];
        base[o_dim<DT>(mt, r + 8)] = o[mt][2];
        base[kMergeStride + o_dim<DT>(mt, r + 8)] = o[mt][3];
    }
    if (lane < 4) {
        mm[warp * 8 + 2 * q] = m0;
        mm[warp * 8 + 2 * q + 1] = m1;
        ml[warp * 8 + 2 * q] = l0;
        ml[warp * 8 + 2 * q + 1] = l1;
    }
    consumer_sync();
    if (aborted || *abort_flag) return;
    const int d = threadIdx.x;  // 128 consumer threads = 128 head-dim entries
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) M = fmaxf(M, mm[w * 8 + g]);
        float acc = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kCWarps; ++w) {
            const float f = exp2f(mm[w * 8 + g] - M);
            acc += f * mo[(w * 8 + g) * kMergeStride + d];
            lsum += f * ml[w * 8 + g];
        }
        const float val = acc * (a.v_scale / lsum);
        const size_t row = static_cast<size_t>(b) * a.num_q_heads + hq0 + g;
        if (direct) {
            static_cast<__nv_bfloat16*>(a.out)[row * D + d] = __float2bfloat16_rn(val);
        } else {
            a.o_part[(row * a.num_splits + split) * D + d] = val;
            if (d == 0) a.lse_part[row * a.num_splits + split] = M + log2f(lsum);
        }
    }
}

template <int DT, int G>
cudaError_t launch_g(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    constexpr size_t smem = mma_smem_bytes<DT>();
    auto kern = decode_mma_kernel<DT, G>;
    static int configured_mask = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 31 && !(configured_mask & (1 << dev))) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured_mask |= 1 << dev;
    }
    dim3 grid(a.num_splits, a.num_kv_heads, a.num_seqs);
    kern<<<grid, kMmaThreads, smem, stream>>>(tk, tv, a);
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dt(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t stream) {
    switch (a.num_q_heads / a.num_kv_heads) {
        case 1: return launch_g<DT, 1>(a, tk, tv, stream);
        case 2: return launch_g<DT, 2>(a, tk, tv, stream);
        case 4: return launch_g<DT, 4>(a, tk, tv, stream);
        case 8: return launch_g<DT, 8>(a, tk, tv, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool decode_mma_supported(pkv_dtype kv, int head_dim, int group, int block_size) {
    if (kv != PKV_BF16 && kv != PKV_FP8_E4M3) return false;
    if (head_dim != 128) return false;
    if (group != 1 && group != 2 && group != 4 && group != 8) return false;
    return block_size == 16 || block_size == 32 || block_size == 64;
}

cudaError_t launch_decode_mma(pkv_dtype kv, const DecodeArgs& a, const void* tmap_k, const void* tmap_v,
                              cudaStream_t stream) {
    const CUtensorMap& tk = *static_cast<const CUtensorMap*>(tmap_k);
    const CUtensorMap& tv = *static_cast<const CUtensorMap*>(tmap_v);
    if (kv == PKV_BF16) return launch_dt<PKV_BF16>(a, tk, tv, stream);
    if (kv == PKV_FP8_E4M3) return launch_dt<PKV_FP8_E4M3>(a, tk, tv, stream);
    return cudaErrorNotSupported;
}

}  // namespace pkv
