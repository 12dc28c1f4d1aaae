// Paged decode attention, CUDA-core (SIMT) design, plus the flash-decoding
// log-sum-exp combine.
//
// "How does TensorRT-LLM work?", "Custom attention kernels": the whole
// attention step runs in one kernel and the scores never leave the chip.
// "Introduction to TensorRT-LLM", figure "TensorRT-LLM Acceleration Stack":
// Flash-Decoding -- the key/value length is split across CTAs and the
// partial results are merged.
//
// One CTA per (split, KV head, sequence).  It serves the whole group of G
// query heads that share the KV head, so every K/V byte is read from HBM
// once.  Tiles of 64 tokens are staged through a 3-deep cp.async pipeline;
// the block table is read per tile.  Per tile:
//   QK   warp w scores rows [16w, 16w+16); a row is split over LPT lanes (one
//        16-byte chunk each) and the G partial dot products are reduced with a
//        transposing butterfly (G-1 + log2(LPT/G) shuffles instead of
//        G*log2(LPT));
//   soft warp g%4 owns head g: tile max, rescale factor, exp2, running sum;
//   PV   thread (token group, chunk) accumulates G x chunk outputs over its
//        rows; groups are merged through shared memory once per split.
// Scores are kept in the log2 domain (q is pre-scaled by scale*log2(e)).
#include <cfloat>
#include <type_traits>

#include "device_common.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kTile = kTileTokens;
constexpr int kStages = 3;

template <int DT, int D>
struct SimtShape {
    using T = KvTraits<DT>;
    static constexpr int E = T::kPerChunk;                 // elements per chunk
    static constexpr int kRowBytes = D * T::kBytes;
    static constexpr int CPR = kRowBytes / 16;             // chunks per row
    static constexpr int LPT = CPR;                        // QK lanes per token
    static constexpr int TPP = 32 / LPT;                   // tokens per warp pass
    static constexpr int NTG = kThreads / CPR;             // PV token groups
    static constexpr size_t kStageBytes = static_cast<size_t>(kTile) * kRowBytes;
};

template <int DT, int D, int G>
constexpr bool simt_ok() {
    using S = SimtShape<DT, D>;
    return S::LPT <= 32 && G <= S::LPT && G * S::E <= 64;
}

template <int DT, int D, int G>
constexpr size_t simt_smem_bytes() {
    using S = SimtShape<DT, D>;
    const size_t stages = 2 * kStages * S::kStageBytes;
    const size_t red = static_cast<size_t>(S::NTG) * G * D * sizeof(float);
    const size_t body = stages > red ? stages : red;
    return body + (static_cast<size_t>(kTile) * G + 3 * G) * sizeof(float);
}

template <int DT, int D, int G, typename QT>
__global__ void __launch_bounds__(kThreads)
decode_simt_kernel(const DecodeArgs a) {
    using S = SimtShape<DT, D>;
    using T = KvTraits<DT>;
    constexpr int E = S::E, CPR = S::CPR, LPT = S::LPT, TPP = S::TPP, NTG = S::NTG;
    constexpr int kRowBytes = S::kRowBytes;
    constexpr int kRowsPerWarp = kTile / kWarps;
    constexpr int kHeadsPerWarp = (G + kWarps - 1) / kWarps;
    constexpr int kLogLPT = __builtin_ctz(LPT);
    constexpr int kLogG = __builtin_ctz(G);

    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t* sK = smem;
    uint8_t* sV = smem + kStages * S::kStageBytes;
    constexpr size_t kBody = simt_smem_bytes<DT, D, G>() - (static_cast<size_t>(kTile) * G + 3 * G) * sizeof(float);
    float* sP = reinterpret_cast<float*>(smem + kBody);  // [kTile][G] scores -> probabilities
    float* sAlpha = sP + kTile * G;                      // [G]
    float* sM = sAlpha + G;                              // [G]
    float* sL = sM + G;                                  // [G]

    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = visible_len(a, b, split == 0 && h == 0 && tid == 0);
    const int t_begin = split * a.split_tokens;
    const int t_end = min(L, t_begin + a.split_tokens);
    const bool direct = a.num_splits == 1;

    // The G rows served here are C queries x gh heads: row g is query
    // q_first + g / gh of the sequence (position L - C + g / gh of the
    // visible length L, attending causally) and head h*gh + g % gh.
    const int Cq = a.num_queries, gh = G / Cq;
    auto qrow = [&](int g) -> size_t {
        return (static_cast<size_t>(b) * a.q_total + a.q_first + g / gh) * a.num_q_heads + static_cast<size_t>(h) * gh +
               g % gh;
    };
    if (t_begin >= t_end) {
        if (direct) {  // empty sequence: zero output rows
            for (int i = tid; i < G * D; i += kThreads) static_cast<QT*>(a.out)[qrow(i / D) * D + i % D] = to_out<QT>(0.f);
        }
        return;
    }

    // q slice of this lane: chunk (lane % LPT) of each of the G rows.
    const int qc = lane % LPT;
    float qf[G][E];
    {
        const QT* qb = static_cast<const QT*>(a.q);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < E; ++e) qf[g][e] = load_q<QT>(qb + qrow(g) * D + qc * E + e) * a.qk_scale_log2;
    }

    float m_run[kHeadsPerWarp], l_run[kHeadsPerWarp];
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
        m_run[i] = -INFINITY;
        l_run[i] = 0.f;
    }
    const int pc = tid % CPR, ptg = tid / CPR;  // PV chunk and token group
    float acc[G][E];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[g][e] = 0.f;

    const int num_tiles = (t_end - t_begin + kTile - 1) / kTile;
    const int32_t* table = a.tables + static_cast<size_t>(b) * a.max_blocks;
    const size_t head_off = static_cast<size_t>(h) * a.block_size;

    auto issue = [&](int tile, int stage) {
        const int tok0 = t_begin + tile * kTile;
        const int n = min(kTile, t_end - tok0);
        uint8_t* dk = sK + stage * S::kStageBytes;
        uint8_t* dv = sV + stage * S::kStageBytes;
        for (int i = tid; i < n * CPR; i += kThreads) {
            const int r = i / CPR, c = i % CPR;
            const int tok = tok0 + r;
            const int blk = table[tok / a.block_size];
            const bool ok = static_cast<unsigned>(blk) < static_cast<unsigned>(a.num_blocks);
            if (!ok && a.err) atomicOr(a.err, PKV_ERRBIT_BLOCK_ID);
            const size_t row = (static_cast<size_t>(ok ? blk : 0) * a.num_kv_heads * a.block_size + head_off +
                                tok % a.block_size) * kRowBytes + c * 16;
            cp_async16(dk + r * kRowBytes + c * 16, a.k_layer + row, ok ? 16 : 0);
            cp_async16(dv + r * kRowBytes + c * 16, a.v_layer + row, ok ? 16 : 0);
        }
    };

#pragma unroll
    for (int i = 0; i < kStages - 1; ++i) {
        if (i < num_tiles) issue(i, i);
        cp_async_commit();
    }

    for (int tile = 0; tile < num_tiles; ++tile) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        {
            const int nt = tile + kStages - 1;
            if (nt < num_tiles) issue(nt, nt % kStages);
            cp_async_commit();
        }
        const int stage = tile % kStages;
        const int n = min(kTile, t_end - (t_begin + tile * kTile));
        const uint8_t* Ks = sK + stage * S::kStageBytes;
        const uint8_t* Vs = sV + stage * S::kStageBytes;

        // ---- QK: scores of this warp's rows
#pragma unroll
        for (int pass = 0; pass < kRowsPerWarp / TPP; ++pass) {
            const int r = warp * kRowsPerWarp + pass * TPP + lane / LPT;
            float part[G];
#pragma unroll
            for (int g = 0; g < G; ++g) part[g] = 0.f;
            if (r < n) {
                float kf[E];
                T::to_float(*reinterpret_cast<const uint4*>(Ks + r * kRowBytes + qc * 16), kf);
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int e = 0; e < E; ++e) part[g] = fmaf(qf[g][e], kf[e], part[g]);
            }
            // transposing butterfly: halve the live heads per step
#pragma unroll
            for (int st = 0; st < kLogG; ++st) {
                const int off = LPT >> (st + 1);
                const int half = G >> (st + 1);
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float send = upper ? part[i] : part[i + half];
                    const float keep = upper ? part[i + half] : part[i];
                    part[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, off);
                }
            }
#pragma unroll
            for (int st = kLogG; st < kLogLPT; ++st) part[0] += __shfl_xor_sync(0xFFFFFFFFu, part[0], LPT >> (st + 1));
            const int j = lane % LPT;
            const int g_mine = j >> (kLogLPT - kLogG);
            if (r < n && (j & ((LPT >> kLogG) - 1)) == 0) sP[r * G + g_mine] = part[0];
        }
        __syncthreads();

        // ---- online softmax, one warp per row; row g sees tokens before L - C + g/gh + 1
#pragma unroll
        for (int i = 0; i < kHeadsPerWarp; ++i) {
            const int g = warp + kWarps * i;
            if (g < G) {
                const int lim = min(n, L - Cq + g / gh + 1 - (t_begin + tile * kTile));
                const float s0 = lane < lim ? sP[lane * G + g] : -INFINITY;
                const float s1 = lane + 32 < lim ? sP[(lane + 32) * G + g] : -INFINITY;
                const float m_new = fmaxf(m_run[i], warp_max(fmaxf(s0, s1)));
                // a row that has seen no token yet keeps max -inf and weights 0
                const float base = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = m_new == -INFINITY ? 1.f : exp2f(m_run[i] - m_new);
                const float p0 = exp2f(s0 - base), p1 = exp2f(s1 - base);
                if (lane < n) sP[lane * G + g] = p0;  // 0 past the row's causal limit
                if (lane + 32 < n) sP[(lane + 32) * G + g] = p1;
                l_run[i] = l_run[i] * alpha + warp_sum(p0 + p1);
                m_run[i] = m_new;
                if (lane == 0) sAlpha[g] = alpha;
            }
        }
        __syncthreads();

        // ---- PV
        {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float al = sAlpha[g];
#pragma unroll
                for (int e = 0; e < E; ++e) acc[g][e] *= al;
            }
            for (int r = ptg; r < n; r += NTG) {
                float vf[E];
                T::to_float(*reinterpret_cast<const uint4*>(Vs + r * kRowBytes + pc * 16), vf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float p = sP[r * G + g];
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[g][e] = fmaf(p, vf[e], acc[g][e]);
                }
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // stages are free; reuse them for the group merge

#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
        const int g = warp + kWarps * i;
        if (g < G && lane == 0) {
            sM[g] = m_run[i];
            sL[g] = l_run[i];
        }
    }
    float* red = reinterpret_cast<float*>(smem);  // [NTG][G][D]
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < E; ++e) red[(ptg * G + g) * D + pc * E + e] = acc[g][e];
    __syncthreads();

    for (int i = tid; i < G * D; i += kThreads) {
        const int g = i / D, d = i % D;
        float sum = 0.f;
#pragma unroll
        for (int t = 0; t < NTG; ++t) sum += red[(t * G + g) * D + d];
        const float l = sL[g];
        const float o = l > 0.f ? sum * (a.v_scale / l) : 0.f;
        if (direct) {
            static_cast<QT*>(a.out)[qrow(g) * D + d] = to_out<QT>(o);
        } else {  // partial rows of this launch: (b, query g / gh, head)
            const size_t row = (static_cast<size_t>(b) * Cq + g / gh) * a.num_q_heads + static_cast<size_t>(h) * gh + g % gh;
            a.o_part[(row * a.num_splits + split) * D + d] = o;
            if (d == 0) a.lse_part[row * a.num_splits + split] = l > 0.f ? sM[g] + log2f(l) : -INFINITY;
        }
    }
}

// Merge the splits of one (sequence, query head) per warp:
// out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M).
template <int D, typename QT>
__global__ void __launch_bounds__(128) combine_kernel(const DecodeArgs a) {
    constexpr int PER = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;  // partial row of this launch: (b * C + c) * Hq + hq
    if (row >= a.num_seqs * a.num_queries * a.num_q_heads) return;
    const int per_seq = a.num_queries * a.num_q_heads;
    const int b = row / per_seq;
    const int L = visible_len(a, b, false);
    const int ns = (L + a.split_tokens - 1) / a.split_tokens;
    const size_t orow = (static_cast<size_t>(b) * a.q_total + a.q_first) * a.num_q_heads + row % per_seq;
    QT* o = static_cast<QT*>(a.out) + orow * D + lane * PER;
    if (ns == 0) {
#pragma unroll
        for (int i = 0; i < PER; ++i) o[i] = to_out<QT>(0.f);
        return;
    }
    const float* lse = a.lse_part + static_cast<size_t>(row) * a.num_splits;
    const float* part = a.o_part + static_cast<size_t>(row) * a.num_splits * D + lane * PER;
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, lse[s]);
    M = warp_max(M);
    float z = 0.f, acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int s = 0; s < ns && M != -INFINITY; ++s) {
        const float w = exp2f(lse[s] - M);  // a split without a token for this query has lse -inf: weight 0
        z += w;
        const float* p = part + static_cast<size_t>(s) * D;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, p[i], acc[i]);
    }
    const float inv = z > 0.f ? 1.f / z : 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) o[i] = to_out<QT>(acc[i] * inv);
}

template <int DT, int D, int G>
cudaError_t launch_one(const DecodeArgs& a, cudaStream_t stream) {
    if constexpr (!simt_ok<DT, D, G>()) {
        return cudaErrorNotSupported;
    } else {
        using QT = typename std::conditional<DT == PKV_F32, float, __nv_bfloat16>::type;
        constexpr size_t smem = simt_smem_bytes<DT, D, G>();
        auto kern = decode_simt_kernel<DT, D, G, QT>;
        static int configured_mask = 0;  // per device bit
        int dev = 0;
        cudaGetDevice(&dev);
        if (dev < 31 && !(configured_mask & (1 << dev))) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
            configured_mask |= 1 << dev;
        }
        dim3 grid(a.num_splits, a.num_kv_heads, a.num_seqs);
        kern<<<grid, kThreads, smem, stream>>>(a);
        return cudaGetLastError();
    }
}

template <int DT, int D>
cudaError_t by_group(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.num_queries * (a.num_q_heads / a.num_kv_heads)) {
        case 1: return launch_one<DT, D, 1>(a, stream);
        case 2: return launch_one<DT, D, 2>(a, stream);
        case 4: return launch_one<DT, D, 4>(a, stream);
        case 8: return launch_one<DT, D, 8>(a, stream);
        case 16: return launch_one<DT, D, 16>(a, stream);
        default: return cudaErrorNotSupported;
    }
}

template <int DT>
cudaError_t by_dim(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.head_dim) {
        case 64: return by_group<DT, 64>(a, stream);
        case 128: return by_group<DT, 128>(a, stream);
        default: return cudaErrorNotSupported;
    }
}

template <int DT, int D>
bool ok_group(int g) {
    switch (g) {
        case 1: return simt_ok<DT, D, 1>();
        case 2: return simt_ok<DT, D, 2>();
        case 4: return simt_ok<DT, D, 4>();
        case 8: return simt_ok<DT, D, 8>();
        case 16: return simt_ok<DT, D, 16>();
        default: return false;
    }
}

template <int DT>
bool ok_dim(int d, int g) {
    if (d == 64) return ok_group<DT, 64>(g);
    if (d == 128) return ok_group<DT, 128>(g);
    return false;
}

}  // namespace

bool decode_simt_supported(pkv_dtype kv, int head_dim, int rows) {
    switch (kv) {
        case PKV_F32: return ok_dim<PKV_F32>(head_dim, rows);
        case PKV_BF16: return ok_dim<PKV_BF16>(head_dim, rows);
        case PKV_FP8_E4M3: return ok_dim<PKV_FP8_E4M3>(head_dim, rows);
    }
    return false;
}

cudaError_t launch_decode_simt(pkv_dtype kv, const DecodeArgs& a, cudaStream_t stream) {
    switch (kv) {
        case PKV_F32: return by_dim<PKV_F32>(a, stream);
        case PKV_BF16: return by_dim<PKV_BF16>(a, stream);
        case PKV_FP8_E4M3: return by_dim<PKV_FP8_E4M3>(a, stream);
    }
    return cudaErrorNotSupported;
}

cudaError_t launch_combine(pkv_dtype q_dtype, const DecodeArgs& a, cudaStream_t stream) {
    const int rows = a.num_seqs * a.num_queries * a.num_q_heads;
    const int blocks = (rows + 3) / 4;
    if (blocks == 0) return cudaSuccess;
    if (q_dtype == PKV_F32) {
        if (a.head_dim == 64) combine_kernel<64, float><<<blocks, 128, 0, stream>>>(a);
        else combine_kernel<128, float><<<blocks, 128, 0, stream>>>(a);
    } else {
        if (a.head_dim == 64) combine_kernel<64, __nv_bfloat16><<<blocks, 128, 0, stream>>>(a);
        else combine_kernel<128, __nv_bfloat16><<<blocks, 128, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace pkv
