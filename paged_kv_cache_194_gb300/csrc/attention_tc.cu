// Multi-query paged attention on the 5th-generation tensor cores (tcgen05
// with TMEM accumulators) for long query lists: prompt chunks, where the
// query rows of one KV head (C queries x gh heads) fill whole 128-row MMA
// tiles.  BF16 pools, head_dim 128.
//
// "How does TensorRT-LLM work?", "In-flight batching": long prompts are
// processed in chunks that attend to the cached prefix; "Custom attention
// kernels": the scores stay on chip.  Query c of the C queries of a sequence
// sits at position L - C + c of its visible length L and attends causally.
//
// Two schedules.  Grid: one CTA per (128 query rows, KV head, sequence), all
// of its tiles.  Balanced (at most 128 query rows per KV head, and fewer
// (sequence, KV head) units than CTA slots, i.e. a few long sequences): 2
// persistent CTAs per SM share out the 64-token tiles of all units equally;
// a CTA reloads Q at each unit it starts, and a unit cut between CTAs is
// merged from their pieces (O / l and log-sum-exp) by the last to finish.
// 7 warps:
//  * warps 4 and 6, TMA producers for K and for V: per 64-token tile, one box
//    {64 columns, bs rows, 1 half} per KV block and half, so a stage holds each of
//    K and V as [half: head_dim 0-63 | 64-127][64 token rows][128 B], 128-byte
//    swizzled -- the K-major operand layout for K and the MN-major one for V.
//  * warp 5, MMA issuer (one thread): S_j = Q K_j^T (M 128 rows, N 64 tokens,
//    K 128) into one of two TMEM score buffers, one tile ahead of the softmax;
//    then O += P_j V_j (M 128 rows, N 128 head dims, K 64 tokens) into the
//    TMEM output accumulator.  tcgen05.commit signals mbarriers.
//  * warps 0-3, softmax and epilogue: thread m owns query row m (TMEM lane m).
//    It reads its 64 scores with tcgen05.ld in one round trip, masks
//    causally (only on tiles its warp does not fully see), and overwrites
//    the score buffer with P as BF16 pairs, which the PV MMA reads as its A
//    operand from tensor memory; no shared-memory P, so a softmax never
//    waits for the previous PV except to rescale O.  Warps without a query
//    row only keep pace with the barriers.  The running max is updated lazily: O (in
//    TMEM) and the running sum are rescaled only when the row max grows by
//    more than 8 in log2 units, so probabilities stay below 2^8 and fp32 keeps
//    full precision; the final division by the sum uses the same base.
//  * Epilogue: O / l, rounded to BF16, written to the output rows (or, for a
//    piece of a shared unit, to the workspace, then merged).
// Shared memory: Q 32 KB, 2 stages x (K 16 KB + V 16 KB) for 64-token
// tiles; TMEM: two 64-column score buffers and a 128-column output
// accumulator (256 allocated); 2 CTAs per SM, so that two softmax warpgroups
// share each SM.  Every mbarrier wait is bounded; on expiry the CTA
// sets PKV_ERRBIT_TIMEOUT, waits (bounded) for its copies and MMAs, frees its
// TMEM and skips its output.
#include <cuda.h>

#include <climits>

#include "tc_common.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 224;              // warps 0-3 softmax, 4 K producer, 5 MMA, 6 V producer
constexpr int kRows = 128;                 // query rows per CTA
constexpr int kTok = 64;                   // tokens per tile
constexpr int kDim = 128;                  // head_dim
constexpr int kQHalf = kRows * 128;        // one 64-column half of the Q tile: 16 KB
constexpr int kHalfBytes = kTok * 128;     // one 64-column half of a K or V tile: 8 KB
constexpr int kQOff = 0;
constexpr int kKVOff = 2 * kQHalf;
constexpr int kStageBytes = 4 * kHalfBytes;  // K (16 KB) + V (16 KB)
constexpr int kAlignSlack = 1024;             // room to align the base to 1024 B
constexpr int kMC = 4;                     // 4-float chunks per merge round
constexpr int kRankMaxSeqs = 128;          // the grid schedule orders units by length up to this many sequences

// mbarriers (8 bytes each) after the tiles: these, then the full and empty
// barriers of the K and V rings
enum Bar { kQReady, kOFree, kGroup, kDone, kFixedBars };

// One configuration: kNS stages in each of the K and V rings.  Two stages
// leave room for 2 CTAs per SM, each with 256 TMEM columns: 2 score buffers
// (kNSB) of 64 columns and the 128-column output accumulator.  With more
// stages a CTA is alone on its SM and takes all 512 columns, i.e. 4 score
// buffers, so S can run up to three tiles ahead of the softmax.  That
// configuration computes the same results but ran slower in every case
// measured (4 to 1024 query rows per KV head): one CTA's producers and MMA
// issuer, not the bytes in flight, set the pace, and two CTAs per SM double
// them.  So the launcher uses two stages.
template <int kNS>
struct Cfg {
    static constexpr int kCtasPerSm = kNS == 2 ? 2 : 1;
    static constexpr int kNSB = kCtasPerSm == 2 ? 2 : 4;
    static constexpr uint32_t kTmemCols = kCtasPerSm == 2 ? 256 : 512;
    static constexpr uint32_t kOCol = kNSB * kTok;
    // per score buffer: S written, P written, PV that read P done
    static constexpr int kSFull = kFixedBars, kPFull = kSFull + kNSB, kPvDone = kPFull + kNSB;
    static constexpr int kKFull = kPvDone + kNSB, kKEmpty = kKFull + kNS;
    static constexpr int kVFull = kKEmpty + kNS, kVEmpty = kVFull + kNS;
    static constexpr int kNumBars = kVEmpty + kNS;
    static_assert(kOCol + kDim <= kTmemCols, "tensor memory");
    static constexpr int kBarOff = kKVOff + kNS * kStageBytes;
    static constexpr int kBarBytes = (8 * kNumBars + 12 + 63) / 64 * 64;  // + TMEM address, abort and merge flags
    static constexpr int kRangeOff = kBarOff + kBarBytes;   // per warp: the balanced schedule's {g0, T, P}
    static constexpr int kMergeOff = kRangeOff + 7 * 3 * 8;  // [kRows] M and [kRows] 1/z of a merge
    static constexpr int kSmem = kMergeOff + 2 * kRows * 4 + kAlignSlack;
    static_assert(kCtasPerSm == 2 ? kSmem <= 115712 : kSmem <= 232448, "shared memory per CTA");
};

__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// 64-token tiles of sequence b (0 past the batch); with one row tile per
// (sequence, KV head) the last query sees the whole visible length.
__device__ __forceinline__ int seq_tiles(const DecodeArgs& a, int b) {
    return b < a.num_seqs ? (visible_len(a, b, false) + kTok - 1) / kTok : 0;
}

// The tiles a CTA processes, in order.  A unit is the 128-row query tile of
// one (sequence, KV head) -- for the balanced schedule, the only row tile --
// and a segment is the run of a unit's tiles one CTA owns.
//  * grid schedule: one unit per CTA, (row tile, KV head, sequence) =
//    blockIdx, all of its tiles;
//  * balanced schedule (query rows <= 128 per KV head): the tiles of all units,
//    flattened in (sequence, KV head, tile) order, T in total, are cut into P
//    equal ranges, CTA c taking [c T / P, (c + 1) T / P).  Units cut by a range
//    boundary are finished by the CTA that publishes its piece last.
template <bool kBal>
struct Walk {
    int b = 0, h = 0, rt_ = 0;      // unit: sequence, KV head, row tile
    int L = 0, t_end_ = 0, nt = 0;  // visible length, tokens the unit reads, its tiles
    int t = 0;                      // tile within the unit
    int k = 0, ntiles = 0;          // tile within the CTA's range, the range's length

    // (balanced schedule: one row tile, whose last query sees the whole length)
    __device__ int rt() const { return kBal ? 0 : rt_; }
    __device__ int t_end() const { return kBal ? L : t_end_; }

    __device__ bool more() const { return k < ntiles; }
    __device__ bool seg_first() const { return k == 0 || t == 0; }
    __device__ bool seg_last() const { return k == ntiles - 1 || t == nt - 1; }
    // the unit lies inside the CTA's range / starts at or before it
    __device__ bool whole() const { return k >= t && k - t + nt <= ntiles; }
    __device__ bool cta_first() const { return k <= t; }

    // Warp-collective (the balanced schedule sums the lengths with shuffles).
    // range: where the balanced schedule leaves {g0, T, P} for segment ends;
    // (ub, uh, urt): the grid schedule's unit.
    __device__ void init(const DecodeArgs& a, int lane, int gh, long long* range, int ub, int uh, int urt) {
        if constexpr (!kBal) {
            rt_ = urt;
            h = uh;
            b = ub;
            L = visible_len(a, b, false);
            const int nq = a.num_queries * gh;
            const int last_row = min(nq, (rt_ + 1) * kRows) - 1;
            t_end_ = L - a.num_queries + last_row / gh + 1;
            nt = t_end_ > 0 ? (t_end_ + kTok - 1) / kTok : 0;
            ntiles = nt;
        } else {
            const int B = a.num_seqs, Hkv = a.num_kv_heads;
            long long tot = 0;
            for (int b0 = 0; b0 < B; b0 += 32) tot += warp_sum_ll(seq_tiles(a, b0 + lane));
            const long long T = tot * Hkv;
            const long long P = T < static_cast<long long>(gridDim.x) ? T : static_cast<long long>(gridDim.x);
            const long long c = blockIdx.x;
            const long long g0 = c < P ? c * T / P : T, g1 = c < P ? (c + 1) * T / P : T;
            if (lane == 0) {
                range[0] = g0;
                range[1] = T;
                range[2] = P;
            }
            ntiles = static_cast<int>(g1 - g0);  // about T / P: a few thousand at most
            if (g0 >= g1) return;
            // locate tile g0: sequence b, with cum = the tiles of the sequences before it
            long long cum = 0;
            for (int b0 = 0; b0 < B; b0 += 32) {
                const long long u = static_cast<long long>(seq_tiles(a, b0 + lane)) * Hkv;
                long long incl = u;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const long long x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += x;
                }
                const long long sum = __shfl_sync(0xFFFFFFFFu, incl, 31);
                if (g0 < cum + sum) {
                    const unsigned m = __ballot_sync(0xFFFFFFFFu, cum + incl > g0);
                    const int l = __ffs(m) - 1;
                    cum += __shfl_sync(0xFFFFFFFFu, incl - u, l);
                    b = b0 + l;
                    break;
                }
                cum += sum;
            }
            L = visible_len(a, b, false);
            nt = (L + kTok - 1) / kTok;
            const long long off = g0 - cum;
            h = static_cast<int>(off / nt);
            t = static_cast<int>(off % nt);
        }
    }
    __device__ void next(const DecodeArgs& a) {
        ++k;
        if constexpr (kBal) {
            if (++t < nt) return;
            t = 0;
            if (++h < a.num_kv_heads) return;
            h = 0;
            for (++b; b < a.num_seqs; ++b) {
                L = visible_len(a, b, false);
                if (L > 0) break;
            }
            if (b < a.num_seqs) nt = (L + kTok - 1) / kTok;
        } else {
            ++t;
        }
    }
};

template <bool kBal, int kNS>
__global__ void __launch_bounds__(kThreads, Cfg<kNS>::kCtasPerSm)
attention_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = su32(smem);
    using Lt = Cfg<kNS>;
    const uint32_t bars = sbase + Lt::kBarOff;
    auto B = [&](int i) { return bars + 8u * i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Lt::kBarOff + 8 * Lt::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Lt::kBarOff + 8 * Lt::kNumBars + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + Lt::kBarOff + 8 * Lt::kNumBars + 8);
    float* merge_m = reinterpret_cast<float*>(smem + Lt::kMergeOff);  // [kRows] M, [kRows] 1/z
    if (smem - smem_raw > kAlignSlack) {  // the base was not aligned enough for the layout
        if (threadIdx.x == 0 && a.err) atomicOr(a.err, PKV_ERRBIT_TIMEOUT);
        return;
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gh = a.num_q_heads / a.num_kv_heads;
    const int C = a.num_queries, nq = C * gh;
    asm volatile("griddepcontrol.wait;\n" ::: "memory");

    auto out_row = [&](int ob, int oh, int n) -> __nv_bfloat16* {
        return static_cast<__nv_bfloat16*>(a.out) +
               ((static_cast<size_t>(ob) * a.q_total + a.q_first + n / gh) * a.num_q_heads +
                static_cast<size_t>(oh) * gh + n % gh) *
                   kDim;
    };
    // Grid schedule: blocks start in linear order, so hand out the longest
    // units first (sequences by visible length, longest first; within one,
    // the later row tiles, which see more tokens, first): the last wave is
    // then made of short units.  For batches of up to kRankMaxSeqs sequences;
    // beyond that, blockIdx order.
    int ub = blockIdx.z, uh = blockIdx.y, urt = blockIdx.x;
    if constexpr (!kBal) {
        if (a.num_seqs <= kRankMaxSeqs) {
            const long long R = gridDim.x, Hkv = gridDim.y, per_seq = R * Hkv;
            const long long i = blockIdx.x + R * (blockIdx.y + Hkv * static_cast<long long>(blockIdx.z));
            const int rank = static_cast<int>(i / per_seq);  // < num_seqs: each rank is one sequence's
            const long long rem = i % per_seq;
            urt = static_cast<int>(R - 1 - rem / Hkv);
            uh = static_cast<int>(rem % Hkv);
            int* pick = reinterpret_cast<int*>(merge_m);
            for (int c = threadIdx.x; c < a.num_seqs; c += kThreads) {  // the rank of sequence c
                const int Lc = visible_len(a, c, false);
                int r = 0;
                for (int o = 0; o < a.num_seqs; ++o) {
                    const int Lo = visible_len(a, o, false);
                    r += (Lo > Lc || (Lo == Lc && o < c)) ? 1 : 0;
                }
                if (r == rank) *pick = c;
            }
            __syncthreads();
            ub = *pick;
        }
    }
    if constexpr (!kBal) {
        // every query of the tile at a negative position: zero rows
        const int rt = urt, h = uh, b = ub, row0 = rt * kRows;
        const int L = visible_len(a, b, rt == 0 && h == 0 && threadIdx.x == 0);
        if (L - C + (min(nq, row0 + kRows) - 1) / gh + 1 <= 0) {
            for (int i = threadIdx.x; i < kRows * kDim; i += kThreads) {
                const int n = row0 + i / kDim;
                if (n < nq) out_row(b, h, n)[i % kDim] = __float2bfloat16_rn(0.f);
            }
            return;
        }
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < Lt::kNumBars; ++i) {
            const uint32_t cnt =
                ((i >= Lt::kPFull && i < Lt::kPFull + Lt::kNSB) || i == kQReady || i == kOFree || i == kGroup) ? 4u
                                                                                                             : 1u;
            bar_init(B(i), cnt);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(su32(tmem_slot)),
                     "r"(Lt::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    auto fail = [&]() {
        *abort_flag = 1;
        if (a.err) atomicOr(a.err, PKV_ERRBIT_TIMEOUT);
    };
    long long* range = reinterpret_cast<long long*>(smem + Lt::kRangeOff) + 3 * warp;  // this warp's {g0, T, P}
    Walk<kBal> w;
    w.init(a, lane, gh, range, ub, uh, urt);

    if (warp == 4 || warp == 6) {
        // ---------------------------------------------- producers: K (warp 4), V (warp 6)
        // K stage s is free once S of its tile is done, V stage s once PV is,
        // so K loads run a tile ahead of V loads.
        const bool is_v = warp == 6;
        const CUtensorMap* map = is_v ? &tmv : &tmk;
        // With as many stages as score buffers, stage s is freed by the same
        // completion that signals score buffer s (S done for K, PV done for
        // V): the producers wait on those barriers and the MMA thread issues
        // two commits per tile fewer (a commit costs about what an MMA does
        // to issue).
        constexpr bool kSame = kNS == Lt::kNSB;
        const int full0 = is_v ? Lt::kVFull : Lt::kKFull;
        const int empty0 = is_v ? (kSame ? Lt::kPvDone : Lt::kVEmpty) : (kSame ? Lt::kSFull : Lt::kKEmpty);
        const int bs = a.block_size;
        const int64_t layer_blk0 = static_cast<int64_t>(a.layer) * a.num_blocks;
        // Block-table entries cache_base .. cache_base + 31 of sequence cache_b,
        // one per lane: one coalesced load per 32 blocks instead of a
        // dependent load per block ahead of each copy.
        int cache = 0, cache_base = 0, cache_b = -1;
        int k = 0;  // tiles issued
        for (; w.more() && !*abort_flag; w.next(a), ++k) {
            const int s = k % kNS;
            const int tok0 = w.t * kTok, n = min(kTok, w.t_end() - tok0), nblk = (n + bs - 1) / bs;
            const int idx0 = tok0 / bs;
            if (w.b != cache_b || idx0 < cache_base || idx0 + nblk > cache_base + 32) {  // (before the wait)
                cache_b = w.b;
                cache_base = idx0;
                const int idx = idx0 + lane;
                cache = idx < a.max_blocks ? __ldg(a.tables + static_cast<size_t>(w.b) * a.max_blocks + idx) : 0;
            }
            if (k >= kNS && !bar_wait(B(empty0 + s), ((k / kNS) - 1) & 1)) {
                if (lane == 0) fail();
                break;
            }
            const uint32_t dst0 = sbase + kKVOff + s * kStageBytes + (is_v ? 2 * kHalfBytes : 0);
            if (lane == 0) bar_expect_tx(B(full0 + s), static_cast<uint32_t>(nblk * bs * 128 * 2));
            __syncwarp();
            // One copy instruction for the whole tile: lane 2 kb + hf copies
            // half hf of block kb (issuing a copy costs a few hundred cycles,
            // about the same for one lane or eight).
            {
                const int kb = lane >> 1, hf = lane & 1;
                int blk = __shfl_sync(0xFFFFFFFFu, cache, (idx0 + kb - cache_base) & 31);
                if (kb < nblk) {
                    if (static_cast<unsigned>(blk) >= static_cast<unsigned>(a.num_blocks)) {
                        if (a.err) atomicOr(a.err, PKV_ERRBIT_BLOCK_ID);
                        blk = 0;  // read an in-bounds block; the flag marks the output invalid
                    }
                    const int y = static_cast<int>(((layer_blk0 + blk) * a.num_kv_heads + w.h) * bs);
                    tma_3d(dst0 + hf * kHalfBytes + kb * bs * 128, map, 0, y, hf, B(full0 + s));
                }
            }
        }
        // drain: the copies in flight land before the CTA frees anything
        if (lane == 0)
            for (int j = k - 1; j >= 0 && j >= k - kNS; --j)
                if (!bar_wait(B(full0 + j % kNS), (j / kNS) & 1)) fail();
    } else if (warp == 5) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            constexpr int NSB = Lt::kNSB;
            // S_j goes to score buffer j % NSB once the PV of tile j - NSB, which
            // read P from it, has been issued (MMAs run in issue order).  The S
            // cursor ws runs up to NSB - 1 tiles ahead of the PV cursor w.  The
            // S of tiles k and k + 1 may block: the softmax of tile k needs only
            // work issued already (S k, PV k - 1) to signal P k and, at a unit's
            // end, to store the next unit's Q.  An S further ahead that would
            // wait (for K, or for a Q the softmax stores only after scores not
            // yet issued) is left for later, so the PVs the softmax may be
            // waiting on still get issued.
            // Operand descriptors.  Their address field holds the shared-memory
            // address / 16, so the descriptor of base + off is the base's plus
            // off / 16 (no carry: a CTA's shared addresses stay below 2^18):
            // the issuing thread, which sets the pace, adds one constant per MMA.
            const uint64_t dq = sdesc(sbase + kQOff, 16);
            const uint64_t dk0 = sdesc(sbase + kKVOff, 16);
            const uint64_t dv0 = sdesc(sbase + kKVOff + 2 * kHalfBytes, kHalfBytes);
            Walk<kBal> ws = w;
            int ns = 0;     // S issued
            int seg_s = 0;  // segments whose Q tile the S cursor has taken
            int seg = 0;    // segments whose first PV has been issued
            for (int k = 0; w.more() && ok && !*abort_flag; w.next(a), ++k) {
                while (ws.more() && ns < k + NSB) {
                    const bool must = ns <= k + 1;
                    const int st = ns % kNS;
                    const bool q_new = ws.seg_first();
                    if (q_new && !(must ? bar_wait(B(kQReady), seg_s & 1) : bar_test(B(kQReady), seg_s & 1))) {
                        ok = !must;
                        break;
                    }
                    if (!(must ? bar_wait(B(Lt::kKFull + st), (ns / kNS) & 1)
                               : bar_test(B(Lt::kKFull + st), (ns / kNS) & 1))) {
                        ok = !must;
                        break;
                    }
                    if (q_new) ++seg_s;
                    fence_after();
                    const uint64_t dk = dk0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
                    const uint32_t sb = tmem + static_cast<uint32_t>((ns % NSB) * kTok);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {  // K = head_dim in 16-wide steps
                        const uint32_t kin = (ks & 3) * 32;
                        mma_bf16(sb, dq + (((ks >> 2) * kQHalf + kin) >> 4), dk + (((ks >> 2) * kHalfBytes + kin) >> 4),
                                 idesc(kTok, 0), ks > 0 ? 1u : 0u);
                    }
                    mma_commit(B(Lt::kSFull + ns % NSB));
                    if constexpr (kNS != NSB) mma_commit(B(Lt::kKEmpty + st));  // K of this stage no longer needed
                    ws.next(a);
                    ++ns;
                }
                if (!ok) break;
                const bool first = w.seg_first();
                // one P barrier per score buffer: the signal of tile k + NSB
                // cannot land on the phase awaited here
                if (!bar_wait(B(Lt::kPFull + k % NSB), (k / NSB) & 1) ||
                    !bar_wait(B(Lt::kVFull + k % kNS), (k / kNS) & 1)) {
                    ok = false;
                    break;
                }
                // a new segment overwrites O: the softmax warps have read out the last one
                if (first && seg > 0 && !bar_wait(B(kOFree), (seg - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (first) ++seg;
                fence_after();
                const uint64_t dv = dv0 + static_cast<uint64_t>(((k % kNS) * kStageBytes) >> 4);
                const uint32_t pb = tmem + static_cast<uint32_t>((k % NSB) * kTok);
#pragma unroll
                for (int ks = 0; ks < kTok / 16; ++ks)  // K = tokens in 16-wide steps: 8 TMEM columns of P each
                    mma_bf16_ta(tmem + Lt::kOCol, pb + 8 * ks, dv + ((ks * 16 * 128) >> 4), idesc(kDim, 1),
                                (!first || ks > 0) ? 1u : 0u);
                mma_commit(B(Lt::kPvDone + k % NSB));
                if constexpr (kNS != NSB) mma_commit(B(Lt::kVEmpty + k % kNS));
            }
            if (!ok) fail();
            mma_commit(B(kDone));  // completes once every MMA issued above has finished
            if (!bar_wait(B(kDone), 0)) fail();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------- softmax + epilogue
        const int m = threadIdx.x;  // query row of the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
        const int n = w.rt() * kRows + m;
        const bool valid = n < nq;
        const bool busy = w.rt() * kRows + 32 * warp < nq;  // the warp holds at least one query row
        const int qc = valid ? n / gh : 0;
        const float qk = a.qk_scale_log2;
        int grp = 0;  // group rendezvous completed
        // the four softmax warps meet (bounded; memory ordered through the mbarrier)
        auto group_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) bar_arrive(B(kGroup));
            const bool r = bar_wait_warp(B(kGroup), grp & 1);
            ++grp;
            return r;
        };
        // Q rows of a unit -> shared memory (swizzled K-major layout); padding
        // rows of busy warps are zero, those of idle warps are never read into
        // an output (each output row depends only on its own S and P rows)
        auto load_q = [&](int qb, int qh) {
            if (busy) {
                const uint4* src = reinterpret_cast<const uint4*>(
                    static_cast<const __nv_bfloat16*>(a.q) +
                    ((static_cast<size_t>(qb) * a.q_total + a.q_first + qc) * a.num_q_heads +
                     static_cast<size_t>(qh) * gh + (valid ? n % gh : 0)) *
                        kDim);
#pragma unroll 4
                for (int ch = 0; ch < 16; ++ch) {
                    const uint4 v = valid ? __ldg(src + ch) : make_uint4(0u, 0u, 0u, 0u);
                    *reinterpret_cast<uint4*>(smem + kQOff + tile_off(m, ch, kQHalf)) = v;
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) bar_arrive(B(kQReady));
        };
        if (w.more()) load_q(w.b, w.h);

        float m_used = -INFINITY, l = 0.f;
        int lim = 0;
        bool ok = true;
        for (int k = 0; w.more(); w.next(a), ++k) {
            const int s = k % Lt::kNSB, tok0 = w.t * kTok;  // score buffer
            if (w.seg_first()) {
                m_used = -INFINITY;
                l = 0.f;
                lim = valid ? w.L - C + qc + 1 : INT_MAX;  // tokens visible to this row
            }
            if (!bar_wait_warp(B(Lt::kSFull + s), (k / Lt::kNSB) & 1)) {
                ok = false;
                break;
            }
            fence_after();
            const uint32_t sa = tmem + lane_off + static_cast<uint32_t>(s * kTok);
            bool rescale = false;
            float alpha = 1.f;
            if (busy) {
                // the whole warp sees every token of the tile: no causal compares
                const bool full = __all_sync(0xFFFFFFFFu, tok0 + kTok <= lim);
                // the row's kTok scores into registers: one round trip to tensor memory
                uint32_t v[kTok];
#pragma unroll
                for (int c4 = 0; c4 < kTok / 32; ++c4) tmem_ld32_nowait(sa + 32 * c4, v + 32 * c4);
                asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
                // the tile's row max over visible tokens (of the raw scores when
                // the scale is positive, then scaled once)
                float mx = -INFINITY;
                if (full && qk > 0.f) {
                    float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int i = 0; i < kTok; i += 2)
                        m4[(i >> 1) & 3] = max3(m4[(i >> 1) & 3], __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                    mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * qk;
                } else {
#pragma unroll
                    for (int i = 0; i < kTok; ++i)
                        if (tok0 + i < lim) mx = fmaxf(mx, __uint_as_float(v[i]) * qk);
                }
                // lazy base: move it (and rescale O and l) only when the max grew by > 8
                const float m_new = fmaxf(m_used, mx);
                rescale = m_used != -INFINITY && m_new > m_used + 8.f;
                const float base_new = m_used == -INFINITY || rescale ? m_new : m_used;
                alpha = rescale ? ex2(m_used - m_new) : 1.f;
                m_used = base_new;
                const float base = m_used == -INFINITY ? 0.f : m_used;
                // probabilities -> P as BF16 pairs over the first kTok/2 columns of
                // this score buffer (P does not depend on O: this overlaps PV k-1)
                uint32_t pk[kTok / 2];
                float lt = 0.f;
                if (full) {
                    // two scores per fma / add instruction (packed f32x2)
                    float l0 = 0.f, l1 = 0.f;
#pragma unroll
                    for (int i = 0; i < kTok / 2; ++i) {
                        float x0, x1;
                        fma2(x0, x1, __uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), qk, qk, -base, -base);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        add2(l0, l1, l0, l1, p0, p1);
                        pk[i] = bf16x2(p0, p1);
                    }
                    lt = l0 + l1;
                } else {
#pragma unroll
                    for (int i = 0; i < kTok / 2; ++i) {
                        const int t0 = tok0 + 2 * i;
                        const float p0 = t0 < lim ? ex2(fmaf(__uint_as_float(v[2 * i]), qk, -base)) : 0.f;
                        const float p1 = t0 + 1 < lim ? ex2(fmaf(__uint_as_float(v[2 * i + 1]), qk, -base)) : 0.f;
                        lt += p0 + p1;
                        pk[i] = bf16x2(p0, p1);
                    }
                }
                l = l * alpha + lt;
                tmem_st32(sa, pk);
            }
            // PV completions, one barrier per score buffer.  A parity wait is
            // unambiguous while the barrier is at most one phase past the one
            // awaited.  Here every PV before S k has finished (S k, just read,
            // was issued after them, and MMAs complete in order), and PV k + 1
            // cannot finish before this softmax signals P k + 1: so the waits
            // below for PV k - 1 (a rescale of O) and PV k (the segment end)
            // see their phase, or the one before it, and need no other wait.
            const bool any_rescale = busy && __any_sync(0xFFFFFFFFu, rescale);
            if (any_rescale) {  // O is stable from PV k - 1 until P k is signalled
                if (!bar_wait_warp(B(Lt::kPvDone + (k - 1) % Lt::kNSB), ((k - 1) / Lt::kNSB) & 1)) {
                    ok = false;
                    break;
                }
                fence_after();
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {  // tcgen05.ld/st are warp-wide
                    uint32_t o[32];
                    const uint32_t oa = tmem + lane_off + Lt::kOCol + 32 * c4;
                    tmem_ld32(oa, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(oa, o);
                }
            }
            // V rows past the tile's tokens: zero (stale or unwritten rows could hold NaN)
            const int nvalid = min(kTok, w.t_end() - tok0);
            if (nvalid < kTok) {
                if (!bar_wait_warp(B(Lt::kVFull + k % kNS), (k / kNS) & 1)) {  // after the copy into this stage
                    ok = false;
                    break;
                }
                uint8_t* vs = smem + kKVOff + (k % kNS) * kStageBytes + 2 * kHalfBytes;
                for (int e = m; e < 2 * (kTok - nvalid) * 8; e += 128) {  // whole 128-byte rows: swizzle irrelevant
                    const int hf = e / ((kTok - nvalid) * 8), rem = e % ((kTok - nvalid) * 8);
                    const int r = nvalid + rem / 8, ch = rem % 8;
                    *reinterpret_cast<uint4*>(vs + hf * kHalfBytes + r * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_async_smem();  // (the PV MMA waits for all four warps' P signals)
            }
            fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(B(Lt::kPFull + s));
            if (!w.seg_last()) continue;

            // ---- segment end.  Every S of this segment is done (S k was the
            // last): the next unit's Q tile may replace this one now, so its
            // first S overlaps this epilogue.
            {
                Walk<kBal> wn = w;
                wn.next(a);
                if (wn.more()) load_q(wn.b, wn.h);
            }
            if (!bar_wait_warp(B(Lt::kPvDone + s), (k / Lt::kNSB) & 1)) {  // PV k
                ok = false;
                break;
            }
            fence_after();
            const float inv = l > 0.f ? a.v_scale / l : 0.f;
            const bool whole = w.whole();
            const int slot = w.cta_first() ? 0 : 1;
            const size_t prow = (static_cast<size_t>(blockIdx.x) * 2 + slot) * nq + (valid ? n : 0);
            if (busy) {
                __nv_bfloat16* orow = out_row(w.b, w.h, valid ? n : 0);
#pragma unroll 1
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t v[32];
                    tmem_ld32(tmem + lane_off + Lt::kOCol + 32 * c4, v);
                    if (!valid) continue;
                    if (whole) {  // O / l -> BF16 output row
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 o;
                            o.x = bf16x2(__uint_as_float(v[8 * q4 + 0]) * inv, __uint_as_float(v[8 * q4 + 1]) * inv);
                            o.y = bf16x2(__uint_as_float(v[8 * q4 + 2]) * inv, __uint_as_float(v[8 * q4 + 3]) * inv);
                            o.z = bf16x2(__uint_as_float(v[8 * q4 + 4]) * inv, __uint_as_float(v[8 * q4 + 5]) * inv);
                            o.w = bf16x2(__uint_as_float(v[8 * q4 + 6]) * inv, __uint_as_float(v[8 * q4 + 7]) * inv);
                            *reinterpret_cast<uint4*>(orow + 32 * c4 + 8 * q4) = o;
                        }
                    } else {  // this CTA's piece: O / l in fp32, and its log-sum-exp
                        float4* dst = reinterpret_cast<float4*>(a.bal_o + prow * kDim + 32 * c4);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(__uint_as_float(v[4 * q4 + 0]) * inv, __uint_as_float(v[4 * q4 + 1]) * inv,
                                                  __uint_as_float(v[4 * q4 + 2]) * inv, __uint_as_float(v[4 * q4 + 3]) * inv);
                    }
                }
            }
            // O is read: the next segment's first PV may overwrite it
            fence_before();
            __syncwarp();
            if (lane == 0) bar_arrive(B(kOFree));
            if (whole) continue;
            if constexpr (kBal) {
                if (valid) a.bal_lse[prow] = l > 0.f ? m_used + log2f(l) : -INFINITY;
                // Publish: every thread's partial writes are fenced before the
                // rendezvous, after which one GPU-scope acq_rel atomic counts the
                // piece (and, for the last one, orders the others' writes before
                // the reads below).
                __threadfence();
                if (!group_sync()) {
                    ok = false;
                    break;
                }
                // the CTAs c_first .. c_first + pieces - 1 own the unit's tiles
                // [ps, ps + nt); CTA c owns [c T / P, (c + 1) T / P)
                const long long T = range[1], P = range[2];
                const long long ps = range[0] + w.k - w.t;
                auto owner = [&](long long x) { return ((x + 1) * P - 1) / T; };
                const long long cf = owner(ps);
                const int pieces = static_cast<int>(owner(ps + w.nt - 1) - cf + 1);
                const int s_first = (cf * T / P < ps) ? 1 : 0;
                int* counter = a.counters + static_cast<size_t>(w.b) * a.num_kv_heads + w.h;
                if (m == 0) *last_flag = atom_add_acq_rel(counter, 1) == pieces - 1 ? 1 : 0;
                if (!group_sync()) {
                    ok = false;
                    break;
                }
                if (!*last_flag) continue;
                __threadfence();
                // pass 1: per row, the largest log-sum-exp M and 1/z, z = sum_j 2^(lse_j - M)
                if (valid) {
                    float M = -INFINITY, z = 0.f;
                    for (int j = 0; j < pieces; ++j) {
                        const float lj =
                            __ldcg(a.bal_lse + (static_cast<size_t>(cf + j) * 2 + (j == 0 ? s_first : 0)) * nq + n);
                        if (lj == -INFINITY) continue;  // a piece with no token for this query
                        const float Mn = fmaxf(M, lj);
                        z = z * exp2f(M - Mn) + exp2f(lj - Mn);
                        M = Mn;
                    }
                    merge_m[m] = M;
                    merge_m[kRows + m] = z > 0.f ? 1.f / z : 0.f;
                }
                if (!group_sync()) {
                    ok = false;
                    break;
                }
                // pass 2: thread m owns 4-float chunks m, m + 128, ... of the rows
                // (32 per row), kMC at a time, with one round of independent loads per piece
                const int nch = (nq * (kDim / 4) + 127) / 128;
#pragma unroll 1
                for (int c0 = 0; c0 < nch; c0 += kMC) {
                    float4 acc[kMC];
#pragma unroll
                    for (int u = 0; u < kMC; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int j = 0; j < pieces; ++j) {
                        const size_t pb = (static_cast<size_t>(cf + j) * 2 + (j == 0 ? s_first : 0)) * nq;
#pragma unroll
                        for (int u = 0; u < kMC; ++u) {
                            const int idx = m + 128 * (c0 + u), r = idx >> 5, d4 = idx & 31;
                            if (c0 + u >= nch || r >= nq) continue;
                            const float lj = __ldcg(a.bal_lse + pb + r);
                            const float4 o4 = __ldcg(reinterpret_cast<const float4*>(a.bal_o + (pb + r) * kDim) + d4);
                            const float wt = lj == -INFINITY ? 0.f : exp2f(lj - merge_m[r]) * merge_m[kRows + r];
                            acc[u].x = fmaf(wt, o4.x, acc[u].x);
                            acc[u].y = fmaf(wt, o4.y, acc[u].y);
                            acc[u].z = fmaf(wt, o4.z, acc[u].z);
                            acc[u].w = fmaf(wt, o4.w, acc[u].w);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kMC; ++u) {
                        const int idx = m + 128 * (c0 + u), r = idx >> 5, d4 = idx & 31;
                        if (c0 + u >= nch || r >= nq) continue;
                        uint2 pk;
                        pk.x = bf16x2(acc[u].x, acc[u].y);
                        pk.y = bf16x2(acc[u].z, acc[u].w);
                        *reinterpret_cast<uint2*>(out_row(w.b, w.h, r) + 4 * d4) = pk;
                    }
                }
                if (m == 0) *counter = 0;  // ready for the next call
                // merge_m is rewritten only after two more rendezvous
            }
        }
        if (!ok) {
            if (lane == 0) fail();
        } else if (kBal && !*abort_flag) {
            // zero the rows of sequences with nothing visible (and report bad lengths once)
            const size_t per_seq = static_cast<size_t>(C) * a.num_q_heads * kDim;
            for (int b = blockIdx.x; b < a.num_seqs; b += gridDim.x) {
                if (visible_len(a, b, m == 0) != 0) continue;
                uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                                    (static_cast<size_t>(b) * a.q_total + a.q_first) * a.num_q_heads * kDim);
                for (size_t i = m; i < per_seq / 8; i += 128) o[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    // teardown: every role has finished its waits (all bounded); free TMEM
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(Lt::kTmemCols)
                     : "memory");
}

template <bool kBal, int kNS>
cudaError_t launch_tc(const DecodeArgs& a, const CUtensorMap* tk, const CUtensorMap* tv, dim3 grid,
                      cudaStream_t stream) {
    constexpr int kSmem = Cfg<kNS>::kSmem;
    static int configured_mask = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 31) return cudaErrorNotSupported;
    if (!(configured_mask & (1 << dev))) {
        cudaError_t e =
            cudaFuncSetAttribute(attention_tc_kernel<kBal, kNS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
        if (e == cudaSuccess)  // the largest carveout, so that two CTAs fit per SM
            e = cudaFuncSetAttribute(attention_tc_kernel<kBal, kNS>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                     cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        configured_mask |= 1 << dev;
    }
    // (Cfg<kNS>::kCtasPerSm CTAs per SM by shared memory; each allocates 256 TMEM columns)
    attention_tc_kernel<kBal, kNS><<<grid, kThreads, kSmem, stream>>>(*tk, *tv, a);
    return cudaGetLastError();
}

}  // namespace

bool attention_tc_supported(pkv_dtype kv, int head_dim, int block_size) {
    return kv == PKV_BF16 && head_dim == kDim && (block_size == 16 || block_size == 32 || block_size == 64);
}

cudaError_t launch_attention_tc(const DecodeArgs& a, const void* tmap_k, const void* tmap_v, cudaStream_t stream) {
    const CUtensorMap* tk = static_cast<const CUtensorMap*>(tmap_k);
    const CUtensorMap* tv = static_cast<const CUtensorMap*>(tmap_v);
    const int nq = a.num_queries * (a.num_q_heads / a.num_kv_heads);
    if (a.bal_max_ctas > 0) {
        if (nq > kRows || !a.bal_o || !a.bal_lse || !a.counters) return cudaErrorInvalidValue;
        return launch_tc<true, 2>(a, tk, tv, dim3(a.bal_max_ctas), stream);
    }
    return launch_tc<false, 2>(a, tk, tv, dim3((nq + kRows - 1) / kRows, a.num_kv_heads, a.num_seqs), stream);
}

}  // namespace pkv
