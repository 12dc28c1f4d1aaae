// C ABI of libpkv.so: argument validation, split planning and launches.
// Everything here runs on the host; it allocates no device memory and never
// synchronises a stream.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "pkv_internal.h"

namespace pkv {

namespace {
thread_local char g_last_cuda_error[256] = "";
// pkv_set_first_wait_limit_for_testing: polls (< 0: off) and the CTA it targets
thread_local int32_t g_test_wait_polls = -1;
thread_local int32_t g_test_wait_cta = -1;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool valid_dtype(pkv_dtype t) { return t == PKV_F32 || t == PKV_BF16 || t == PKV_FP8_E4M3; }

pkv_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return PKV_OK;
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    set_last_error(e);
    return PKV_ERR_CUDA;
}

int g_sms[64] = {0};

// Balanced persistent schedule: at most this many sequences (each CTA scans
// the lengths once), at most kBalCtasPerSm CTAs per SM.
constexpr int kMaxBalancedSeqs = 4096;
constexpr int kBalCtasPerSm = 2;

size_t counters_bytes(int B, int Hkv) { return round_up(static_cast<size_t>(B) * Hkv * sizeof(int32_t), 256); }
size_t fixed_bytes(int B, int Hq, int D, int64_t ns) {
    if (ns <= 1) return 0;
    const size_t rows = static_cast<size_t>(B) * Hq * ns;
    return round_up(rows * D * sizeof(float), 256) + round_up(rows * sizeof(float), 256);
}
int bal_ctas() { return (num_sms() > 0 ? num_sms() : 148) * kBalCtasPerSm; }
size_t bal_o_bytes(int ctas, int G, int D) { return round_up(static_cast<size_t>(ctas) * 2 * G * D * sizeof(float), 256); }
size_t bal_bytes(int ctas, int G, int D) {
    return bal_o_bytes(ctas, G, D) + round_up(static_cast<size_t>(ctas) * 2 * G * sizeof(float), 256);
}

// Queries per launch.  A launch serves rows = queries x gh query rows per KV
// head: at most kMmaMaxRows for the tensor-core design; for the SIMT design
// a power of two up to kSimtMaxRows.  Longer query lists run as several
// launches over consecutive query chunks.
int mma_chunk(int gh, int C) {
    const int cap = gh <= kMmaMaxRows ? kMmaMaxRows / gh : 1;
    return C < cap ? C : cap;
}
int simt_chunk(const pkv_pool* p, int gh, int C) {
    int cap = gh <= kSimtMaxRows ? kSimtMaxRows / gh : 1;
    if (C < cap) cap = C;
    int c = 1;
    while (c * 2 <= cap) c *= 2;
    while (c > 1 && !decode_simt_supported(p->d.kv_dtype, p->d.head_dim, c * gh)) c /= 2;
    return c;
}
// Template row bound of the tensor-core kernel for `rows` rows.
int row_bound(int rows) {
    int p = 1;
    while (p < rows) p *= 2;
    return p;
}
constexpr int kMaxQueries = 1 << 20;
constexpr int kTcMinRows = 8;  // query rows per KV head from which AUTO takes the tcgen05 design
// Up to this many query rows per KV head (one 128-row tile) the tcgen05
// design can run the balanced persistent schedule.
constexpr int kTcBalMaxRows = 128;
// The tcgen05 design takes the balanced schedule when one CTA per (sequence,
// KV head) would leave CTA slots idle (a few long sequences).  With enough
// units the grid keeps every SM busy, and whole units need no Q reload or
// merge at segment ends, so the grid is as fast or faster.
bool tc_balanced(int num_seqs, int num_kv_heads, int64_t rows) {
    return rows <= kTcBalMaxRows && num_seqs <= kMaxBalancedSeqs &&
           static_cast<int64_t>(num_seqs) * num_kv_heads < bal_ctas();
}
// Rows of one balanced-schedule partial slot: the template row bound of the
// largest launch (a KV-head pair's 2 * gh rows for decode).
int bal_rows(int gh, int C) {
    const int r = row_bound(mma_chunk(gh, C) * gh);
    const int pair = (C == 1 && 2 * gh <= 8) ? row_bound(2 * gh) : 0;
    return r > pair ? r : pair;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// TMA descriptors over the whole K and V pools, viewed as 2D tensors
// [rows = layers*blocks*kv_heads*block_size][head_dim]; one box is one
// (block, kv head) chunk of 64 BF16 or 128 E4M3 columns, 128-byte swizzled.
bool ensure_tmaps(pkv_pool* p) {
    if (p->tmap_state != 0) return p->tmap_state == 1;
    p->tmap_state = -1;
    const pkv_pool_desc& d = p->d;
    if (d.kv_dtype != PKV_BF16 && d.kv_dtype != PKV_FP8_E4M3) return false;
    const uint64_t rows = static_cast<uint64_t>(d.num_layers) * d.num_blocks * d.num_kv_heads * d.block_size;
    if (rows > static_cast<uint64_t>(INT32_MAX)) return false;
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const bool bf16 = d.kv_dtype == PKV_BF16;
    if (bf16 && d.head_dim == 128) {
        // One box per (block, kv head): dims {64 columns, rows, 2 halves} with
        // the half stride (128 B) inside the row stride (256 B), so the box
        // lands as [half][bs rows][128 B].
        const cuuint64_t dims3[3] = {64, rows, 2};
        const cuuint64_t strides3[2] = {256, 128};
        const cuuint32_t box3[3] = {64, static_cast<cuuint32_t>(d.block_size), 2};
        const cuuint32_t estr3[3] = {1, 1, 1};
        bool ok3 = true;
        for (int i = 0; i < 2 && ok3; ++i) {
            CUresult r = enc(i == 0 ? &p->tmap_k : &p->tmap_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                             i == 0 ? d.k_base : d.v_base, dims3, strides3, box3, estr3,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            ok3 = r == CUDA_SUCCESS;
        }
        if (ok3) {
            p->tmap_3d = 1;
            p->tmap_state = 1;
            // Boxes of one 64-column half of a block (the tcgen05 kernel keeps
            // the two halves of a tile apart).
            const cuuint32_t boxh[3] = {64, static_cast<cuuint32_t>(d.block_size), 1};
            bool okh = true;
            for (int i = 0; i < 2 && okh; ++i) {
                CUresult r = enc(i == 0 ? &p->tmap_kh : &p->tmap_vh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                 i == 0 ? d.k_base : d.v_base, dims3, strides3, boxh, estr3,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
                okh = r == CUDA_SUCCESS;
            }
            p->tmap_half = okh ? 1 : 0;
            // Boxes of two adjacent KV heads of a block (the rows of head h+1
            // follow those of head h): 8 KB per box at 16-token blocks.
            p->tmap_pair = 0;
            if (d.block_size == 16 && d.num_kv_heads % 2 == 0) {
                const cuuint32_t box2[3] = {64, static_cast<cuuint32_t>(2 * d.block_size), 2};
                bool ok2 = true;
                for (int i = 0; i < 2 && ok2; ++i) {
                    CUresult r = enc(i == 0 ? &p->tmap_k2 : &p->tmap_v2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                     i == 0 ? d.k_base : d.v_base, dims3, strides3, box2, estr3,
                                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
                    ok2 = r == CUDA_SUCCESS;
                }
                p->tmap_pair = ok2 ? 1 : 0;
            }
            return true;
        }
    }
    p->tmap_3d = 0;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.head_dim), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.head_dim) * p->elem_bytes};
    const cuuint32_t box[2] = {bf16 ? 64u : 128u, static_cast<cuuint32_t>(d.block_size)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    for (int i = 0; i < 2; ++i) {
        CUresult r = enc(i == 0 ? &p->tmap_k : &p->tmap_v, dt, 2, i == 0 ? d.k_base : d.v_base, dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return false;
    }
    p->tmap_state = 1;
    return true;
}
}  // namespace

void set_last_error(cudaError_t e) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
}

int dtype_bytes(pkv_dtype t) {
    switch (t) {
        case PKV_F32: return 4;
        case PKV_BF16: return 2;
        case PKV_FP8_E4M3: return 1;
    }
    return 0;
}

size_t workspace_counter_bytes(int num_seqs, int num_kv_heads) { return counters_bytes(num_seqs, num_kv_heads); }

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64 && g_sms[dev] > 0) return g_sms[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) g_sms[dev] = n;
    return n;
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char* pkv_status_string(pkv_status s) {
    switch (s) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported geometry or dtype";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_DEVICE_BOUNDS: return "device-side index out of bounds";
        case PKV_ERR_OUT_OF_BLOCKS: return "out of KV blocks";
        case PKV_ERR_INCONSISTENT: return "block manager invariant violated";
    }
    return "unknown status";
}

const char* pkv_last_cuda_error(void) { return g_last_cuda_error; }

void pkv_set_first_wait_limit_for_testing(int32_t polls, int32_t cta) {
    g_test_wait_polls = polls < 0 ? -1 : polls;
    g_test_wait_cta = cta < 0 ? -1 : cta;
}

int64_t kv_bytes_per_token(int32_t num_layers, int32_t num_kv_heads, int32_t head_dim, pkv_dtype dtype) {
    return 2LL * num_layers * num_kv_heads * head_dim * dtype_bytes(dtype);
}

size_t kv_pool_tensor_bytes(const pkv_pool_desc* d) {
    if (!d || !valid_dtype(d->kv_dtype)) return 0;
    return static_cast<size_t>(d->num_layers) * d->num_blocks * d->num_kv_heads * d->block_size *
           d->head_dim * dtype_bytes(d->kv_dtype);
}

pkv_status kv_pool_create(const pkv_pool_desc* d, pkv_pool** out) {
    if (!d || !out) return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    if (!valid_dtype(d->kv_dtype)) return PKV_ERR_INVALID_ARG;
    if (d->num_layers < 1 || d->num_blocks < 1 || d->num_kv_heads < 1) return PKV_ERR_INVALID_ARG;
    if (d->block_size != 16 && d->block_size != 32 && d->block_size != 64) return PKV_ERR_UNSUPPORTED;
    if (d->head_dim != 64 && d->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (!d->k_base || !d->v_base || !aligned(d->k_base, 16) || !aligned(d->v_base, 16))
        return PKV_ERR_INVALID_ARG;
    if (d->error_word && !aligned(d->error_word, 4)) return PKV_ERR_INVALID_ARG;
    // slots and element offsets are int64; keep one layer's slot count in int32
    if (static_cast<int64_t>(d->num_blocks) * d->block_size > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    float ks = 1.f, vs = 1.f;
    if (d->kv_dtype == PKV_FP8_E4M3) {
        if (!(std::isfinite(d->k_scale) && d->k_scale > 0.f && std::isfinite(d->v_scale) && d->v_scale > 0.f))
            return PKV_ERR_INVALID_ARG;
        ks = d->k_scale;
        vs = d->v_scale;
    }
    // CUtensorMap needs 64-byte alignment
    pkv_pool* p = static_cast<pkv_pool*>(std::aligned_alloc(64, round_up(sizeof(pkv_pool), 64)));
    if (!p) return PKV_ERR_INVALID_ARG;
    std::memset(p, 0, sizeof(pkv_pool));
    p->d = *d;
    p->d.k_scale = ks;
    p->d.v_scale = vs;
    p->elem_bytes = dtype_bytes(d->kv_dtype);
    p->layer_bytes = static_cast<size_t>(d->num_blocks) * d->num_kv_heads * d->block_size * d->head_dim *
                     p->elem_bytes;
    volatile float one = 1.f;  // one binary32 division each, on the host
    p->k_inv_scale = one / ks;
    p->v_inv_scale = one / vs;
    *out = p;
    return PKV_OK;
}

void kv_pool_destroy(pkv_pool* p) { std::free(p); }

pkv_status kv_append(const pkv_pool* p, int32_t layer, const void* k, const void* v, pkv_dtype in_dtype,
                     const int64_t* slot_mapping, int32_t num_tokens, void* stream) {
    if (!p || layer < 0 || layer >= p->d.num_layers || num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (in_dtype != PKV_F32 && in_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (p->d.kv_dtype == PKV_F32 && in_dtype != PKV_F32) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8))
        return PKV_ERR_INVALID_ARG;
    return cuda_status(launch_kv_append(p, layer, k, v, in_dtype, slot_mapping, num_tokens,
                                        static_cast<cudaStream_t>(stream)));
}

pkv_status paged_multi_query_plan(const pkv_pool* p, int32_t num_seqs, int32_t num_queries, int32_t num_q_heads,
                                  int32_t max_seq_len, int32_t split_tokens, int32_t* split_out,
                                  int32_t* nsplit_out, size_t* ws_out) {
    if (!p || num_seqs < 0 || num_q_heads < 1 || max_seq_len < 0 || split_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (num_queries < 1 || num_queries > kMaxQueries) return PKV_ERR_INVALID_ARG;
    if (num_q_heads % p->d.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    int S = split_tokens;
    if (S > 0) {
        if (S % kTileTokens != 0 || S % p->d.block_size != 0) return PKV_ERR_INVALID_ARG;
    } else {
        // Auto: 1024-token splits, halved (down to one tile) while the batch
        // would give fewer than two CTAs per SM.
        const int sms = num_sms() > 0 ? num_sms() : 148;
        const int64_t pairs = static_cast<int64_t>(num_seqs) * p->d.num_kv_heads;
        S = 1024;
        while (S > kTileTokens && pairs * ((max_seq_len + S - 1) / S) < 2LL * sms) S /= 2;
        if (S % p->d.block_size != 0) S = p->d.block_size > kTileTokens ? p->d.block_size : kTileTokens;
    }
    int64_t ns = max_seq_len > 0 ? (static_cast<int64_t>(max_seq_len) + S - 1) / S : 1;
    if (ns < 1) ns = 1;
    if (ns > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    // layout: [counters][partials of whichever schedule the call runs], sized
    // for the largest query chunk of either design (the tensor-core one's)
    const int gh = num_q_heads / p->d.num_kv_heads;
    const int cq = mma_chunk(gh, num_queries);
    size_t body = fixed_bytes(num_seqs, cq * num_q_heads, p->d.head_dim, ns);
    if (split_tokens == 0 && num_seqs <= kMaxBalancedSeqs) {
        size_t bb = bal_bytes(bal_ctas(), bal_rows(gh, num_queries), p->d.head_dim);
        // the tcgen05 design's balanced schedule: one slot row per query row
        if (static_cast<int64_t>(num_queries) * gh <= kTcBalMaxRows) {
            const size_t bt = bal_bytes(bal_ctas(), num_queries * gh, p->d.head_dim);
            if (bt > bb) bb = bt;
        }
        if (bb > body) body = bb;
    }
    size_t ws = body > 0 ? counters_bytes(num_seqs, p->d.num_kv_heads) + body : 0;
    if (split_out) *split_out = S;
    if (nsplit_out) *nsplit_out = static_cast<int32_t>(ns);
    if (ws_out) *ws_out = ws;
    return PKV_OK;
}

pkv_status paged_decode_plan(const pkv_pool* p, int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                             int32_t split_tokens, int32_t* split_out, int32_t* nsplit_out, size_t* ws_out) {
    return paged_multi_query_plan(p, num_seqs, 1, num_q_heads, max_seq_len, split_tokens, split_out, nsplit_out,
                                  ws_out);
}

int32_t paged_decode_algo(const pkv_pool* p, int32_t G, pkv_algo algo) {
    if (!p || G < 1) return -1;
    pkv_pool* mp = const_cast<pkv_pool*>(p);
    const bool mma_ok = decode_mma_supported(p->d.kv_dtype, p->d.head_dim, G, p->d.block_size);
    const bool simt_ok = decode_simt_supported(p->d.kv_dtype, p->d.head_dim, G);
    if (algo == PKV_ALGO_MMA) return (mma_ok && ensure_tmaps(mp)) ? PKV_ALGO_MMA : -1;
    if (algo == PKV_ALGO_SIMT) return simt_ok ? PKV_ALGO_SIMT : -1;
    if (algo != PKV_ALGO_AUTO) return -1;
    if (mma_ok && ensure_tmaps(mp)) return PKV_ALGO_MMA;
    return simt_ok ? PKV_ALGO_SIMT : -1;
}

}  // extern "C"

namespace pkv {
namespace {
// The kernel design a call runs: PKV_ALGO_TC (tcgen05, whole query list in
// one launch; the default from kTcMinRows query rows per KV head), MMA or
// SIMT, or -1 when the request cannot be served.  fused: the decode step's
// append runs inside the launch (tensor-core design only).
int design_for(const pkv_pool* p, int C, int gh, int split_tokens, pkv_algo algo, bool fused) {
    pkv_pool* mp = const_cast<pkv_pool*>(p);  // the handle caches its TMA descriptors
    const bool tc_fits = attention_tc_supported(p->d.kv_dtype, p->d.head_dim, p->d.block_size) && !fused &&
                         split_tokens == 0 && static_cast<int64_t>(C) * gh <= (1 << 24);
    const bool mma_fits = decode_mma_supported(p->d.kv_dtype, p->d.head_dim, mma_chunk(gh, C) * gh, p->d.block_size);
    const bool simt_fits = decode_simt_supported(p->d.kv_dtype, p->d.head_dim, simt_chunk(p, gh, C) * gh);
    int d = -1;
    if (algo == PKV_ALGO_TC) {
        d = tc_fits && ensure_tmaps(mp) && p->tmap_half == 1 ? PKV_ALGO_TC : -1;
    } else if (algo == PKV_ALGO_MMA) {
        d = mma_fits && ensure_tmaps(mp) ? PKV_ALGO_MMA : -1;
    } else if (algo == PKV_ALGO_SIMT) {
        d = simt_fits ? PKV_ALGO_SIMT : -1;
    } else if (algo == PKV_ALGO_AUTO) {
        if (tc_fits && C > 1 && C * gh >= kTcMinRows && ensure_tmaps(mp) && p->tmap_half == 1)
            d = PKV_ALGO_TC;
        else if (mma_fits && ensure_tmaps(mp))
            d = PKV_ALGO_MMA;
        else if (simt_fits)
            d = PKV_ALGO_SIMT;
    }
    if (fused && (d != PKV_ALGO_MMA || C != 1 || gh > 8)) return -1;
    return d;
}

// Attention for C queries per sequence; with new_k != nullptr (decode only)
// the kernel also appends each sequence's newest token.
pkv_status attention_call(const void* q, pkv_dtype q_dtype, const pkv_pool* p, int32_t layer,
                          const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                          int32_t num_seqs, int32_t num_queries, int32_t num_q_heads, int32_t max_seq_len,
                          float scale, int32_t split_tokens, pkv_algo algo, void* workspace, size_t workspace_bytes,
                          void* out, void* stream, const void* new_k, const void* new_v, pkv_dtype new_dtype,
                          bool dry_run = false) {
    if (!p || layer < 0 || layer >= p->d.num_layers) return PKV_ERR_INVALID_ARG;
    if (num_queries < 1 || num_queries > kMaxQueries) return PKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_q_heads < 1 || max_blocks_per_seq < 1 || max_seq_len < 0) return PKV_ERR_INVALID_ARG;
    if (num_q_heads % p->d.num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * p->d.block_size)
        return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
    const pkv_dtype want_q = p->d.kv_dtype == PKV_F32 ? PKV_F32 : PKV_BF16;
    if (q_dtype != want_q) return PKV_ERR_UNSUPPORTED;
    if (algo != PKV_ALGO_AUTO && algo != PKV_ALGO_SIMT && algo != PKV_ALGO_MMA && algo != PKV_ALGO_TC)
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    if (!q || !out || !block_tables || !seq_lens) return PKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PKV_ERR_INVALID_ARG;
    const int gh = num_q_heads / p->d.num_kv_heads;  // query heads per KV head
    const int cq_mma = mma_chunk(gh, num_queries);  // the largest chunk: sizes the fixed-split partials
    const int design = design_for(p, num_queries, gh, split_tokens, algo, new_k != nullptr);
    if (design < 0) return PKV_ERR_UNSUPPORTED;
    const bool use_tc = design == PKV_ALGO_TC, use_mma = design == PKV_ALGO_MMA;

    int32_t S = 0, NS = 0;
    size_t need = 0;
    pkv_status st =
        paged_multi_query_plan(p, num_seqs, num_queries, num_q_heads, max_seq_len, split_tokens, &S, &NS, &need);
    if (st != PKV_OK) return st;
    const bool tc_bal = use_tc && split_tokens == 0 && tc_balanced(num_seqs, p->d.num_kv_heads, static_cast<int64_t>(num_queries) * gh);
    if ((!use_tc || tc_bal) && need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
        return PKV_ERR_WORKSPACE;
    if (dry_run) return PKV_OK;  // every host-side check passed; nothing enqueued

    DecodeArgs a{};
    a.q = q;
    a.out = out;
    a.k_layer = static_cast<const uint8_t*>(p->d.k_base) + static_cast<size_t>(layer) * p->layer_bytes;
    a.v_layer = static_cast<const uint8_t*>(p->d.v_base) + static_cast<size_t>(layer) * p->layer_bytes;
    a.tables = block_tables;
    a.lens = seq_lens;
    a.err = p->d.error_word;
    a.layer = layer;
    a.tma_3d = p->tmap_3d;
    a.max_blocks = max_blocks_per_seq;
    a.max_len = max_seq_len;
    a.num_seqs = num_seqs;
    a.q_total = num_queries;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = p->d.num_kv_heads;
    a.head_dim = p->d.head_dim;
    a.block_size = p->d.block_size;
    a.num_blocks = p->d.num_blocks;
    a.split_tokens = S;
    a.num_splits = NS;
    const bool balanced = use_mma && split_tokens == 0 && num_seqs <= kMaxBalancedSeqs;
    const float log2e = 1.4426950408889634f;
    a.qk_scale_log2 = scale * p->d.k_scale * log2e;
    a.v_scale = p->d.v_scale;
    if (g_test_wait_polls >= 0) {
        a.test_wait_on = 1;
        a.test_wait_polls = static_cast<uint32_t>(g_test_wait_polls);
        a.test_wait_cta = g_test_wait_cta;
    }
    if (new_k) {
        a.new_k = static_cast<const uint8_t*>(new_k);
        a.new_v = static_cast<const uint8_t*>(new_v);
        a.new_dtype = new_dtype;
        a.k_inv_scale = p->k_inv_scale;
        a.v_inv_scale = p->v_inv_scale;
        a.k_layer_w = static_cast<uint8_t*>(p->d.k_base) + static_cast<size_t>(layer) * p->layer_bytes;
        a.v_layer_w = static_cast<uint8_t*>(p->d.v_base) + static_cast<size_t>(layer) * p->layer_bytes;
    }
    if (need > 0) {
        uint8_t* w = static_cast<uint8_t*>(workspace);
        a.counters = reinterpret_cast<int32_t*>(w);
        uint8_t* body = w + counters_bytes(num_seqs, p->d.num_kv_heads);
        if (balanced || tc_bal) {
            a.bal_max_ctas = bal_ctas();
            a.bal_o = reinterpret_cast<float*>(body);
            const int rows = tc_bal ? num_queries * gh : bal_rows(gh, num_queries);
            a.bal_lse = reinterpret_cast<float*>(body + bal_o_bytes(a.bal_max_ctas, rows, p->d.head_dim));
        } else if (NS > 1) {
            const size_t rows = static_cast<size_t>(num_seqs) * cq_mma * num_q_heads * NS;
            a.o_part = reinterpret_cast<float*>(body);
            a.lse_part = reinterpret_cast<float*>(body + round_up(rows * p->d.head_dim * sizeof(float), 256));
        }
    }
    // Decode on BF16 pools of 16-token blocks: one CTA serves two adjacent KV
    // heads, so each block arrives as one 8 KB box instead of two 4 KB ones
    // (per-box cost dominates at 4 KB).
    const bool pair = use_mma && num_queries == 1 && p->tmap_pair == 1 && p->tmap_3d == 1 && 2 * gh <= 8;
    a.heads_per_cta = pair ? 2 : 1;
    const void* tk = pair ? &p->tmap_k2 : &p->tmap_k;
    const void* tv = pair ? &p->tmap_v2 : &p->tmap_v;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (use_tc) {  // the balanced schedule (bal_max_ctas > 0) or one CTA per row tile
        a.heads_per_cta = 1;
        a.q_first = 0;
        a.num_queries = num_queries;
        a.len_trim = 0;
        if (!tc_bal) a.bal_max_ctas = 0;
        return cuda_status(launch_attention_tc(a, &p->tmap_kh, &p->tmap_vh, s));
    }
    // one launch (plus combine) per query chunk; a chunk reads only the tokens
    // its last query can see
    for (int c0 = 0; c0 < num_queries;) {
        int cq = use_mma ? mma_chunk(gh, num_queries - c0) : simt_chunk(p, gh, num_queries - c0);
        a.q_first = c0;
        a.num_queries = cq;
        a.len_trim = num_queries - c0 - cq;
        cudaError_t e = use_mma ? launch_decode_mma(p->d.kv_dtype, a, tk, tv, s) : launch_decode_simt(p->d.kv_dtype, a, s);
        if (e != cudaSuccess) return cuda_status(e);
        if (!balanced && NS > 1) {
            e = launch_combine(q_dtype, a, s);
            if (e != cudaSuccess) return cuda_status(e);
        }
        c0 += cq;
    }
    return PKV_OK;
}
}  // namespace

pkv_status decode_attention_check(const void* q, pkv_dtype q_dtype, const pkv_pool* p, int32_t layer,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len, float scale,
                                  int32_t split_tokens, pkv_algo algo, void* workspace, size_t workspace_bytes,
                                  void* out) {
    return attention_call(q, q_dtype, p, layer, block_tables, max_blocks_per_seq, seq_lens, num_seqs, 1, num_q_heads,
                          max_seq_len, scale, split_tokens, algo, workspace, workspace_bytes, out, nullptr, nullptr,
                          nullptr, PKV_BF16, true);
}
}  // namespace pkv

extern "C" {

pkv_status paged_multi_query_attention(const void* q, pkv_dtype q_dtype, const pkv_pool* p, int32_t layer,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* seq_lens, int32_t num_seqs, int32_t num_queries,
                                       int32_t num_q_heads, int32_t max_seq_len, float scale, int32_t split_tokens,
                                       pkv_algo algo, void* workspace, size_t workspace_bytes, void* out,
                                       void* stream) {
    return pkv::attention_call(q, q_dtype, p, layer, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                               num_queries, num_q_heads, max_seq_len, scale, split_tokens, algo, workspace,
                               workspace_bytes, out, stream, nullptr, nullptr, PKV_BF16);
}

int32_t paged_multi_query_algo(const pkv_pool* p, int32_t num_queries, int32_t num_q_heads, int32_t split_tokens,
                               pkv_algo algo) {
    if (!p || num_queries < 1 || num_queries > pkv::kMaxQueries || num_q_heads < 1 ||
        num_q_heads % p->d.num_kv_heads != 0 || split_tokens < 0)
        return -1;
    return pkv::design_for(p, num_queries, num_q_heads / p->d.num_kv_heads, split_tokens, algo, false);
}

pkv_status paged_decode_append_attention(const void* q, pkv_dtype q_dtype, const void* k_new, const void* v_new,
                                         pkv_dtype in_dtype, const pkv_pool* p, int32_t layer,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_seq_len, float scale, int32_t split_tokens, pkv_algo algo,
                                         void* workspace, size_t workspace_bytes, void* out, void* stream) {
    if (!p) return PKV_ERR_INVALID_ARG;
    if (in_dtype != PKV_BF16 && in_dtype != PKV_F32) return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 0 && (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16))) return PKV_ERR_INVALID_ARG;
    return pkv::attention_call(q, q_dtype, p, layer, block_tables, max_blocks_per_seq, seq_lens, num_seqs, 1,
                               num_q_heads, max_seq_len, scale, split_tokens, algo, workspace, workspace_bytes, out,
                               stream, num_seqs > 0 ? k_new : nullptr, v_new, in_dtype);
}

pkv_status paged_decode_attention(const void* q, pkv_dtype q_dtype, const pkv_pool* p, int32_t layer,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_seq_len, float scale, int32_t split_tokens, pkv_algo algo,
                                  void* workspace, size_t workspace_bytes, void* out, void* stream) {
    return paged_multi_query_attention(q, q_dtype, p, layer, block_tables, max_blocks_per_seq, seq_lens, num_seqs, 1,
                                       num_q_heads, max_seq_len, scale, split_tokens, algo, workspace,
                                       workspace_bytes, out, stream);
}

}  // extern "C"
