// Internal declarations shared by the translation units of libpkv.so.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached through the runtime)
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "pkv.h"

// The validated pool handle behind the opaque pkv_pool type.
struct pkv_pool {
    pkv_pool_desc d;
    int elem_bytes;          // bytes per stored element
    size_t layer_bytes;      // bytes of one layer of one pool tensor
    float k_inv_scale;       // binary32 1/k_scale (FP8 pools), else 1
    float v_inv_scale;
    int tmap_state;          // 0: not encoded yet, 1: ready, -1: unavailable
    int tmap_3d;             // BF16: 1 = one 3D box per block row pair, 0 = two 2D boxes
    CUtensorMap tmap_k;      // TMA descriptors of the whole K / V pool (2D: head_dim x rows)
    CUtensorMap tmap_v;
    int tmap_pair;           // 1: tmap_k2 / tmap_v2 are ready (3D boxes of two adjacent KV heads of a block)
    CUtensorMap tmap_k2;
    CUtensorMap tmap_v2;
    int tmap_half;           // 1: tmap_kh / tmap_vh are ready (3D boxes of one 64-column half of a block)
    CUtensorMap tmap_kh;
    CUtensorMap tmap_vh;
};

namespace pkv {

constexpr int kTileTokens = 64;  // tokens one decode CTA stages per pipeline step

int dtype_bytes(pkv_dtype t);
int num_sms();  // SM count of the current device (cached)
void set_last_error(cudaError_t e);
// Bytes at the front of a decode workspace that hold the per-(sequence, KV
// head) piece counters (int32 [num_seqs][num_kv_heads], rounded up to 256).
size_t workspace_counter_bytes(int num_seqs, int num_kv_heads);
// Every host-side check of paged_decode_attention with these arguments,
// without enqueuing anything: PKV_OK when the call would be launched.
pkv_status decode_attention_check(const void* q, pkv_dtype q_dtype, const pkv_pool* p, int32_t layer,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len, float scale,
                                  int32_t split_tokens, pkv_algo algo, void* workspace, size_t workspace_bytes,
                                  void* out);

// ---------------------------------------------------------------- append
cudaError_t launch_kv_append(const pkv_pool* pool, int layer, const void* k, const void* v,
                             pkv_dtype in_dtype, const int64_t* slots, int num_tokens,
                             cudaStream_t stream);

// ---------------------------------------------------------------- decode
struct DecodeArgs {
    const void* q;
    void* out;
    const uint8_t* k_layer;   // base of the layer in the K pool
    const uint8_t* v_layer;
    const int32_t* tables;
    const int32_t* lens;
    float* o_part;            // [B][num_queries][Hq][num_splits][D] fp32 (split partials)
    float* lse_part;          // [B][num_queries][Hq][num_splits] log2-domain log-sum-exp
    int32_t* counters;        // [B][Hkv] finished pieces per (sequence, KV head); zero between calls
    float* bal_o;             // balanced schedule: [CTA][2 slots][NQ][D] fp32 partials (NQ query rows per KV head)
    float* bal_lse;           // balanced schedule: [CTA][2 slots][NQ] log2-sum-exp
    int bal_max_ctas;         // > 0 selects the balanced persistent schedule (grid <= this)
    int32_t* err;             // optional error word
    int layer;
    int tma_3d;               // TMA descriptor kind (see pkv_pool::tmap_3d)
    int max_blocks;
    int max_len;              // host bound of seq_lens (<= max_blocks * block_size)
    int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks;
    // Queries: q/out hold q_total queries per sequence, the last q_total
    // positions, each attending causally.  One launch serves queries
    // [q_first, q_first + num_queries); every token it may read lies before
    // seq_len - len_trim (len_trim = q_total - q_first - num_queries).
    // Decode: q_total = num_queries = 1, q_first = len_trim = 0.
    int num_queries;
    int q_total, q_first, len_trim;
    int heads_per_cta;        // tensor-core design: 1, or 2 (adjacent KV heads share a CTA; decode, 16-token blocks)
    // Fused append (tensor-core decode): the newest token of sequence b
    // (position seq_lens[b] - 1) has rows new_k / new_v [B][Hkv][D] of dtype
    // new_dtype (PKV_BF16 or PKV_F32); the CTA whose tile holds that position
    // encodes them like kv_append, writes them to the pool and into its
    // staged tile.  new_k == nullptr: no append.
    const uint8_t* new_k;
    const uint8_t* new_v;
    int new_dtype;
    float k_inv_scale, v_inv_scale;  // FP8 pools: binary32 1/scale, as kv_append uses
    uint8_t* k_layer_w;       // writable views of k_layer / v_layer (fused append only)
    uint8_t* v_layer_w;
    int split_tokens, num_splits;
    float qk_scale_log2;      // scale * k_scale * log2(e)
    float v_scale;            // v_scale (FP8) or 1
    // Test hook (pkv_set_first_wait_limit_for_testing): with test_wait_on,
    // the consumers' first wait for a loaded stage in CTA test_wait_cta (its
    // linear block index; every CTA when < 0) gives up after test_wait_polls
    // polls, exactly as an expired wait does.  Zero-initialised: off.
    int test_wait_on;
    uint32_t test_wait_polls;
    int test_wait_cta;
};

// Returns cudaErrorNotSupported when no kernel matches (dtype, D, query rows
// per KV head).
cudaError_t launch_decode_simt(pkv_dtype kv, const DecodeArgs& a, cudaStream_t stream);
bool decode_simt_supported(pkv_dtype kv, int head_dim, int rows);
cudaError_t launch_decode_mma(pkv_dtype kv, const DecodeArgs& a, const void* tmap_k, const void* tmap_v,
                              cudaStream_t stream);
bool decode_mma_supported(pkv_dtype kv, int head_dim, int rows, int block_size);
constexpr int kMmaMaxRows = 64;   // query rows per KV head one tensor-core launch serves
constexpr int kSimtMaxRows = 16;  // the same for the SIMT design
cudaError_t launch_combine(pkv_dtype q_dtype, const DecodeArgs& a, cudaStream_t stream);
// tcgen05 multi-query attention (long query lists); one launch for all queries.
bool attention_tc_supported(pkv_dtype kv, int head_dim, int block_size);
cudaError_t launch_attention_tc(const DecodeArgs& a, const void* tmap_k, const void* tmap_v, cudaStream_t stream);

}  // namespace pkv
