/*
 * pkv.h -- C ABI of libpkv.so: paged KV cache decode attention on GB300
 * (sm_103a).
 *
 * What the operations are (page title, section):
 *   - "How does TensorRT-LLM work?", "The paged KV cache": KV memory is one
 *     pool of equal fixed-size blocks handed out on demand; a small per-request
 *     table lists the request's blocks in order; decode attends over every
 *     earlier token, whose keys and values are kept in that cache.
 *   - "Introduction to TensorRT-LLM", "2. Paged KV Cache": fixed-size token
 *     blocks, virtual-to-physical block tables; section "4. Optimized
 *     Attention Kernels" names FlashAttention and Flash-Decoding (fused
 *     kernels, split over the key/value length).
 *   - "TensorRT-LLM, in depth", "First principles": kv_bytes_per_token =
 *     2 * layers * kv_heads * head_dim * bytes_per_elem; grouped-query
 *     attention (Llama-3-8B: 32 query heads share 8 KV heads).
 *   - "TensorRT-LLM, in depth", "Quantization": an FP8 KV cache halves the
 *     cache bytes.
 *
 * Conventions for every entry point:
 *   - Device buffers are plain device pointers owned by the caller (e.g. torch
 *     tensors).  The library never allocates or frees device memory and never
 *     synchronises the stream; work is enqueued on `stream` (a cudaStream_t,
 *     NULL = legacy default stream).
 *   - Every dense tensor is C-contiguous.  q, out, k, v, the pool bases and the
 *     workspace must be 16-byte aligned; int32/int64 arrays naturally aligned.
 *   - Host-checkable faults return an error before anything is enqueued.
 *     Index faults that only the device can see (a block id outside the pool,
 *     a slot outside the pool, a length beyond the block table) never touch
 *     memory out of bounds: the offending access is skipped and, when the pool
 *     has an error word, a bit is OR-ed into it (PKV_ERRBIT_*).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or index */
    PKV_ERR_UNSUPPORTED = 2,   /* geometry or dtype this build has no kernel for */
    PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    PKV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    PKV_ERR_DEVICE_BOUNDS = 5, /* reserved for callers decoding the error word */
    PKV_ERR_OUT_OF_BLOCKS = 6, /* block manager: the free list cannot cover the request */
    PKV_ERR_INCONSISTENT = 7   /* block manager: an internal invariant does not hold */
} pkv_status;

/* Element types.  PKV_FP8_E4M3 is OCP E4M3 (bias 7, max 448, no infinities). */
typedef enum pkv_dtype { PKV_F32 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

/* Bits OR-ed into the pool's error word by the kernels. */
#define PKV_ERRBIT_BLOCK_ID 1 /* block table entry outside [0, num_blocks) */
#define PKV_ERRBIT_SLOT 2     /* slot_mapping entry outside [-1, num_blocks*block_size) */
#define PKV_ERRBIT_SEQ_LEN 4  /* seq_lens entry < 0 or > max_seq_len of the call */
#define PKV_ERRBIT_TIMEOUT 8  /* a bounded pipeline wait expired; that CTA skipped its output */

/* Kernel design used by paged_decode_attention. */
typedef enum pkv_algo {
    PKV_ALGO_AUTO = 0, /* best available for the pool's dtype and geometry */
    PKV_ALGO_SIMT = 1, /* CUDA-core dot products (every dtype) */
    PKV_ALGO_MMA = 2,  /* tensor-core QK^T and PV with warp-level mma (BF16 / FP8 pools) */
    PKV_ALGO_TC = 3    /* multi-query only: tcgen05 MMAs with TMEM accumulators, 128 query
                          rows per CTA (BF16 pools, head_dim 128, fixed splits not used);
                          AUTO picks it from 8 query rows per KV head (2 or more queries) */
} pkv_algo;

/*
 * Pool geometry.  The K pool and the V pool are each one device tensor laid
 * out [num_layers][num_blocks][num_kv_heads][block_size][head_dim] in
 * kv_dtype, so that one (block, kv head) is a contiguous run of
 * block_size*head_dim elements.  A slot is block_id*block_size + offset.
 * k_scale / v_scale are the per-tensor dequantisation scales of an FP8 pool
 * (value = e4m3 * scale; appends store e4m3(x * (1/scale)), with 1/scale
 * rounded once to binary32); they are ignored for other dtypes.
 * error_word: optional device int32 the kernels OR PKV_ERRBIT_* into; may be
 * NULL.  Supported: block_size in {16, 32, 64}, head_dim in {64, 128}.
 */
typedef struct pkv_pool_desc {
    int32_t num_layers;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    pkv_dtype kv_dtype;
    float k_scale;
    float v_scale;
    void* k_base;        /* device */
    void* v_base;        /* device */
    int32_t* error_word; /* device, optional */
} pkv_pool_desc;

/* Opaque host handle: a validated copy of the descriptor.  It owns no device
 * memory; destroying it leaves the caller's tensors untouched. */
typedef struct pkv_pool pkv_pool;

/* Validate `desc` and create a handle.  INVALID_ARG / UNSUPPORTED on a bad
 * descriptor ("TensorRT-LLM, in depth", "The paged KV cache and block reuse":
 * the KV cache manager splits reserved memory into fixed-size blocks). */
pkv_status kv_pool_create(const pkv_pool_desc* desc, pkv_pool** out);
void kv_pool_destroy(pkv_pool* pool);

/* Bytes of one pool tensor (K or V) for the descriptor's geometry. */
size_t kv_pool_tensor_bytes(const pkv_pool_desc* desc);

/* "TensorRT-LLM, in depth", "First principles": bytes of K and V that one
 * token occupies across all layers: 2 * layers * kv_heads * head_dim * size. */
int64_t kv_bytes_per_token(int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                           pkv_dtype dtype);

/*
 * KV append ("How does TensorRT-LLM work?", "The paged KV cache": every new
 * token adds one more set of keys/values, written into the request's blocks).
 *   k, v          device [num_tokens][num_kv_heads][head_dim] in in_dtype
 *                 (PKV_F32 or PKV_BF16; an F32 pool takes F32 only).
 *   slot_mapping  device int64 [num_tokens]; token t goes to slot
 *                 slot_mapping[t] of layer `layer`; -1 skips the token.
 * Conversion: same dtype copies bits; F32->BF16 rounds to nearest even;
 * ->FP8 stores e4m3_rn_satfinite(fp32(x) * fp32(1/scale)).  Two tokens that
 * name the same slot race (undefined which one lands).
 */
pkv_status kv_append(const pkv_pool* pool, int32_t layer, const void* k, const void* v,
                     pkv_dtype in_dtype, const int64_t* slot_mapping, int32_t num_tokens,
                     void* stream);

/*
 * Split planning for paged_decode_attention.  Flash-decoding splits each
 * sequence's tokens into chunks, attends to each chunk in its own CTA and
 * merges the partial results by their log-sum-exp.  Outputs (any may be
 * NULL): the fixed split size a fixed-split call uses (split_tokens, or the
 * automatic choice from the batch shape and the SM count when it is 0), the
 * number of such splits of the longest sequence, and the workspace bytes the
 * call needs whichever schedule it runs (0 only for a fixed-split call whose
 * single split covers max_seq_len).  split_tokens, when given, must be a
 * positive multiple of 64 and of block_size.
 */
pkv_status paged_decode_plan(const pkv_pool* pool, int32_t num_seqs, int32_t num_q_heads,
                             int32_t max_seq_len, int32_t split_tokens, int32_t* split_tokens_out,
                             int32_t* num_splits_out, size_t* workspace_bytes_out);

/*
 * Paged decode attention ("How does TensorRT-LLM work?", "Custom attention
 * kernels" and "The paged KV cache"): for every sequence b and query head hq,
 *     out[b][hq][:] = softmax_t(scale * q[b][hq] . K_t) V_t,
 *     t = 0 .. seq_lens[b]-1,
 * where K_t / V_t are row t % block_size of block block_tables[b][t /
 * block_size] of the pool's layer `layer`, KV head hq / (num_q_heads /
 * num_kv_heads) (grouped-query attention), times k_scale / v_scale for FP8.
 *   q             device [num_seqs][num_q_heads][head_dim], q_dtype = F32 for
 *                 an F32 pool, BF16 otherwise.
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]; only the first
 *                 ceil(seq_lens[b]/block_size) entries of row b are read.
 *   seq_lens      device int32 [num_seqs].  A length of 0 gives a zero row.
 *   max_seq_len   host upper bound of seq_lens (sizes the grid); must be
 *                 <= max_blocks_per_seq * block_size.  Longer device lengths
 *                 are clamped to it and flagged PKV_ERRBIT_SEQ_LEN.
 *   workspace     device scratch of at least the planned bytes (may be NULL
 *                 when the plan needs none).  Its first 4*num_seqs*num_kv_heads
 *                 bytes (rounded up to 256) are per-(sequence, KV head)
 *                 counters that must be zero before the first call; every
 *                 call leaves them zero again (a call that reports
 *                 PKV_ERRBIT_TIMEOUT may not: clear them then).  The rest is
 *                 overwritten.  Calls that share a workspace must be
 *                 stream-ordered.
 *   out           device [num_seqs][num_q_heads][head_dim] in q_dtype.
 *   split_tokens  0: the tensor-core design balances the batch itself (a
 *                 persistent grid of 2 CTAs per SM, each streaming an equal
 *                 share of the (sequence, KV head, 64-token tile) list, with
 *                 an in-kernel log-sum-exp merge of shared sequences); the
 *                 SIMT design picks a split size.  > 0: fixed splits of that
 *                 many tokens and a separate combine kernel.
 *   algo          PKV_ALGO_AUTO, or a specific kernel design.
 * Softmax and accumulation are fp32; the output is rounded to q_dtype (RN).
 */
pkv_status paged_decode_attention(const void* q, pkv_dtype q_dtype, const pkv_pool* pool,
                                  int32_t layer, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                                  float scale, int32_t split_tokens, pkv_algo algo,
                                  void* workspace, size_t workspace_bytes, void* out,
                                  void* stream);

/*
 * Multi-query paged attention: the last num_queries (C) tokens of every
 * sequence ask a query each, attending causally -- query c, at position
 * seq_lens[b] - C + c, sees tokens 0 .. seq_lens[b] - C + c.  This is how a
 * decode step verifies C drafted tokens ("How does TensorRT-LLM work?",
 * "Speculative decoding": the real model checks several guessed tokens in one
 * pass) and how a chunk of a prompt attends to the cache ("How does
 * TensorRT-LLM work?", "In-flight batching": chunked prefill).
 *   q    device [num_seqs][C][num_q_heads][head_dim];
 *   out  device [num_seqs][C][num_q_heads][head_dim];
 * other arguments as paged_decode_attention (which is the C = 1 case);
 * 1 <= C <= 2^20.  The tcgen05 design (PKV_ALGO_TC) serves every query in
 * one launch.  Normally that is one CTA per 128 query rows of a (sequence,
 * KV head), the longest sequences' CTAs first.  With at most 128 query rows
 * per KV head and fewer (sequence, KV head) pairs than CTA slots (a few long
 * sequences) it uses the balanced schedule instead: persistent CTAs share out
 * the 64-token tiles of all pairs equally and merge the pairs they split,
 * which needs the workspace.  With the other designs
 * one launch serves a chunk of consecutive queries: up to 64 query rows per KV
 * head (chunk x num_q_heads / num_kv_heads) for the warp-level tensor-core
 * design, a power of two up to 16 (fewer for FP8 and BF16 pools with large
 * groups) for the SIMT design; longer query lists run as several launches on
 * the stream, each reading only the tokens its last query sees.
 * Workspace (from paged_multi_query_plan) is shared by those launches in
 * stream order.  A query whose position is negative (seq_lens[b] < C) gets a
 * zero row.
 */
pkv_status paged_multi_query_plan(const pkv_pool* pool, int32_t num_seqs, int32_t num_queries,
                                  int32_t num_q_heads, int32_t max_seq_len, int32_t split_tokens,
                                  int32_t* split_tokens_out, int32_t* num_splits_out,
                                  size_t* workspace_bytes_out);
/* The kernel design paged_multi_query_attention would run for this request:
 * PKV_ALGO_TC, PKV_ALGO_MMA or PKV_ALGO_SIMT, or -1 when it cannot be served. */
int32_t paged_multi_query_algo(const pkv_pool* pool, int32_t num_queries, int32_t num_q_heads,
                               int32_t split_tokens, pkv_algo requested);
pkv_status paged_multi_query_attention(const void* q, pkv_dtype q_dtype, const pkv_pool* pool,
                                       int32_t layer, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                       int32_t num_seqs, int32_t num_queries, int32_t num_q_heads,
                                       int32_t max_seq_len, float scale, int32_t split_tokens,
                                       pkv_algo algo, void* workspace, size_t workspace_bytes,
                                       void* out, void* stream);

/*
 * One decode step of one layer in a single launch: append each sequence's
 * newest token, then attend ("How does TensorRT-LLM work?", "In-flight
 * batching": every decode step adds one token's keys and values to the cache
 * and attends over all of them).  Same result, bit for bit, as kv_append of
 * k_new / v_new at the slot of position seq_lens[b] - 1 (taken from the block
 * table) followed by paged_decode_attention.
 *   k_new, v_new  device [num_seqs][num_kv_heads][head_dim] of in_dtype
 *                 (PKV_BF16 or PKV_F32), 16-byte aligned; row b is written
 *                 at position seq_lens[b] - 1 (nothing for seq_lens[b] = 0).
 * other arguments as paged_decode_attention (workspace from
 * paged_decode_plan).  Served by the tensor-core design only (BF16/FP8 pools,
 * head_dim 128, block size 16/32/64, at most 8 query heads per KV head);
 * otherwise PKV_ERR_UNSUPPORTED before anything is enqueued.  A table entry
 * outside the pool at the newest position skips the pool write and sets
 * PKV_ERRBIT_BLOCK_ID; a length above max_seq_len skips it and sets
 * PKV_ERRBIT_SEQ_LEN.
 */
pkv_status paged_decode_append_attention(const void* q, pkv_dtype q_dtype, const void* k_new,
                                         const void* v_new, pkv_dtype in_dtype, const pkv_pool* pool,
                                         int32_t layer, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                         int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                                         float scale, int32_t split_tokens, pkv_algo algo,
                                         void* workspace, size_t workspace_bytes, void* out,
                                         void* stream);

/*
 * paged_decode_attention without a caller-provided workspace, for callers that
 * may not allocate device memory where they run decode attention (plug-ins
 * whose device memory the host application plans once up front, loops that
 * must never enter an allocator, fixed memory budgets).  The pages have no
 * counterpart to this entry point; it is an interface convenience.
 *
 * Same arguments and results as paged_decode_attention, minus the workspace:
 * the split-K partials go to a fixed device array owned by the library
 * (PKV_STATIC_SCRATCH_BYTES; every GPU that loads the library holds it until
 * the process exits).  Allocates nothing.  The first call that needs scratch
 * on a device looks up the array's device address with that device current;
 * make that first call before any stream capture.  A call whose plan needs
 * more than PKV_STATIC_SCRATCH_BYTES (see paged_decode_plan) returns
 * PKV_ERR_WORKSPACE, and a call any other check rejects returns its status,
 * before enqueuing anything.  All calls share the one array, which keeps what
 * the previous call left: calls that overlap on the GPU race and must be
 * ordered by the caller.  Each call that uses the array first clears its own
 * per-(sequence, KV head) counters there, in stream order (a memset on
 * `stream` of 4 * num_seqs * num_kv_heads bytes rounded up to 256), so calls
 * of different shapes, and a call after one that reported
 * PKV_ERRBIT_TIMEOUT, need no clearing by the caller.
 */
#define PKV_STATIC_SCRATCH_BYTES (16 * 1024 * 1024)
pkv_status paged_decode_attention_static_ws(const void* q, pkv_dtype q_dtype, const pkv_pool* pool,
                                            int32_t layer, const int32_t* block_tables,
                                            int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                            int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                                            float scale, int32_t split_tokens, pkv_algo algo, void* out,
                                            void* stream);

/* The kernel design paged_decode_attention would run for this pool, group
 * size (num_q_heads / num_kv_heads; for multi-query attention, times
 * the queries of one launch) and request: PKV_ALGO_SIMT or PKV_ALGO_MMA, or
 * -1 when the request cannot be served.  PKV_ALGO_AUTO picks MMA for BF16/FP8
 * pools with head_dim 128, block size 16/32/64 and 1 <= group <= 64 (when the
 * driver provides TMA descriptors), SIMT otherwise. */
int32_t paged_decode_algo(const pkv_pool* pool, int32_t group, pkv_algo requested);

/*
 * Host-side block manager ("How does TensorRT-LLM work?", "The paged KV
 * cache": a pool of equal blocks handed out one at a time, a per-request
 * table of its blocks in order, blocks returned the moment a request
 * finishes, and requests that begin with the same text pointing at the same
 * blocks; "TensorRT-LLM, in depth", "In-flight batching and the scheduler":
 * a request that cannot get a block for its next token is paused; "The paged
 * KV cache and block reuse": reuse only for identical token prefixes).
 *
 * Host memory only; no CUDA call.  Blocks are reference counted: a block is
 * free when no sequence's table holds it.  Freed blocks go to the tail of an
 * LRU free list and stay matchable by content until they are reallocated.
 * A full block written by tokens with ids is identified by a 64-bit hash of
 * the whole id prefix up to it; only such blocks are shared, so a shared block
 * is never written again.  Slots are block * block_size + offset.  Not
 * thread-safe: one manager per scheduler thread.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* free_order: a permutation of 0..num_blocks-1 (NULL = ascending) giving the
 * order in which free blocks are handed out. */
pkv_status kv_block_manager_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                                   const int32_t* free_order, pkv_block_manager** out);
void kv_block_manager_destroy(pkv_block_manager* bm);
int32_t kv_bm_num_free(const pkv_block_manager* bm);
pkv_status kv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id);
/* Drop a finished sequence: each of its blocks loses one reference. */
pkv_status kv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id);
/* Reserve the next n_tokens positions of a sequence and write their slots
 * (slots_out may be NULL).  token_ids (may be NULL) identify the tokens for
 * prefix reuse.  PKV_ERR_OUT_OF_BLOCKS, with nothing changed, when the free
 * list or max_blocks_per_seq cannot cover them. */
pkv_status kv_bm_grow(pkv_block_manager* bm, int64_t seq_id, int32_t n_tokens, const int32_t* token_ids,
                      int64_t* slots_out);
/* One decode step: the slot of each listed sequence's next token; a sequence
 * that cannot get a block keeps its length and gets slot -1 (paused); the
 * number of paused sequences goes to *n_paused. */
pkv_status kv_bm_decode_slots(pkv_block_manager* bm, const int64_t* seq_ids, int32_t n, int64_t* slots_out,
                              int32_t* n_paused);
/* For an empty sequence about to hold a prompt of n_tokens ids: share every
 * cached full block of the longest matching prefix (at most (n_tokens-1) /
 * block_size blocks, so the last prompt token is always appended).  The
 * sequence's length becomes the reused token count. */
pkv_status kv_bm_match_prefix(pkv_block_manager* bm, int64_t seq_id, const int32_t* token_ids, int32_t n_tokens,
                              int32_t* reused_tokens_out);
int32_t kv_bm_seq_len(const pkv_block_manager* bm, int64_t seq_id);
/* Host tables [n][width] (padded with -1) and lengths of the listed sequences. */
pkv_status kv_bm_block_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int32_t n, int32_t width,
                              int32_t* tables_out, int32_t* lens_out);
/* Free list in hand-out order (up to cap entries); returns its length. */
int32_t kv_bm_free_list(const pkv_block_manager* bm, int32_t* out, int32_t cap);
int32_t kv_bm_block_ref(const pkv_block_manager* bm, int32_t block);
/* Verify every invariant; PKV_ERR_INCONSISTENT if one fails. */
pkv_status kv_bm_check(const pkv_block_manager* bm);

/*
 * Test hook for the failure path of the bounded pipeline waits.  The pages
 * name no interface for it; "TensorRT-LLM, in depth", section "In-flight
 * batching and the scheduler", has a request that cannot go on paused rather
 * than failed, and its "Failure modes" heading lists failure handling.  Every
 * wait of the tensor-core decode design (PKV_ALGO_MMA: decode, fused decode,
 * multi-query) is bounded; an expired one sets PKV_ERRBIT_TIMEOUT, stops the
 * CTA's pipeline, waits with the full bound for the copies the CTA has in
 * flight, skips the CTA's output and returns.  This makes such an expiry
 * happen on demand, without a fault or a hang:
 *   polls >= 0  later launches of that design made from the calling host
 *               thread give up the consumer warps' first wait for a loaded
 *               stage after `polls` polls (0: without looking), in the CTA
 *               whose linear block index is `cta` (every CTA when cta < 0);
 *   polls < 0   normal bounds again (the default).
 * Only that first wait is shortened; the waits that guard copies in flight
 * keep their bound.  After a call that reported PKV_ERRBIT_TIMEOUT, the
 * workspace's counters may be non-zero (clear them before reusing it), and
 * the output rows of the units the stopped CTAs took part in are unwritten.
 */
void pkv_set_first_wait_limit_for_testing(int32_t polls, int32_t cta);

/* Human-readable name of a status. */
const char* pkv_status_string(pkv_status status);

/* Message of the last CUDA error seen by this thread's calls ("" if none). */
const char* pkv_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
