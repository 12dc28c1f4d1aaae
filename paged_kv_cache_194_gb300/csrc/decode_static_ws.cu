// paged_decode_attention for callers that cannot allocate device memory.
//
// Some hosts of this library may not allocate device memory at the point where
// they run decode attention: plug-ins whose device memory is planned once up
// front by the host application, latency-critical loops that must never enter
// an allocator (or its failure path), and systems running under a fixed,
// pre-committed memory budget.  This entry point serves them: the split-K
// partial results live in a file-scope device array that the library owns
// for the life of the process, so a call allocates nothing.  The caller still
// provides every input and the output.
//
// The array's size is fixed (PKV_STATIC_SCRATCH_BYTES); every GPU on which the
// library is loaded holds it until the process exits.  All calls share it:
// calls that overlap on the GPU (different streams without ordering, or
// different host threads) race on it.  It keeps whatever the previous call
// left there.  The only words that must start at zero are the per-(sequence,
// KV head) piece counters at its front, and where they sit depends on the
// call's shape (a later call with more sequences or KV heads finds its
// counters in bytes an earlier call filled with partial sums; a call whose
// pipeline wait expired may leave counters non-zero).  So every call that
// uses the array first clears its own counter bytes, in stream order on the
// call's stream (one small memset; no allocation), and then launches.
#include <cstdio>

#include "pkv_internal.h"

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_STATIC_SCRATCH_BYTES];

namespace {

// Device address of g_decode_scratch per device; resolved on the first call
// made with that device current.
void* g_scratch_addr[64] = {nullptr};

}  // namespace

extern "C" pkv_status paged_decode_attention_static_ws(const void* q, pkv_dtype q_dtype, const pkv_pool* pool,
                                                       int32_t layer, const int32_t* block_tables,
                                                       int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                                       int32_t num_seqs, int32_t num_q_heads, int32_t max_seq_len,
                                                       float scale, int32_t split_tokens, pkv_algo algo, void* out,
                                                       void* stream) {
    if (!pool) return PKV_ERR_INVALID_ARG;
    size_t need = 0;
    const pkv_status st =
        paged_decode_plan(pool, num_seqs, num_q_heads, max_seq_len, split_tokens, nullptr, nullptr, &need);
    if (st != PKV_OK) return st;
    if (need > static_cast<size_t>(PKV_STATIC_SCRATCH_BYTES)) return PKV_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) {
            pkv::set_last_error(e);
            return PKV_ERR_CUDA;
        }
        if (dev < 0 || dev >= 64) return PKV_ERR_UNSUPPORTED;
        if (!g_scratch_addr[dev]) {  // once per device, with that device current
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_decode_scratch);
            if (e != cudaSuccess) {
                pkv::set_last_error(e);
                return PKV_ERR_CUDA;
            }
            g_scratch_addr[dev] = p;
        }
        scratch = g_scratch_addr[dev];
        // a rejected call enqueues nothing: check every argument before the memset
        const pkv_status chk = pkv::decode_attention_check(
            q, q_dtype, pool, layer, block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, max_seq_len,
            scale, split_tokens, algo, scratch, static_cast<size_t>(PKV_STATIC_SCRATCH_BYTES), out);
        if (chk != PKV_OK) return chk;
        // this call's counters must start at zero whatever earlier calls left
        e = cudaMemsetAsync(scratch, 0, pkv::workspace_counter_bytes(num_seqs, pool->d.num_kv_heads),
                            static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) {
            pkv::set_last_error(e);
            return PKV_ERR_CUDA;
        }
    }
    return paged_decode_attention(q, q_dtype, pool, layer, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                                  num_q_heads, max_seq_len, scale, split_tokens, algo, scratch,
                                  need > 0 ? static_cast<size_t>(PKV_STATIC_SCRATCH_BYTES) : 0, out, stream);
}
