// KV append: scatter each new token's K and V rows into the pool slots named
// by the slot mapping ("How does TensorRT-LLM work?", "The paged KV cache":
// every new token adds one more set of keys/values to the request's blocks).
//
// One thread writes one 16-byte chunk of one pool row; a (token, head) row of
// head_dim elements is a contiguous run in both the input and the pool, so
// consecutive threads read and write consecutive 16-byte chunks.
#include "device_common.cuh"

namespace pkv {
namespace {

constexpr int kAppendThreads = 256;

template <int PDT, int IDT>
__global__ void __launch_bounds__(kAppendThreads)
kv_append_kernel(const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
                 const int64_t* __restrict__ slots, int num_tokens, int kv_heads, int head_dim,
                 int block_size, int64_t num_slots, uint8_t* __restrict__ k_layer,
                 uint8_t* __restrict__ v_layer, float k_inv, float v_inv, int32_t* err) {
    // let a dependent decode launch start its set-up now; it waits for this
    // grid to finish before it reads anything
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    constexpr int kPoolBytes = PDT == PKV_F32 ? 4 : (PDT == PKV_BF16 ? 2 : 1);
    constexpr int kInBytes = IDT == PKV_F32 ? 4 : 2;
    constexpr int kPer = 16 / kPoolBytes;  // elements per output chunk
    const int chunks_per_row = head_dim / kPer;
    const int64_t rows = static_cast<int64_t>(num_tokens) * kv_heads;
    const int64_t total = rows * chunks_per_row * 2;  // K rows then V rows
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const bool is_v = i >= rows * chunks_per_row;
        const int64_t j = is_v ? i - rows * chunks_per_row : i;
        const int c = static_cast<int>(j % chunks_per_row);
        const int64_t row = j / chunks_per_row;  // token * kv_heads + head
        const int t = static_cast<int>(row / kv_heads);
        const int h = static_cast<int>(row % kv_heads);
        const int64_t slot = slots[t];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_slots) {
            if (err && c == 0 && h == 0 && !is_v) atomicOr(err, PKV_ERRBIT_SLOT);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int64_t off = slot % block_size;
        const uint8_t* src = (is_v ? v : k) + (row * head_dim + static_cast<int64_t>(c) * kPer) * kInBytes;
        uint8_t* dst = (is_v ? v_layer : k_layer) +
                       (((blk * kv_heads + h) * block_size + off) * head_dim + static_cast<int64_t>(c) * kPer) *
                           kPoolBytes;
        *reinterpret_cast<uint4*>(dst) = append_chunk<PDT, IDT>(src, is_v ? v_inv : k_inv);
    }
}

template <int PDT, int IDT>
cudaError_t launch(const pkv_pool* p, int layer, const void* k, const void* v, const int64_t* slots, int T,
                   cudaStream_t stream) {
    const pkv_pool_desc& d = p->d;
    const int per = 16 / p->elem_bytes;
    const int64_t total = static_cast<int64_t>(T) * d.num_kv_heads * (d.head_dim / per) * 2;
    const int64_t want = (total + kAppendThreads - 1) / kAppendThreads;
    const int blocks = static_cast<int>(want < 65535 * 16 ? want : 65535 * 16);
    uint8_t* kl = static_cast<uint8_t*>(d.k_base) + static_cast<size_t>(layer) * p->layer_bytes;
    uint8_t* vl = static_cast<uint8_t*>(d.v_base) + static_cast<size_t>(layer) * p->layer_bytes;
    kv_append_kernel<PDT, IDT><<<blocks, kAppendThreads, 0, stream>>>(
        static_cast<const uint8_t*>(k), static_cast<const uint8_t*>(v), slots, T, d.num_kv_heads,
        d.head_dim, d.block_size, static_cast<int64_t>(d.num_blocks) * d.block_size, kl, vl,
        p->k_inv_scale, p->v_inv_scale, d.error_word);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kv_append(const pkv_pool* p, int layer, const void* k, const void* v, pkv_dtype in,
                             const int64_t* slots, int T, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    switch (p->d.kv_dtype) {
        case PKV_F32:
            if (in == PKV_F32) return launch<PKV_F32, PKV_F32>(p, layer, k, v, slots, T, stream);
            break;
        case PKV_BF16:
            if (in == PKV_BF16) return launch<PKV_BF16, PKV_BF16>(p, layer, k, v, slots, T, stream);
            if (in == PKV_F32) return launch<PKV_BF16, PKV_F32>(p, layer, k, v, slots, T, stream);
            break;
        case PKV_FP8_E4M3:
            if (in == PKV_BF16) return launch<PKV_FP8_E4M3, PKV_BF16>(p, layer, k, v, slots, T, stream);
            if (in == PKV_F32) return launch<PKV_FP8_E4M3, PKV_F32>(p, layer, k, v, slots, T, stream);
            break;
    }
    return cudaErrorNotSupported;
}

}  // namespace pkv
