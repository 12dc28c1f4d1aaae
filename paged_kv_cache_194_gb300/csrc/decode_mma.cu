// Dispatch of the tensor-core attention design (kernels in decode_mma.cuh,
// instantiated per KV dtype in decode_mma_bf16.cu and decode_mma_fp8.cu).
#include "decode_mma.cuh"

namespace pkv {

bool decode_mma_supported(pkv_dtype kv, int head_dim, int rows, int block_size) {
    if (kv != PKV_BF16 && kv != PKV_FP8_E4M3) return false;
    if (head_dim != kD) return false;
    if (rows < 1 || rows > kMmaMaxRows) return false;
    return block_size == 16 || block_size == 32 || block_size == 64;
}

cudaError_t launch_decode_mma(pkv_dtype kv, const DecodeArgs& a, const void* tmap_k, const void* tmap_v,
                              cudaStream_t stream) {
    const CUtensorMap& tk = *static_cast<const CUtensorMap*>(tmap_k);
    const CUtensorMap& tv = *static_cast<const CUtensorMap*>(tmap_v);
    if (kv == PKV_BF16) return launch_decode_mma_bf16(a, tk, tv, stream);
    if (kv == PKV_FP8_E4M3) return launch_decode_mma_fp8(a, tk, tv, stream);
    return cudaErrorNotSupported;
}

}  // namespace pkv
