// Tensor-core attention kernels for FP8-E4M3 pools (every query-row bound,
// both schedules); the design is described in decode_mma.cuh.
#include "decode_mma.cuh"

namespace pkv {

cudaError_t launch_decode_mma_fp8(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                  cudaStream_t stream) {
    return launch_dt<PKV_FP8_E4M3>(a, tk, tv, stream);
}

}  // namespace pkv
