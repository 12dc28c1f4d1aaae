// Tensor-core attention kernels for BF16 pools (every query-row bound, both
// schedules); the design is described in decode_mma.cuh.
#include "decode_mma.cuh"

namespace pkv {

cudaError_t launch_decode_mma_bf16(const DecodeArgs& a, const CUtensorMap& tk, const CUtensorMap& tv,
                                   cudaStream_t stream) {
    return launch_dt<PKV_BF16>(a, tk, tv, stream);
}

}  // namespace pkv
