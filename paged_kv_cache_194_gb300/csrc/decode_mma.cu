// Paged decode attention, tensor-core design (not built yet: every
// configuration reports "unsupported" and the SIMT design serves it).
#include "pkv_internal.h"

namespace pkv {

bool decode_mma_supported(pkv_dtype, int, int, int) { return false; }

cudaError_t launch_decode_mma(pkv_dtype, const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace pkv
