// Chunked gated delta rule on tcgen05 tensor cores (bf16 operands, f32 state).
#include "gdn_common.cuh"
#include "gdn_launch.h"

namespace gdn {

bool chunk_tc_supported(const DeltaArgs& a, gdn_dtype_t dt) {
    (void)a; (void)dt;
    return false;
}

cudaError_t launch_chunk_tc(const DeltaArgs& a, cudaStream_t s) {
    (void)a; (void)s;
    return cudaErrorNotSupported;
}

}  // namespace gdn
