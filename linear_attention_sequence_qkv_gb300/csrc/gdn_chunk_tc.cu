// gdn_chunk_tc.cu -- chunked gated delta rule on the tcgen05 tensor cores
// (bf16/fp16 activations). Not yet routed: every dtype uses the CUDA-core kernel.
#include "gdn_common.cuh"

namespace gdn {

bool chunk_tc_supports(const gdn_desc &) { return false; }

cudaError_t launch_chunk_tc(const Problem &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
