// chunk_tc.cu -- tensor-core chunked forward (placeholder until the tcgen05
// kernel lands): reports no supported shapes so that every call takes the
// generic kernel.
#include "kernels.h"

namespace delta {

bool chunk_tc_supports(const FwdArgs &) { return false; }

cudaError_t launch_chunk_tc(const FwdArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace delta
