// fused_tc.cu -- single-kernel GDN / linear-attention prefill on tcgen05 (placeholder).
#include "common.cuh"
#include "launch.h"

namespace gdn {

bool fused_supported(const PrefillArgs&) { return false; }
cudaError_t launch_fused(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
