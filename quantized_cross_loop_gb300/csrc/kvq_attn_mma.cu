// kvq_attn_mma.cu — tensor-core decode attention over packed K/V (placeholder
// until the MMA kernel lands: the launcher reports "not built").
#include "kvq_attn_common.cuh"

namespace kvq {
cudaError_t launch_attn_mma(const AttnArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace kvq
