// tcgen05 tensor-core split-KV tree-verify attention (placeholder until the
// kernel lands: no descriptor selects it).
#include "tv_internal.cuh"

namespace tv {

bool tc_supported(int, int, int, int) { return false; }
int tc_key_tile(int) { return 64; }
cudaError_t launch_attn_tc(const AttnParams&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace tv
