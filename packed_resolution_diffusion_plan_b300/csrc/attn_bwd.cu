// Varlen joint attention backward with fused 2D RoPE (placeholder).
#include "attn_common.cuh"

namespace mf {

cudaError_t launch_attn_bwd(const BwdArgs&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                            const CUtensorMap&, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mf
