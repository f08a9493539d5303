// Launchers not yet implemented report MSA_ERR_UNSUPPORTED.
#include "msa_internal.h"
namespace msa {
msa_status launch_attn_bwd(const msa_plan_s*, const void*, const void*, const void*, const int32_t*, const int32_t*,
                           const void*, const float*, const void*, const void*, const void*, float, float*, float*,
                           float*, float*, float*, cudaStream_t) {
  return set_error(MSA_ERR_UNSUPPORTED, "bwd not built");
}
}  // namespace msa
