// K2: backward ring step (placeholder until the tcgen05 kernel lands).
#include "kernels.h"

namespace cpa {

size_t step_bwd_smem_bytes(int) { return 0; }

cp_attn_status launch_step_bwd(int, dim3, size_t, cudaStream_t, const CUtensorMap&,
                               const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                               const BwdParams&) {
  return fail(CP_ATTN_ERR_UNSUPPORTED, "step_bwd: backward kernel not built yet");
}

}  // namespace cpa
