// fa_bwd.cu -- backward pass (placeholder until the kernels land).
#include "fa_internal.h"

namespace fa {
int launch_bwd(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
               const BwdParams&, int, cudaStream_t) {
  return FA_ERR_LAUNCH;
}
}  // namespace fa
