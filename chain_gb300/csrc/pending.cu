// pending.cu -- entry points whose kernels are not built yet report
// "unsupported" instead of falling back to anything else.
#include "internal.h"

namespace chain {
cudaError_t launch_attn_fwd_f32(const AttnFwdArgs &, const WaitCfg &, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace chain
