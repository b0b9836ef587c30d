// prefill.cu -- dispatch of the GDN prefill (sm_103a).
#include "common.cuh"
#include "kernels.h"

namespace gdn {

cudaError_t launch_prefill_sequential(const PrefillParams& p, int dtype, cudaStream_t stream);

size_t prefill_workspace_bytes(int Hk, int Hv, int D, int n, int total_tokens, int max_seqlen) {
  (void)Hk; (void)Hv; (void)D; (void)n; (void)total_tokens; (void)max_seqlen;
  return 0;
}

cudaError_t launch_prefill(const PrefillParams& p, int dtype, cudaStream_t stream) {
  return launch_prefill_sequential(p, dtype, stream);
}

}  // namespace gdn
