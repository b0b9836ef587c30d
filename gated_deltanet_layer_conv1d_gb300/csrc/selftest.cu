// selftest.cu -- a check of the bounded device-side wait that every kernel of the library
// uses (sm_103a).
//
// One thread initialises an mbarrier that nothing ever arrives on and waits for its first
// phase with mbar_wait_bounded under the caller's budget.  The wait must give up, report
// GDN_ERR_TIMEOUT to the status word and return, leaving the context usable: the same path
// a kernel takes when a copy or a peer it waits for never comes.  Nothing faults, traps or
// spins without a limit.
#include "common.cuh"
#include "kernels.h"

namespace gdn {
namespace {

__global__ void gdn_wait_selftest_kernel(uint64_t budget_ns, int32_t* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!mbar_wait_bounded(&bar, 0, budget_ns)) report(status, GDN_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t budget_ns, int32_t* status, cudaStream_t stream) {
  gdn_wait_selftest_kernel<<<1, 32, 0, stream>>>(budget_ns, status);
  return cudaGetLastError();
}

}  // namespace gdn
