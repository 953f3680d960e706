// Diagnostic for the failure path: one kernel whose bounded wait can never be
// satisfied.  It runs the same wait helpers as the layer's kernels (an
// mbarrier phase that nobody completes, or a device counter that nobody
// raises), so each wait gives up after kWaitLimitNs, records kErrTimeout in
// the device error word and returns; nothing faults and nothing hangs.  The
// host then reads TERN_ETIMEOUT from tern_device_status and the context stays
// usable.
#include "tern_device.cuh"
#include "tern_internal.h"

namespace tern {
namespace {

// Stays zero: no code writes it.
__device__ unsigned long long g_never_raised = 0;

__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(int which, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;  // one waiting thread
  if (which == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    (void)mbar_wait(&bar, 0, err);  // phase 0 needs one arrival; none comes
  } else {
    (void)wait_counter_at_least(&g_never_raised, 1ull, err);
  }
}

}  // namespace

cudaError_t launch_wait_timeout_probe(int which, int* err, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(which, err);
  return cudaGetLastError();
}

}  // namespace tern
