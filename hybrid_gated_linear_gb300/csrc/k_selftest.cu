// k_selftest.cu -- a self-test of the device-side failure detection.
//
// Every tile kernel of this library waits on mbarriers with wait_bar (tc_pipe.cuh), which
// gives up after a clock limit, raises the CTA's abort flag (so the CTA's other roles stop
// waiting too), and the CTA records LIZARD_ERR_TIMEOUT in the workspace's status word.
// No input of the operator can make a wait run out, so this entry point does it on
// purpose and safely: one CTA arms a barrier with an expected byte count and issues no
// copy and no MMA, so nothing is in flight that could fault or would need draining; one
// role waits with the given short limit, a second with the normal limit and leaves when
// the first aborts.
#include "lizard_dev.cuh"
#include "lizard_internal.h"
#include "tc_pipe.cuh"

namespace lz {
namespace {

using namespace tc;

__global__ void __launch_bounds__(64) wait_timeout_kernel(unsigned* status, long long limit) {
  __shared__ __align__(8) Ctl<1> ctl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&ctl.bar[0], 1u);
    ctl.abort = 0;
    fence_mbar_init();
  }
  cta_sync();
  if (warp == 0 && lane == 0) {
    // the one arrival the phase needs, plus 16 bytes that no copy will ever deliver
    mbar_arrive_expect_tx(&ctl.bar[0], 16u);
    if (!wait_bar(&ctl, 0, 0, limit)) ctl.abort = 1;
  } else if (warp == 1 && lane == 0) {
    if (!wait_bar(&ctl, 0, 0)) ctl.abort = 1;  // returns once warp 0 has given up
  }
  cta_sync();
  if (threadIdx.x == 0 && ctl.abort) raise_status(status, kDevTimeout);
}

}  // namespace
}  // namespace lz

extern "C" lizard_status lizard_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                                      int64_t wait_cycles, void* stream) {
  lz::set_last_launches(0);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 15u) != 0 ||
      workspace_bytes < lz::kWsHeader)
    return LIZARD_ERR_WORKSPACE;
  if (wait_cycles < 1 || wait_cycles > lz::tc::kWaitCycles) return LIZARD_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync(workspace, 0, lz::kWsHeader, s) != cudaSuccess) return LIZARD_ERR_CUDA;
  lz::wait_timeout_kernel<<<1, 64, 0, s>>>(static_cast<unsigned*>(workspace),
                                           (long long)wait_cycles);
  lz::set_last_launches(1);
  return cudaGetLastError() == cudaSuccess ? LIZARD_OK : LIZARD_ERR_CUDA;
}
