// selftest.cu -- one bounded mbarrier wait of the kind every pipelined kernel
// here uses, so that the give-up path can be exercised without a real hang.
//
// With expire set, nothing ever arrives on the barrier: the wait gives up
// after limit_ns, the kernel records DSA_STATUS_TIMEOUT in the status word and
// returns, and the context stays usable.  Without it the barrier is completed
// before the wait, which must then succeed and record nothing.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "dsa_internal.cuh"
#include "sm100.cuh"

namespace dsa {

namespace {

using namespace sm100;

__global__ void k_bounded_wait(int* status, int expire, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (!expire) mbar_arrive(&bar);
  if (!mbar_wait(&bar, 0, &abort_flag, limit_ns)) flag_status(status, DSA_STATUS_TIMEOUT);
}

}  // namespace

int bounded_wait_selftest(int expire, unsigned long long limit_ns, int* status, cudaStream_t s) {
  k_bounded_wait<<<1, 32, 0, s>>>(status, expire, limit_ns);
  count_launch();
  return check_launch("bounded wait self-test");
}

}  // namespace dsa
