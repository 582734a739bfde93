// selftest.cu -- exercises the failure-detection path of the kernels without
// a GPU fault: one thread waits, with the same bounded mbarrier wait every
// pipeline stage uses, on a barrier that nothing will ever arrive on.  When
// the (short) limit expires it records ATTN_ERR_DEVICE_TIMEOUT in the device
// status word and the kernel returns normally, so the context stays usable.
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

__global__ void __launch_bounds__(32) selftest_timeout_kernel(unsigned* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival that never comes
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, status, &abort_flag, limit_ns);
}

}  // namespace

cudaError_t launch_selftest_timeout(unsigned long long limit_ns, unsigned* status, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace attn
