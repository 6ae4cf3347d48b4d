// diag.cu -- check of the bounded mbarrier wait that every pipeline of the
// library uses (common.cuh: mbar_wait).
#include "launch.h"

namespace msa {

// One thread waits on two mbarriers that nothing arrives on; each wait runs
// to the wait limit, and the first records the timeout.
__global__ void wait_check_kernel(DevError* err, long long* waits_ns) {
  __shared__ uint64_t bars[2];
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_ns();
    const bool a = mbar_wait(&bars[0], 0, err, 900);
    const uint64_t t1 = global_ns();
    const bool b = mbar_wait(&bars[1], 0, err, 901);
    const uint64_t t2 = global_ns();
    waits_ns[0] = a ? -1 : static_cast<long long>(t1 - t0);
    waits_ns[1] = b ? -1 : static_cast<long long>(t2 - t1);
  }
}

cudaError_t launch_wait_check(DevError* err, long long* waits_ns, cudaStream_t stream) {
  if (const cudaError_t e0 = launch_prologue(); e0 != cudaSuccess) return e0;
  wait_check_kernel<<<1, 32, 0, stream>>>(err, waits_ns);
  return cudaGetLastError();
}

}  // namespace msa
