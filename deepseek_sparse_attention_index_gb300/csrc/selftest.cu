// Self-test of the bounded waits every kernel of this library relies on
// (tc::mbar_wait): one thread waits on an mbarrier phase that nothing
// completes.  After the wait's limit (tc::kWaitCycles, about a second) it
// must give up, report DSA_DEVERR_TIMEOUT through err_flag and return, so
// the CUDA context stays usable.  No fault, trap or hang is involved.
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace dsa {

namespace {

__global__ void wait_timeout_selftest_kernel(int32_t *err_flag, long long *out) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);    // one arrival completes phase 0; none comes
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const long long t0 = clock64();
    const bool done = tc::mbar_wait(&bar, 0, &abort_flag);
    const long long waited = clock64() - t0;
    if (!done) raise_flag(err_flag, DSA_DEVERR_TIMEOUT);
    out[0] = done ? 1 : 0;
    out[1] = waited;
    out[2] = tc::kWaitCycles;
  }
}

}  // namespace

}  // namespace dsa

extern "C" int dsa_selftest_wait_timeout(int32_t *err_flag, long long *out, dsa_stream_t stream) {
  if (!err_flag || !out) return DSA_ERR_INVALID_ARG;
  dsa::wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err_flag,
                                                                                         out);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}
