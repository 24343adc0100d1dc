// rz_selftest.cu -- exercises the library's bounded pipeline wait on the GPU
// without faulting or hanging it: one warp waits on an mbarrier that nothing
// will ever arrive on, with the same bounded wait every pipeline stage of the
// GEMM kernels uses, and must give up after the given limit and report
// RZ_DEVERR_TIMEOUT through the caller's error word.
#include <cuda_runtime.h>

#include <cstdint>

#include "rz.h"
#include "rz_internal.h"
#include "rz_ptx.cuh"

namespace rz {
namespace {

__global__ void wait_timeout_kernel(int* err, unsigned long long limit_ns, int* done) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // phase 0 never completes: no thread arrives and no copy is issued
    const bool ok = mbar_wait(&bar, 0, &abort_flag, limit_ns);
    if (!ok && err) atomicOr(err, RZ_DEVERR_TIMEOUT);
    if (done) *done = ok ? 1 : 2;
  }
}

}  // namespace
}  // namespace rz

extern "C" int rz_selftest_wait_timeout(int32_t* err_flag, int32_t* done_out, uint32_t limit_us,
                                        rz_stream_t stream) {
  if (!err_flag || limit_us == 0 || limit_us > 2000000u) return RZ_ERR_INVALID_ARG;
  if (!rz::device_ok()) return RZ_ERR_UNSUPPORTED;
  rz::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      err_flag, 1000ull * limit_us, done_out);
  return cudaGetLastError() == cudaSuccess ? RZ_OK : RZ_ERR_CUDA;
}
