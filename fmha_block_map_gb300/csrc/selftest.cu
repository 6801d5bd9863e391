// fbm_selftest_wait_timeout: runs the bounded mbarrier wait of the tcgen05
// kernels on a barrier that nothing ever arrives on, so that the expiry path
// (error bit, clean return, usable context) can be checked on a GPU without
// faulting or hanging it.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace fbm {
fbm_status set_message(fbm_status st, const char *msg);
uint32_t *device_error_word();

namespace {
__global__ void k_wait_selftest(uint32_t *err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(smem_u32(&bar), 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // no thread arrives on `bar`: the wait gives up after limit_ns
    if (!tc::mbar_wait_for(smem_u32(&bar), 0, limit_ns)) set_error(err, FBM_DEVERR_TIMEOUT);
  }
}
}  // namespace
}  // namespace fbm

extern "C" fbm_status fbm_selftest_wait_timeout(uint64_t limit_ns, void *stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return fbm::set_message(FBM_ERR_INVALID_ARG, "fbm_selftest_wait_timeout: limit_ns in (0, 1e10]");
  uint32_t *err = fbm::device_error_word();
  if (!err) return fbm::set_message(FBM_ERR_CUDA, "fbm_selftest_wait_timeout: error word lookup failed");
  fbm::k_wait_selftest<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err, limit_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fbm::set_message(FBM_ERR_CUDA, cudaGetErrorString(e));
  return FBM_OK;
}
