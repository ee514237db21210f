// pkv_selftest_wait: the bounded-wait path of the kernels, on its own.
//
// Every pipeline wait in the attention and write kernels is an mbarrier wait bounded in wall
// time; on expiry the kernel records PKV_DEVERR_TIMEOUT in the device error word and unwinds
// instead of hanging.  This kernel waits on an mbarrier that nothing ever completes, with the
// same wait routine and a caller-chosen limit, so a test can make the wait run out without
// breaking a real pipeline (no copies or MMAs in flight), then read the status with pkv_check
// and keep using the context.

#include "tc_ptx.cuh"

namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(unsigned int* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
    abort_flag = 0;
  }
  __syncwarp();
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, &abort_flag, limit_ns)) pkv_raise(err, PKV_DEVERR_TIMEOUT);
}

}  // namespace

extern "C" pkv_status pkv_selftest_wait(uint64_t limit_ns, void* stream) {
  pkv_clear_error();
  pkv_set_launches(0);
  if (limit_ns == 0 || limit_ns > 10000000000ull)
    return pkv_fail(PKV_ERR_INVALID_ARG, "pkv_selftest_wait: limit must be in (0, 10 s]");
  unsigned int* err = pkv_device_error_word();
  if (!err) return pkv_fail(PKV_ERR_CUDA, "pkv_selftest_wait: device error word unavailable");
  wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, limit_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return pkv_fail(PKV_ERR_CUDA, "pkv_selftest_wait: launch failed: %s", cudaGetErrorString(e));
  pkv_set_launches(1);
  return PKV_OK;
}
