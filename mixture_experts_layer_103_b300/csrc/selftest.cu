// Self-test of the bounded device waits used by the pipelined GEMM kernels.  One thread
// initialises an mbarrier that nothing will ever arrive on and waits on it with the same
// bounded wait the GEMMs use; the wait gives up after the requested time, the kernel
// records MOE_ERR_TIMEOUT in the caller's error word and returns normally, so the CUDA
// context stays usable.  (No fault, trap or unbounded spin is involved.)
#include "moe_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

__global__ void wait_timeout_kernel(int32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = ptx::smem_u32(&bar);
    ptx::mbar_init(b, 1);
    ptx::fence_mbar_init();
    if (!ptx::mbar_wait(b, 0, timeout_ns)) set_device_error(err, MOE_ERR_TIMEOUT);
  }
}

cudaError_t launch_wait_timeout(int32_t* err, uint64_t timeout_ns, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace moe
