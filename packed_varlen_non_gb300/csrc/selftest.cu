// Failure-detection self-test: one CTA waits on a shared-memory barrier that
// nothing arrives on, through the same bounded wait the attention kernel
// uses, and records the timeout in a device word instead of hanging.
#include "device_common.cuh"

namespace h3 {

namespace {

__global__ void selftest_bounded_wait_kernel(uint64_t timeout_ns, uint32_t* flag) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    dev::mbar_init(dev::smem_u32(&bar), 1);
    dev::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Phase 0 never completes: the wait must give up after timeout_ns.
    const bool ok = dev::mbar_wait_bounded(dev::smem_u32(&bar), 0, &abort_flag, flag, timeout_ns);
    if (ok) atomicExch(flag, 0xdeadu);  // would mean the barrier completed on its own
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_bounded_wait(uint64_t timeout_ns, uint32_t* d_flag, cudaStream_t stream) {
  selftest_bounded_wait_kernel<<<1, 32, 0, stream>>>(timeout_ns, d_flag);
  return cudaGetLastError();
}

}  // namespace h3
