// selftest.cu -- exercises the kernels' bounded-wait path on the GPU without a
// fault: one warp waits on an mbarrier that nothing ever arrives on, through the
// same wait routine the GEMM roles use.  The wait must give up after the
// configured limit, record FGF8_DEVERR_TIMEOUT with its role bit in the status
// word, and let the kernel return normally, leaving the context usable.
#include "gemm_persistent.cuh"

namespace fgf8 {
namespace {

__global__ void __launch_bounds__(32, 1) wait_selftest_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t never;
  __shared__ uint32_t abort_flag;
  const uint32_t bar = ptx::smem_u32(&never);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    abort_flag = 0u;
    ptx::fence_mbar_init();
  }
  __syncwarp();
  PairWaitCtl ctl{&abort_flag, 0u, status, timeout_ns, FGF8_DEVERR_ROLE_SELFTEST};
  pwait(bar, 0u, ctl);   // phase 0 never completes: returns false after timeout_ns
}

}  // namespace

int launch_wait_selftest(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(4, "wait self-test launch: %s", cudaGetErrorString(e));
  return 0;
}

}  // namespace fgf8
