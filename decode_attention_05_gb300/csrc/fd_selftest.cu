// fd_selftest.cu -- a check of the kernels' failure path: an in-kernel wait that runs
// out must end with an error status the host can read, never with a hang or a trap.
//
// One CTA initialises an mbarrier that nothing will ever complete and waits on it with
// the same bounded wait (mbar_wait_for) the partial kernels use on their copy ring;
// when the limit passes it raises FD_DEVFLAG_TIMEOUT in the workspace header, exactly
// as a partial kernel does, and returns.  No copy is in flight and nothing else waits,
// so the context stays usable.
#include "fd_device.cuh"

namespace fd {
namespace {

__global__ void fd_wait_selftest_kernel(uint32_t* flags, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_for(smem_addr(&bar), 0, limit_ns))
    atomicOr(flags, kDevFlagTimeout);
}

}  // namespace
}  // namespace fd

extern "C" fd_status fd_selftest_bounded_wait(void* workspace, uint32_t limit_us, void* stream) {
  if (!workspace) return fd::record_error(FD_ERR_INVALID_ARG, "workspace is NULL");
  if (limit_us == 0 || limit_us > 2000000u)
    return fd::record_error(FD_ERR_INVALID_ARG, "limit_us must be in [1, 2000000]");
  fd::fd_wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(
      static_cast<uint32_t*>(workspace), (uint64_t)limit_us * 1000ull);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fd::record_error(FD_ERR_CUDA, cudaGetErrorString(e));
  return FD_OK;
}
