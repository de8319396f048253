// diag.cu -- check of the device-side failure path.
//
// Every mbarrier wait in the attention kernel is bounded: when a phase does
// not complete in time the waiting thread records an error code in the
// workspace error word, raises the CTA's abort flag and returns, so a broken
// pipeline ends with SP_ERR_DEVICE_TIMEOUT instead of hanging the GPU.
// sp_check_barrier_timeout runs that same wait on a barrier that nothing
// ever completes, with a short limit, to show the path works on the device.
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace sp {
namespace {

constexpr int kErrDiagTimeout = 0x1f0;

__global__ void barrier_timeout_kernel(int* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_s;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);  // one arrival expected; none comes
    abort_s = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_s, err, kErrDiagTimeout, timeout_ns);
}

}  // namespace
}  // namespace sp

extern "C" sp_status sp_check_barrier_timeout(void* workspace, int timeout_us,
                                              sp_stream_t stream) {
  sp::NvtxRange nvtx_range("sp_check_barrier_timeout");
  sp::g_last_launches = 0;
  if (!workspace || !sp::aligned(workspace, 256)) return SP_ERR_WORKSPACE;
  if (timeout_us < 1 || timeout_us > 1000000) return SP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(workspace);
  if (cudaMemsetAsync(err, 0, sizeof(int), st) != cudaSuccess) return SP_ERR_CUDA;
  sp::barrier_timeout_kernel<<<1, 32, 0, st>>>(err, 1000ull * timeout_us);
  if (cudaGetLastError() != cudaSuccess) return SP_ERR_CUDA;
  sp::g_last_launches = 1;
  return SP_OK;
}
