// Diagnostic kernel for the bounded waits (see mxg_diag_bounded_wait in mxg.h).
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace mxg {
namespace {

__global__ void bounded_wait_kernel(int32_t* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing arrives on the barrier: phase 0 never completes
    ptx::mbar_wait(b, 0, &abort_flag, status, timeout_ns);
  }
}

}  // namespace
}  // namespace mxg

extern "C" mxg_status mxg_diag_bounded_wait(int32_t* d_status, uint64_t timeout_ns, void* stream) {
  if (d_status == nullptr) return MXG_ERR_NULL;
  if (timeout_ns > 10000000000ull) return MXG_ERR_SHAPE;  // at most 10 s
  mxg::bounded_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(d_status, timeout_ns);
  return cudaGetLastError() == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}
