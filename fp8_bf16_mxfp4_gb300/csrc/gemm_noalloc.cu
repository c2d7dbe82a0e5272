// Grouped MX forward GEMM that allocates nothing: its scratch lives in a
// file-scope device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// GEMM: an inference-engine plugin whose device memory is budgeted up front
// and handed out by its host framework (it owns no allocator of its own), or a
// latency-critical path that must never enter an allocator (a cudaMalloc can
// synchronise the device and wait on the allocator's lock).  This entry point
// serves them with a fixed scratch area that is part of the library image on
// every GPU that loads it.
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mxg {
namespace {

// 32 MiB: enough for the packed scales of forward problems up to, for
// example, 8 experts x 14336 x 4096 weights with 8192 routed rows.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

static __device__ __align__(256) uint8_t g_fwd_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on `dev` (set up once per device, with
// that device current).  Host code must not use the symbol itself: on the host
// it names a shadow object, not device memory.
mxg_status scratch_for_device(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDev) return MXG_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) { cudaGetLastError(); return MXG_ERR_CUDA; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) { cudaGetLastError(); return MXG_ERR_CUDA; }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fwd_scratch);
    if (prev != dev) cudaSetDevice(prev);
    if (e != cudaSuccess || p == nullptr) { cudaGetLastError(); return MXG_ERR_CUDA; }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MXG_OK;
}

}  // namespace
}  // namespace mxg

extern "C" mxg_status grouped_gemm_fwd_noalloc(const mxg_mx_operand* A, const mxg_mx_operand* W,
                                               const int32_t* d_m_splits, int32_t G, int64_t N,
                                               void* out, int64_t ld_out, int32_t out_dtype,
                                               int32_t* d_status, void* stream) {
  // the forward's own argument checks come first, so that malformed arguments
  // get the status grouped_gemm_fwd gives them
  if (d_m_splits == nullptr) return MXG_ERR_NULL;
  const mxg_status chk = mxg::fwd_host_checks(A, W, G, N, out, ld_out, out_dtype, d_status);
  if (chk != MXG_OK) return chk;
  const size_t need = mxg_gemm_workspace_size(MXG_PASS_FWD, G, A->rows, N, A->cols, 32);
  if (need == 0) return MXG_ERR_SHAPE;
  if (need > mxg::kNoAllocScratchBytes) return MXG_ERR_WORKSPACE;  // problem too large
  cudaPointerAttributes attr;
  if (cudaPointerGetAttributes(&attr, W->data) != cudaSuccess) {
    cudaGetLastError();
    return MXG_ERR_DEVICE;
  }
  void* scratch = nullptr;
  const mxg_status st = mxg::scratch_for_device(attr.device, &scratch);
  if (st != MXG_OK) return st;
  return grouped_gemm_fwd(A, W, d_m_splits, G, N, out, ld_out, out_dtype, scratch,
                          mxg::kNoAllocScratchBytes, d_status, stream);
}
