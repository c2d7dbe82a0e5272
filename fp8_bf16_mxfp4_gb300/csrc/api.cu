// C-ABI layer of libmxg: argument checks, device checks and dispatch.
//
// Host checks never touch the GPU, so the error paths can be exercised on a
// machine without one.  Device placement is taken from the operands' pointers
// (not from the calling thread's current device): the review "Check operand
// device instead of current CUDA device" on ROCm TransformerEngine PR #745.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mxg {

static std::atomic<uint64_t> g_wait_timeout_ns{2000000000ull};
uint64_t wait_timeout_ns() { return g_wait_timeout_ns.load(std::memory_order_relaxed); }
static std::atomic<int> g_gemm_cta_group{2};
int gemm_cta_group() { return g_gemm_cta_group.load(std::memory_order_relaxed); }

namespace {

constexpr int kMaxDevices = 64;
struct DevInfo {
  int checked = 0;  // 0 unknown, 1 ok, -1 unsupported
  int num_sms = 0;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// All non-null pointers must be device (or managed) memory of one device that
// is an sm_103 part.  On success *dev and *num_sms describe it.
mxg_status check_device(std::initializer_list<const void*> ptrs, int* dev, int* num_sms) {
  int d = -1;
  for (const void* p : ptrs) {
    if (p == nullptr) continue;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
      cudaGetLastError();
      return MXG_ERR_DEVICE;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return MXG_ERR_DEVICE;
    if (d < 0) d = attr.device;
    else if (attr.device != d) return MXG_ERR_DEVICE;
  }
  if (d < 0 || d >= kMaxDevices) return MXG_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_dev[d].checked == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) {
      cudaGetLastError();
      return MXG_ERR_CUDA;
    }
    g_dev[d].checked = (major == 10 && minor == 3) ? 1 : -1;
    g_dev[d].num_sms = sms;
  }
  if (g_dev[d].checked != 1) return MXG_ERR_DEVICE;
  *dev = d;
  *num_sms = g_dev[d].num_sms;
  return MXG_OK;
}

// Makes `dev` current for the scope of a call and restores the caller's.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

inline mxg_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MXG_OK;
  cudaGetLastError();
  return MXG_ERR_CUDA;
}

inline int64_t code_bytes(int elem, int64_t cols) { return elem == MXG_E2M1 ? cols / 2 : cols; }
inline bool valid_elem(int32_t e) { return e == MXG_E2M1 || e == MXG_E4M3; }
// A quantizer's elem argument: the element format, optionally with the
// MXG_SCALE_ROUND_UP rule flag (carried on to the launchers).
inline bool valid_quant_elem(int32_t e) { return valid_elem(e & ~MXG_SCALE_ROUND_UP); }

// Host checks of one MX GEMM operand.  An operand with no elements (rows == 0,
// or cols == 0 where `allow_no_cols`) may have NULL data and scale pointers.
// Packed scales are accepted only where `allow_packed`.
mxg_status check_operand(const mxg_mx_operand* op, bool allow_no_cols = false, bool allow_packed = false) {
  if (op == nullptr) return MXG_ERR_NULL;
  if (!valid_elem(op->elem)) return MXG_ERR_UNSUPPORTED;
  const bool packed = op->scale_layout == MXG_SCALE_PACKED;
  if (!(op->scale_layout == MXG_SCALE_PLAIN || (packed && allow_packed))) return MXG_ERR_UNSUPPORTED;
  if (op->rows < 0 || op->cols < 0 || op->cols % 32 != 0) return MXG_ERR_SHAPE;
  if (op->cols == 0 && !allow_no_cols) return MXG_ERR_SHAPE;
  if (op->ld < code_bytes(op->elem, op->cols) || (!packed && op->scale_ld < op->cols / 32)) return MXG_ERR_SHAPE;
  if (op->ld % 16 != 0) return MXG_ERR_ALIGN;
  if (op->rows == 0 || op->cols == 0) return MXG_OK;
  if (op->data == nullptr || op->scale == nullptr) return MXG_ERR_NULL;
  if (!aligned16(op->data) || (packed && !aligned16(op->scale))) return MXG_ERR_ALIGN;
  return MXG_OK;
}

// `rows` == 0 allows a NULL output.
mxg_status check_out(const void* out, int64_t rows, int64_t ld_out, int64_t ncols, int32_t dtype) {
  if (dtype != MXG_OUT_BF16 && dtype != MXG_OUT_F32) return MXG_ERR_UNSUPPORTED;
  if (ld_out < ncols) return MXG_ERR_SHAPE;
  // the epilogue writes whole 32-byte sectors
  const int64_t esz = dtype == MXG_OUT_BF16 ? 2 : 4;
  if ((ld_out * esz) % 32 != 0) return MXG_ERR_ALIGN;
  if (rows == 0) return MXG_OK;
  if (out == nullptr) return MXG_ERR_NULL;
  if (!aligned(out, 32)) return MXG_ERR_ALIGN;
  return MXG_OK;
}

// Host checks of one blockwise operand (rows may be 0; cols a multiple of
// 128, 0 only where allowed).
mxg_status check_bw_operand(const mxg_bw_operand* op, bool allow_no_cols = false) {
  if (op == nullptr) return MXG_ERR_NULL;
  if (op->reserved0 != 0 || op->reserved1 != 0) return MXG_ERR_UNSUPPORTED;
  if (op->rows < 0 || op->cols < 0 || op->cols % 128 != 0) return MXG_ERR_SHAPE;
  if (op->cols == 0 && !allow_no_cols) return MXG_ERR_SHAPE;
  if (op->ld < op->cols || op->ld % 16 != 0 || op->scale_ld < 0) return op->ld % 16 ? MXG_ERR_ALIGN : MXG_ERR_SHAPE;
  if (op->rows == 0 || op->cols == 0) return MXG_OK;
  if (op->data == nullptr || op->scale == nullptr) return MXG_ERR_NULL;
  if (!aligned16(op->data) || !aligned(op->scale, 4)) return MXG_ERR_ALIGN;
  return MXG_OK;
}

BwGemmArgs bw_args(int pass, int G, const mxg_bw_operand* A, const mxg_bw_operand* B,
                   const int32_t* splits, int64_t S, int64_t N, int64_t K, void* out,
                   int64_t ld_out, int32_t dtype, int acc, void* ws, int32_t* st) {
  BwGemmArgs a{};
  a.pass = pass;
  a.G = G;
  a.a_data = static_cast<const uint8_t*>(A->data); a.a_ld = A->ld;
  a.a_scale = A->scale; a.a_scale_ld = A->scale_ld;
  a.a_rows = A->rows; a.a_cols = A->cols;
  a.b_data = static_cast<const uint8_t*>(B->data); a.b_ld = B->ld;
  a.b_scale = B->scale; a.b_scale_ld = B->scale_ld;
  a.b_rows = B->rows; a.b_cols = B->cols;
  a.splits = splits;
  a.total_rows = S;
  a.N = N; a.K = K;
  a.out = out; a.ld_out = ld_out; a.out_dtype = dtype; a.accumulate = acc;
  a.ws = ws; a.status = st;
  return a;
}

}  // namespace
}  // namespace mxg

using namespace mxg;

extern "C" {

int32_t mxg_version(void) { return 200; }

void mxg_set_wait_timeout_ns(uint64_t ns) { g_wait_timeout_ns.store(ns ? ns : 1, std::memory_order_relaxed); }
uint64_t mxg_get_wait_timeout_ns(void) { return wait_timeout_ns(); }
mxg_status mxg_set_gemm_cta_group(int32_t n) {
  if (n != 1 && n != 2) return MXG_ERR_SHAPE;
  mxg::g_gemm_cta_group.store(n, std::memory_order_relaxed);
  return MXG_OK;
}
int32_t mxg_get_gemm_cta_group(void) { return mxg::gemm_cta_group(); }

const char* mxg_status_string(mxg_status s) {
  switch (s) {
    case MXG_OK: return "ok";
    case MXG_ERR_NULL: return "a required pointer is NULL";
    case MXG_ERR_SHAPE: return "sizes inconsistent or not divisible as required";
    case MXG_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case MXG_ERR_SPLITS: return "m_splits has a negative entry or does not sum to the row count";
    case MXG_ERR_UNSUPPORTED: return "format combination or option not supported";
    case MXG_ERR_DEVICE: return "pointer not on one sm_103 device";
    case MXG_ERR_CUDA: return "CUDA runtime error";
    case MXG_ERR_TIMEOUT: return "a bounded in-kernel wait ran out";
    case MXG_ERR_WORKSPACE: return "workspace missing or too small";
    case MXG_ERR_CAPACITY: return "padded rows exceed the output capacity";
  }
  return "unknown status";
}

int64_t mx_padded_rows_capacity(int64_t rows, int32_t G, int32_t pad) {
  if (rows < 0 || G < 1 || pad < 1) return -1;
  const int64_t nonempty = rows < G ? rows : (int64_t)G;  // experts that can add padding
  return ((rows + nonempty * (pad - 1)) / pad) * pad;
}

mxg_status mxg_check_status(int32_t* d_status, void* stream) {
  if (d_status == nullptr) return MXG_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, d_status, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(d_status, 0, sizeof(int32_t), st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    cudaGetLastError();
    return MXG_ERR_CUDA;
  }
  return static_cast<mxg_status>(v);
}

mxg_status mx_quantize_rowwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                               int32_t elem, void* q, int64_t ld_q, uint8_t* s, int64_t ld_s,
                               void* stream) {
  if (!valid_quant_elem(elem)) return MXG_ERR_UNSUPPORTED;
  if (rows < 0 || cols <= 0 || cols % 32 != 0) return MXG_ERR_SHAPE;
  if (ld_x < cols || ld_q < code_bytes(elem & ~MXG_SCALE_ROUND_UP, cols) || ld_s < cols / 32) return MXG_ERR_SHAPE;
  // codes are written 16 bytes per block (E2M1) or two 16-byte halves (E4M3)
  if (ld_x % 8 != 0 || ld_q % 16 != 0) return MXG_ERR_ALIGN;
  if (rows == 0) return MXG_OK;  // nothing to read or write; pointers may be NULL
  if (x == nullptr || q == nullptr || s == nullptr) return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned16(q)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, q, s}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_mx_rowwise(x, rows, cols, ld_x, elem, q, ld_q, s, ld_s,
                                       static_cast<cudaStream_t>(stream), sms));
}

int64_t mx_packed_scale_bytes(int64_t rows, int64_t cols, int32_t G) {
  if (rows < 0 || cols < 0 || cols % 32 != 0 || G < 1 || G > kMaxExperts) return -1;
  const int64_t nonempty = rows < G ? rows : (int64_t)G;
  const int64_t rt_max = (rows + nonempty * 127) / 128;
  return (cols + 127) / 128 * rt_max * 512;
}

mxg_status mx_quantize_rowwise_packed(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                      int32_t elem, void* q, int64_t ld_q, uint8_t* s_packed,
                                      int64_t s_bytes, const int32_t* d_m_splits, int32_t G,
                                      int32_t* d_status, void* stream) {
  if (!valid_quant_elem(elem)) return MXG_ERR_UNSUPPORTED;
  if (G < 1 || G > kMaxExperts) return MXG_ERR_SHAPE;
  if (rows < 0 || cols <= 0 || cols % 32 != 0) return MXG_ERR_SHAPE;
  if (d_m_splits == nullptr && rows % G != 0) return MXG_ERR_SHAPE;
  if (ld_x < cols || ld_q < code_bytes(elem & ~MXG_SCALE_ROUND_UP, cols)) return MXG_ERR_SHAPE;
  if (ld_x % 8 != 0 || ld_q % 16 != 0) return MXG_ERR_ALIGN;
  if (d_m_splits != nullptr && d_status == nullptr) return MXG_ERR_NULL;
  const int64_t need = mx_packed_scale_bytes(rows, cols, G);
  if (s_bytes < need) return MXG_ERR_SHAPE;
  // the split check still runs when there are no rows (a non-zero split is an error)
  if (rows == 0 && d_m_splits == nullptr) return MXG_OK;
  if ((rows > 0 && (x == nullptr || q == nullptr)) || (need > 0 && s_packed == nullptr)) return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(s_packed)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, q, s_packed, d_m_splits, d_status}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  const int64_t nonempty = rows < G ? rows : (int64_t)G;
  const int64_t rt_bound = d_m_splits ? (rows + nonempty * 127) / 128 : (int64_t)G * ((rows / G + 127) / 128);
  return cuda_status(launch_mx_rowwise_packed(x, rows, cols, ld_x, elem, q, ld_q, s_packed, d_m_splits, G,
                                              d_m_splits ? 0 : rows / G, rt_bound, d_status,
                                              static_cast<cudaStream_t>(stream), sms));
}

int64_t mx_packed_colwise_scale_bytes(int64_t cols, int64_t capacity, int32_t G) {
  if (cols < 0 || capacity < 0 || cols % 32 != 0 || capacity % 32 != 0 || G < 1 || G > kMaxExperts) return -1;
  return (capacity / 128 + G) * ((cols + 127) / 128) * 512;
}

mxg_status mx_quantize_colwise_segment_padded_packed(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                                     const int32_t* d_m_splits, int32_t G, int32_t pad_multiple,
                                                     int32_t elem, void* qT, int64_t ld_q, uint8_t* s_packed,
                                                     int64_t s_bytes, int64_t capacity, int64_t* d_pad_offsets,
                                                     int32_t* d_status, void* stream) {
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (!valid_quant_elem(elem)) return MXG_ERR_UNSUPPORTED;
  if (G < 1 || G > kMaxExperts) return MXG_ERR_SHAPE;
  if (pad_multiple <= 0 || pad_multiple % 32 != 0) return MXG_ERR_SHAPE;
  if (rows < 0 || cols <= 0 || cols % 32 != 0 || capacity < 0 || capacity % 32 != 0) return MXG_ERR_SHAPE;
  if (ld_x < cols || ld_q < code_bytes(elem & ~MXG_SCALE_ROUND_UP, capacity)) return MXG_ERR_SHAPE;
  if (ld_x % 8 != 0 || ld_q % 16 != 0) return MXG_ERR_ALIGN;
  const int64_t need = mx_packed_colwise_scale_bytes(cols, capacity, G);
  if (s_bytes < need) return MXG_ERR_SHAPE;
  if ((rows > 0 && x == nullptr) || (capacity > 0 && qT == nullptr) || (need > 0 && s_packed == nullptr))
    return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned16(qT) || !aligned16(s_packed) || !aligned(d_pad_offsets, 8)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, d_m_splits, qT, s_packed, d_pad_offsets, d_status}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_mx_colwise(x, rows, cols, ld_x, d_m_splits, G, pad_multiple, elem, qT, ld_q,
                                       s_packed, 0, capacity, d_pad_offsets, d_status,
                                       static_cast<cudaStream_t>(stream), sms, nullptr, 0, nullptr, 0,
                                       need > 0 ? need : 0));
}

mxg_status mx_quantize_colwise_segment_padded(const void* x, int64_t rows, int64_t cols,
                                              int64_t ld_x, const int32_t* d_m_splits,
                                              int32_t G, int32_t pad_multiple, int32_t elem,
                                              void* qT, int64_t ld_q, uint8_t* sT, int64_t ld_s,
                                              int64_t capacity, int64_t* d_pad_offsets,
                                              int32_t* d_status, void* stream) {
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (!valid_quant_elem(elem)) return MXG_ERR_UNSUPPORTED;
  if (G < 1 || G > kMaxExperts) return MXG_ERR_SHAPE;
  if (pad_multiple <= 0 || pad_multiple % 32 != 0) return MXG_ERR_SHAPE;
  if (rows < 0 || cols <= 0 || cols % 32 != 0 || capacity < 0 || capacity % 32 != 0)
    return MXG_ERR_SHAPE;
  if (ld_x < cols || ld_q < code_bytes(elem & ~MXG_SCALE_ROUND_UP, capacity) || ld_s < capacity / 32) return MXG_ERR_SHAPE;
  if (ld_x % 8 != 0 || ld_q % 16 != 0) return MXG_ERR_ALIGN;
  // x may be NULL when there are no rows; qT / sT when there is no capacity
  if ((rows > 0 && x == nullptr) || (capacity > 0 && (qT == nullptr || sT == nullptr)))
    return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned16(qT) || !aligned(d_pad_offsets, 8)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, d_m_splits, qT, sT, d_pad_offsets, d_status}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_mx_colwise(x, rows, cols, ld_x, d_m_splits, G, pad_multiple, elem, qT,
                                       ld_q, sT, ld_s, capacity, d_pad_offsets, d_status,
                                       static_cast<cudaStream_t>(stream), sms));
}

mxg_status mx_quantize_dual_segment_padded(const void* x, int64_t rows, int64_t cols,
                                           int64_t ld_x, const int32_t* d_m_splits, int32_t G,
                                           int32_t pad_multiple, int32_t elem, void* q,
                                           int64_t ld_q, uint8_t* s, int64_t ld_s, void* qT,
                                           int64_t ld_qT, uint8_t* sT, int64_t ld_sT,
                                           int64_t capacity, int64_t* d_pad_offsets,
                                           int32_t* d_status, void* stream) {
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (!valid_quant_elem(elem)) return MXG_ERR_UNSUPPORTED;
  if (G < 1 || G > kMaxExperts) return MXG_ERR_SHAPE;
  if (pad_multiple <= 0 || pad_multiple % 32 != 0) return MXG_ERR_SHAPE;
  if (rows < 0 || cols <= 0 || cols % 32 != 0 || capacity < 0 || capacity % 32 != 0)
    return MXG_ERR_SHAPE;
  if (ld_x < cols || ld_q < code_bytes(elem & ~MXG_SCALE_ROUND_UP, cols) || ld_s < cols / 32 ||
      ld_qT < code_bytes(elem & ~MXG_SCALE_ROUND_UP, capacity) || ld_sT < capacity / 32)
    return MXG_ERR_SHAPE;
  if (ld_x % 8 != 0 || ld_q % 16 != 0 || ld_qT % 16 != 0) return MXG_ERR_ALIGN;
  // x, q, s may be NULL when there are no rows; qT / sT when there is no capacity
  if ((rows > 0 && (x == nullptr || q == nullptr || s == nullptr)) ||
      (capacity > 0 && (qT == nullptr || sT == nullptr)))
    return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(qT) || !aligned(d_pad_offsets, 8))
    return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, q, s, d_m_splits, qT, sT, d_pad_offsets, d_status}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  // with no rows the row-wise half has nothing to write; the launch still
  // validates the splits and fills the padded offsets
  return cuda_status(launch_mx_colwise(x, rows, cols, ld_x, d_m_splits, G, pad_multiple, elem, qT,
                                       ld_qT, sT, ld_sT, capacity, d_pad_offsets, d_status,
                                       static_cast<cudaStream_t>(stream), sms,
                                       rows > 0 ? q : nullptr, ld_q, s, ld_s));
}

size_t mxg_gemm_workspace_size(int32_t pass, int32_t G, int64_t S, int64_t N, int64_t K,
                               int32_t pad_multiple) {
  if (G < 1 || G > kMaxExperts || S < 0 || N <= 0 || K <= 0) return 0;
  if (pass < MXG_PASS_FWD || pass > MXG_PASS_WGRAD) return 0;
  if (pass == MXG_PASS_WGRAD && (pad_multiple <= 0 || pad_multiple % 32 != 0)) return 0;
  return gemm_workspace_bytes(pass, G, S, N, K, pad_multiple);
}

}  // extern "C"

// The forward's host checks that precede the workspace check, in the order
// the forward entry points apply them.
mxg_status mxg::fwd_host_checks(const mxg_mx_operand* A, const mxg_mx_operand* W, int32_t G, int64_t N,
                           const void* out, int64_t ld_out, int32_t out_dtype, const int32_t* d_status) {
  mxg_status st;
  if ((st = check_operand(A, false, true)) != MXG_OK || (st = check_operand(W, false, true)) != MXG_OK)
    return st;
  if (d_status == nullptr) return MXG_ERR_NULL;
  if ((st = check_out(const_cast<void*>(out), A->rows, ld_out, N, out_dtype)) != MXG_OK) return st;
  if (G < 1 || G > kMaxExperts || N <= 0 || N % 32 != 0) return MXG_ERR_SHAPE;
  if (W->rows == 0) return MXG_ERR_SHAPE;
  if (A->cols != W->cols || W->rows != (int64_t)G * N) return MXG_ERR_SHAPE;
  const bool a8w4 = A->elem == MXG_E4M3 && W->elem == MXG_E2M1;
  if (A->elem == MXG_E2M1 && W->elem == MXG_E4M3) return MXG_ERR_UNSUPPORTED;
  if (a8w4) {
    if (A->cols % 128 != 0) return MXG_ERR_SHAPE;
    if (!aligned(W->data, 32) || W->ld % 32 != 0) return MXG_ERR_ALIGN;
  }
  return MXG_OK;
}

namespace {
// The forward pass; d_m_splits == NULL means one expert of all A->rows rows
// (the dense entry point, G == 1).
mxg_status fwd_impl(const mxg_mx_operand* A, const mxg_mx_operand* W, const int32_t* d_m_splits,
                    int32_t G, int64_t N, void* out, int64_t ld_out, int32_t out_dtype, void* ws,
                    size_t ws_bytes, int32_t* d_status, void* stream) {
  mxg_status st;
  if ((st = fwd_host_checks(A, W, G, N, out, ld_out, out_dtype, d_status)) != MXG_OK) return st;
  const size_t need = gemm_workspace_bytes(MXG_PASS_FWD, G, A->rows, N, A->cols, 32);
  if (ws_bytes < need || (need > 0 && ws == nullptr)) return MXG_ERR_WORKSPACE;
  if (ws != nullptr && !aligned(ws, 256)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  if ((st = check_device({A->data, A->scale, W->data, W->scale, d_m_splits, out, ws, d_status},
                         &dev, &sms)) != MXG_OK)
    return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  GemmArgs a{};
  a.pass = MXG_PASS_FWD;
  a.G = G;
  a.a_data = static_cast<const uint8_t*>(A->data); a.a_ld = A->ld;
  a.a_scale = A->scale; a.a_scale_ld = A->scale_ld;
  a.a_rows = A->rows; a.a_cols = A->cols; a.a_elem = A->elem;
  a.b_data = static_cast<const uint8_t*>(W->data); a.b_ld = W->ld;
  a.b_scale = W->scale; a.b_scale_ld = W->scale_ld;
  a.b_rows = W->rows; a.b_cols = W->cols; a.b_elem = W->elem;
  a.a_packed = A->scale_layout == MXG_SCALE_PACKED;
  a.b_packed = W->scale_layout == MXG_SCALE_PACKED;
  a.splits = d_m_splits;
  a.total_rows = A->rows;
  a.N = N; a.K = A->cols;
  a.pad = 32;
  a.out = out; a.ld_out = ld_out; a.out_dtype = out_dtype; a.accumulate = 0;
  a.ws = ws; a.ws_bytes = ws_bytes; a.status = d_status;
  return launch_grouped_gemm(a, static_cast<cudaStream_t>(stream), sms);
}
}  // namespace

extern "C" {

mxg_status grouped_gemm_fwd(const mxg_mx_operand* A, const mxg_mx_operand* W,
                            const int32_t* d_m_splits, int32_t G, int64_t N, void* out,
                            int64_t ld_out, int32_t out_dtype, void* ws, size_t ws_bytes,
                            int32_t* d_status, void* stream) {
  if (d_m_splits == nullptr) return MXG_ERR_NULL;
  return fwd_impl(A, W, d_m_splits, G, N, out, ld_out, out_dtype, ws, ws_bytes, d_status, stream);
}

mxg_status mx_gemm_dense(const mxg_mx_operand* A, const mxg_mx_operand* B, void* out, int64_t ld_out,
                         int32_t out_dtype, void* ws, size_t ws_bytes, int32_t* d_status, void* stream) {
  if (B == nullptr) return MXG_ERR_NULL;
  return fwd_impl(A, B, nullptr, 1, B->rows, out, ld_out, out_dtype, ws, ws_bytes, d_status, stream);
}

mxg_status grouped_gemm_dgrad(const mxg_mx_operand* dY, const mxg_mx_operand* Wt,
                              const int32_t* d_m_splits, int32_t G, void* out, int64_t ld_out,
                              int32_t out_dtype, void* ws, size_t ws_bytes, int32_t* d_status,
                              void* stream) {
  mxg_status st;
  if ((st = check_operand(dY, false, true)) != MXG_OK || (st = check_operand(Wt, false, true)) != MXG_OK)
    return st;
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (G < 1 || G > kMaxExperts) return MXG_ERR_SHAPE;
  const int64_t N = dY->cols, K = Wt->rows;
  if (K <= 0 || K % 32 != 0 || Wt->cols != (int64_t)G * N) return MXG_ERR_SHAPE;
  if ((st = check_out(out, dY->rows, ld_out, K, out_dtype)) != MXG_OK) return st;
  if (dY->elem != Wt->elem) return MXG_ERR_UNSUPPORTED;  // a8w4 is forward-only
  const size_t need = gemm_workspace_bytes(MXG_PASS_DGRAD, G, dY->rows, N, K, 32);
  if (ws_bytes < need || (need > 0 && ws == nullptr)) return MXG_ERR_WORKSPACE;
  if (ws != nullptr && !aligned(ws, 256)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  if ((st = check_device({dY->data, dY->scale, Wt->data, Wt->scale, d_m_splits, out, ws, d_status},
                         &dev, &sms)) != MXG_OK)
    return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  GemmArgs a{};
  a.pass = MXG_PASS_DGRAD;
  a.G = G;
  a.a_data = static_cast<const uint8_t*>(dY->data); a.a_ld = dY->ld;
  a.a_scale = dY->scale; a.a_scale_ld = dY->scale_ld;
  a.a_rows = dY->rows; a.a_cols = dY->cols; a.a_elem = dY->elem;
  a.b_data = static_cast<const uint8_t*>(Wt->data); a.b_ld = Wt->ld;
  a.b_scale = Wt->scale; a.b_scale_ld = Wt->scale_ld;
  a.b_rows = Wt->rows; a.b_cols = Wt->cols; a.b_elem = Wt->elem;
  a.a_packed = dY->scale_layout == MXG_SCALE_PACKED;
  a.b_packed = Wt->scale_layout == MXG_SCALE_PACKED;
  a.splits = d_m_splits;
  a.total_rows = dY->rows;
  a.N = N; a.K = K;
  a.pad = 32;
  a.out = out; a.ld_out = ld_out; a.out_dtype = out_dtype; a.accumulate = 0;
  a.ws = ws; a.ws_bytes = ws_bytes; a.status = d_status;
  return launch_grouped_gemm(a, static_cast<cudaStream_t>(stream), sms);
}

mxg_status grouped_gemm_wgrad(const mxg_mx_operand* dYt, const mxg_mx_operand* Xt,
                              const int32_t* d_m_splits, int32_t G, int64_t total_rows,
                              int32_t pad_multiple, void* out, int32_t out_dtype,
                              int32_t accumulate, void* ws, size_t ws_bytes, int32_t* d_status,
                              void* stream) {
  mxg_status st;
  if ((st = check_operand(dYt, true, true)) != MXG_OK || (st = check_operand(Xt, true, true)) != MXG_OK)
    return st;
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (G < 1 || G > kMaxExperts || total_rows < 0) return MXG_ERR_SHAPE;
  if (pad_multiple <= 0 || pad_multiple % 32 != 0) return MXG_ERR_SHAPE;
  const int64_t N = dYt->rows, K = Xt->rows;
  if (N <= 0 || K <= 0 || N % 32 != 0 || K % 32 != 0 || dYt->cols != Xt->cols) return MXG_ERR_SHAPE;
  if ((st = check_out(out, 1, K, K, out_dtype)) != MXG_OK) return st;
  if (accumulate && out_dtype != MXG_OUT_F32) return MXG_ERR_UNSUPPORTED;
  if (dYt->elem != Xt->elem) return MXG_ERR_UNSUPPORTED;
  const size_t need = gemm_workspace_bytes(MXG_PASS_WGRAD, G, dYt->cols, N, K, pad_multiple);
  if (ws_bytes < need || (need > 0 && ws == nullptr)) return MXG_ERR_WORKSPACE;
  if (ws != nullptr && !aligned(ws, 256)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  if ((st = check_device({dYt->data, dYt->scale, Xt->data, Xt->scale, d_m_splits, out, ws, d_status},
                         &dev, &sms)) != MXG_OK)
    return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  GemmArgs a{};
  a.pass = MXG_PASS_WGRAD;
  a.G = G;
  a.a_data = static_cast<const uint8_t*>(dYt->data); a.a_ld = dYt->ld;
  a.a_scale = dYt->scale; a.a_scale_ld = dYt->scale_ld;
  a.a_rows = dYt->rows; a.a_cols = dYt->cols; a.a_elem = dYt->elem;
  a.b_data = static_cast<const uint8_t*>(Xt->data); a.b_ld = Xt->ld;
  a.b_scale = Xt->scale; a.b_scale_ld = Xt->scale_ld;
  a.b_rows = Xt->rows; a.b_cols = Xt->cols; a.b_elem = Xt->elem;
  a.a_packed = dYt->scale_layout == MXG_SCALE_PACKED;
  a.b_packed = Xt->scale_layout == MXG_SCALE_PACKED;
  a.splits = d_m_splits;
  a.total_rows = total_rows;
  a.N = N; a.K = K;
  a.pad = pad_multiple;
  a.out = out; a.ld_out = K; a.out_dtype = out_dtype; a.accumulate = accumulate ? 1 : 0;
  a.ws = ws; a.ws_bytes = ws_bytes; a.status = d_status;
  return launch_grouped_gemm(a, static_cast<cudaStream_t>(stream), sms);
}


// ------------------------------------------------------------------ blockwise FP8

mxg_status bw_quantize_1x128(const void* x, int64_t rows, int64_t cols, int64_t ld_x, void* q,
                             int64_t ld_q, float* s, int64_t ld_s, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 128 != 0) return MXG_ERR_SHAPE;
  if (ld_x < cols || ld_q < cols || ld_s < rows) return MXG_ERR_SHAPE;
  if (ld_x % 8 != 0 || ld_q % 8 != 0) return MXG_ERR_ALIGN;
  if (rows == 0) return MXG_OK;
  if (x == nullptr || q == nullptr || s == nullptr) return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned(q, 8) || !aligned(s, 4)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, q, s}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_bw_rowwise(x, rows, cols, ld_x, q, ld_q, s, ld_s, false,
                                       static_cast<cudaStream_t>(stream), sms));
}

mxg_status bw_quantize_128x128(const void* w, int64_t rows, int64_t cols, int64_t ld_w, void* q,
                               int64_t ld_q, float* s, void* qT, int64_t ld_qT, float* sT,
                               void* stream) {
  if ((qT == nullptr) != (sT == nullptr)) return MXG_ERR_NULL;
  if (rows < 0 || cols <= 0 || rows % 128 != 0 || cols % 128 != 0) return MXG_ERR_SHAPE;
  if (ld_w < cols || ld_q < cols || (qT != nullptr && ld_qT < rows)) return MXG_ERR_SHAPE;
  if (rows / 128 > 65535 || cols / 128 > 0x7FFFFFFF) return MXG_ERR_SHAPE;
  if (ld_w % 8 != 0 || ld_q % 16 != 0 || (qT != nullptr && ld_qT % 16 != 0)) return MXG_ERR_ALIGN;
  if (rows == 0) return MXG_OK;
  if (w == nullptr || q == nullptr || s == nullptr) return MXG_ERR_NULL;
  if (!aligned16(w) || !aligned16(q) || !aligned16(qT) || !aligned(s, 4) || !aligned(sT, 4))
    return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({w, q, s, qT, sT}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_bw_weight(w, rows, cols, ld_w, q, ld_q, s, 0, qT, ld_qT, sT, 0, false,
                                      static_cast<cudaStream_t>(stream), sms));
}

mxg_status bw_quantize_colwise_padded(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                      const int32_t* d_m_splits, int32_t G, void* qT,
                                      int64_t ld_q, float* sT, int64_t ld_s, int64_t capacity,
                                      int64_t* d_pad_offsets, int32_t* d_status, void* stream) {
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (G < 1 || G > kMaxExperts) return MXG_ERR_SHAPE;
  if (rows < 0 || cols <= 0 || cols % 32 != 0 || capacity < 0 || capacity % 128 != 0)
    return MXG_ERR_SHAPE;
  if (ld_x < cols || ld_q < capacity || ld_s < cols) return MXG_ERR_SHAPE;
  if (ld_x % 8 != 0 || ld_q % 16 != 0) return MXG_ERR_ALIGN;
  if ((rows > 0 && x == nullptr) || (capacity > 0 && (qT == nullptr || sT == nullptr)))
    return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned16(qT) || !aligned(sT, 4) || !aligned(d_pad_offsets, 8))
    return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, d_m_splits, qT, sT, d_pad_offsets, d_status}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_bw_colwise(x, rows, cols, ld_x, d_m_splits, G, qT, ld_q, sT, ld_s,
                                       capacity, d_pad_offsets, d_status, false,
                                       static_cast<cudaStream_t>(stream), sms));
}

// ---- power-of-two blockwise scales, written as MX (UE8M0 per 32) operands

mxg_status bw_quantize_1x128_pow2(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                  void* q, int64_t ld_q, uint8_t* s, int64_t ld_s, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 128 != 0) return MXG_ERR_SHAPE;
  if (ld_x < cols || ld_q < cols || ld_s < cols / 32) return MXG_ERR_SHAPE;
  if (ld_x % 8 != 0 || ld_q % 8 != 0 || ld_s % 4 != 0) return MXG_ERR_ALIGN;
  if (rows == 0) return MXG_OK;
  if (x == nullptr || q == nullptr || s == nullptr) return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned(q, 8) || !aligned(s, 4)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, q, s}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_bw_rowwise(x, rows, cols, ld_x, q, ld_q, s, ld_s, true,
                                       static_cast<cudaStream_t>(stream), sms));
}

mxg_status bw_quantize_128x128_pow2(const void* w, int64_t rows, int64_t cols, int64_t ld_w,
                                    void* q, int64_t ld_q, uint8_t* s, int64_t ld_s, void* qT,
                                    int64_t ld_qT, uint8_t* sT, int64_t ld_sT, void* stream) {
  if ((qT == nullptr) != (sT == nullptr)) return MXG_ERR_NULL;
  if (rows < 0 || cols <= 0 || rows % 128 != 0 || cols % 128 != 0) return MXG_ERR_SHAPE;
  if (ld_w < cols || ld_q < cols || ld_s < cols / 32) return MXG_ERR_SHAPE;
  if (qT != nullptr && (ld_qT < rows || ld_sT < rows / 32)) return MXG_ERR_SHAPE;
  if (rows / 128 > 65535 || cols / 128 > 0x7FFFFFFF) return MXG_ERR_SHAPE;
  if (ld_w % 8 != 0 || ld_q % 16 != 0 || ld_s % 4 != 0) return MXG_ERR_ALIGN;
  if (qT != nullptr && (ld_qT % 16 != 0 || ld_sT % 4 != 0)) return MXG_ERR_ALIGN;
  if (rows == 0) return MXG_OK;
  if (w == nullptr || q == nullptr || s == nullptr) return MXG_ERR_NULL;
  if (!aligned16(w) || !aligned16(q) || !aligned16(qT) || !aligned(s, 4) || !aligned(sT, 4))
    return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({w, q, s, qT, sT}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_bw_weight(w, rows, cols, ld_w, q, ld_q, s, ld_s, qT, ld_qT, sT, ld_sT,
                                      true, static_cast<cudaStream_t>(stream), sms));
}

mxg_status bw_quantize_colwise_padded_pow2(const void* x, int64_t rows, int64_t cols,
                                           int64_t ld_x, const int32_t* d_m_splits, int32_t G,
                                           void* qT, int64_t ld_q, uint8_t* sT, int64_t ld_s,
                                           int64_t capacity, int64_t* d_pad_offsets,
                                           int32_t* d_status, void* stream) {
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (G < 1 || G > kMaxExperts) return MXG_ERR_SHAPE;
  if (rows < 0 || cols <= 0 || cols % 32 != 0 || capacity < 0 || capacity % 128 != 0)
    return MXG_ERR_SHAPE;
  if (ld_x < cols || ld_q < capacity || ld_s < capacity / 32) return MXG_ERR_SHAPE;
  if (ld_x % 8 != 0 || ld_q % 16 != 0 || ld_s % 4 != 0) return MXG_ERR_ALIGN;
  if ((rows > 0 && x == nullptr) || (capacity > 0 && (qT == nullptr || sT == nullptr)))
    return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned16(qT) || !aligned(sT, 4) || !aligned(d_pad_offsets, 8))
    return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, d_m_splits, qT, sT, d_pad_offsets, d_status}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_bw_colwise(x, rows, cols, ld_x, d_m_splits, G, qT, ld_q, sT, ld_s,
                                       capacity, d_pad_offsets, d_status, true,
                                       static_cast<cudaStream_t>(stream), sms));
}

}  // extern "C"

namespace {
// Shared checks and launch of the dual blockwise quantizers (row-wise 1x128
// and column-wise padded-to-128 from one read of x).
mxg_status bw_dual(const void* x, int64_t rows, int64_t cols, int64_t ld_x, const int32_t* d_m_splits,
                   int32_t G, void* q, int64_t ld_q, void* s, int64_t ld_s, void* qT, int64_t ld_qT, void* sT,
                   int64_t ld_sT, int64_t capacity, int64_t* d_pad_offsets, int32_t* d_status, bool pow2,
                   void* stream) {
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (G < 1 || G > kMaxExperts) return MXG_ERR_SHAPE;
  if (rows < 0 || cols <= 0 || cols % 128 != 0 || capacity < 0 || capacity % 128 != 0) return MXG_ERR_SHAPE;
  // row-wise scales: fp32 block-column-major (ld_s >= rows) or UE8M0 [rows, cols/32]
  if (ld_x < cols || ld_q < cols || ld_qT < capacity || ld_s < (pow2 ? cols / 32 : rows) ||
      ld_sT < (pow2 ? capacity / 32 : cols))
    return MXG_ERR_SHAPE;
  if (ld_x % 8 != 0 || ld_q % 8 != 0 || ld_qT % 16 != 0 || (pow2 && (ld_s % 4 != 0 || ld_sT % 4 != 0)))
    return MXG_ERR_ALIGN;
  if ((rows > 0 && (x == nullptr || q == nullptr || s == nullptr)) ||
      (capacity > 0 && (qT == nullptr || sT == nullptr)))
    return MXG_ERR_NULL;
  if (!aligned16(x) || !aligned(q, 8) || !aligned(s, 4) || !aligned16(qT) || !aligned(sT, 4) ||
      !aligned(d_pad_offsets, 8))
    return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  mxg_status st = check_device({x, d_m_splits, q, s, qT, sT, d_pad_offsets, d_status}, &dev, &sms);
  if (st != MXG_OK) return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return cuda_status(launch_bw_colwise(x, rows, cols, ld_x, d_m_splits, G, qT, ld_qT, sT, ld_sT, capacity,
                                       d_pad_offsets, d_status, pow2, static_cast<cudaStream_t>(stream), sms,
                                       rows > 0 ? q : nullptr, ld_q, s, ld_s));
}
}  // namespace

extern "C" {

mxg_status bw_quantize_dual_padded(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                   const int32_t* d_m_splits, int32_t G, void* q, int64_t ld_q, float* s,
                                   int64_t ld_s, void* qT, int64_t ld_qT, float* sT, int64_t ld_sT,
                                   int64_t capacity, int64_t* d_pad_offsets, int32_t* d_status, void* stream) {
  return bw_dual(x, rows, cols, ld_x, d_m_splits, G, q, ld_q, s, ld_s, qT, ld_qT, sT, ld_sT, capacity,
                 d_pad_offsets, d_status, false, stream);
}

mxg_status bw_quantize_dual_padded_pow2(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                        const int32_t* d_m_splits, int32_t G, void* q, int64_t ld_q,
                                        uint8_t* s, int64_t ld_s, void* qT, int64_t ld_qT, uint8_t* sT,
                                        int64_t ld_sT, int64_t capacity, int64_t* d_pad_offsets,
                                        int32_t* d_status, void* stream) {
  return bw_dual(x, rows, cols, ld_x, d_m_splits, G, q, ld_q, s, ld_s, qT, ld_qT, sT, ld_sT, capacity,
                 d_pad_offsets, d_status, true, stream);
}

size_t bw_gemm_workspace_size(int32_t G) {
  if (G < 1 || G > kMaxExperts) return 0;
  return bw_gemm_workspace_bytes(G);
}

mxg_status bw_grouped_gemm_fwd(const mxg_bw_operand* A, const mxg_bw_operand* W,
                               const int32_t* d_m_splits, int32_t G, int64_t N, void* out,
                               int64_t ld_out, int32_t out_dtype, void* ws, size_t ws_bytes,
                               int32_t* d_status, void* stream) {
  mxg_status st;
  if ((st = check_bw_operand(A)) != MXG_OK || (st = check_bw_operand(W)) != MXG_OK) return st;
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (G < 1 || G > kMaxExperts || N <= 0 || N % 128 != 0) return MXG_ERR_SHAPE;
  if ((st = check_out(out, A->rows, ld_out, N, out_dtype)) != MXG_OK) return st;
  if (A->cols != W->cols || W->rows != (int64_t)G * N) return MXG_ERR_SHAPE;
  if (A->scale_ld < A->rows || W->scale_ld < W->cols / 128) return MXG_ERR_SHAPE;
  if (ws_bytes < bw_gemm_workspace_bytes(G) || ws == nullptr) return MXG_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  if ((st = check_device({A->data, A->scale, W->data, W->scale, d_m_splits, out, ws, d_status},
                         &dev, &sms)) != MXG_OK)
    return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return launch_grouped_bw_gemm(bw_args(MXG_PASS_FWD, G, A, W, d_m_splits, A->rows, N, A->cols,
                                        out, ld_out, out_dtype, 0, ws, d_status),
                                static_cast<cudaStream_t>(stream), sms);
}

mxg_status bw_grouped_gemm_dgrad(const mxg_bw_operand* dY, const mxg_bw_operand* Wt,
                                 const int32_t* d_m_splits, int32_t G, void* out, int64_t ld_out,
                                 int32_t out_dtype, void* ws, size_t ws_bytes, int32_t* d_status,
                                 void* stream) {
  mxg_status st;
  if ((st = check_bw_operand(dY)) != MXG_OK || (st = check_bw_operand(Wt)) != MXG_OK) return st;
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (G < 1 || G > kMaxExperts) return MXG_ERR_SHAPE;
  const int64_t N = dY->cols, K = Wt->rows;
  if (K <= 0 || K % 128 != 0 || Wt->cols != (int64_t)G * N) return MXG_ERR_SHAPE;
  if ((st = check_out(out, dY->rows, ld_out, K, out_dtype)) != MXG_OK) return st;
  if (dY->scale_ld < dY->rows || Wt->scale_ld < Wt->cols / 128) return MXG_ERR_SHAPE;
  if (ws_bytes < bw_gemm_workspace_bytes(G) || ws == nullptr) return MXG_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  if ((st = check_device({dY->data, dY->scale, Wt->data, Wt->scale, d_m_splits, out, ws, d_status},
                         &dev, &sms)) != MXG_OK)
    return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return launch_grouped_bw_gemm(bw_args(MXG_PASS_DGRAD, G, dY, Wt, d_m_splits, dY->rows, N, K,
                                        out, ld_out, out_dtype, 0, ws, d_status),
                                static_cast<cudaStream_t>(stream), sms);
}

mxg_status bw_grouped_gemm_wgrad(const mxg_bw_operand* dYt, const mxg_bw_operand* Xt,
                                 const int32_t* d_m_splits, int32_t G, int64_t total_rows,
                                 void* out, int32_t out_dtype, int32_t accumulate, void* ws,
                                 size_t ws_bytes, int32_t* d_status, void* stream) {
  mxg_status st;
  if ((st = check_bw_operand(dYt, true)) != MXG_OK || (st = check_bw_operand(Xt, true)) != MXG_OK)
    return st;
  if (d_m_splits == nullptr || d_status == nullptr) return MXG_ERR_NULL;
  if (G < 1 || G > kMaxExperts || total_rows < 0) return MXG_ERR_SHAPE;
  const int64_t N = dYt->rows, K = Xt->rows;
  if (N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0 || dYt->cols != Xt->cols) return MXG_ERR_SHAPE;
  if ((st = check_out(out, 1, K, K, out_dtype)) != MXG_OK) return st;
  if (accumulate && out_dtype != MXG_OUT_F32) return MXG_ERR_UNSUPPORTED;
  if (dYt->scale_ld < N || Xt->scale_ld < K) return MXG_ERR_SHAPE;
  if (Xt->cols > 0 && (!aligned16(Xt->scale) || Xt->scale_ld % 4 != 0)) return MXG_ERR_ALIGN;
  if (ws_bytes < bw_gemm_workspace_bytes(G) || ws == nullptr) return MXG_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return MXG_ERR_ALIGN;
  int dev = 0, sms = 0;
  if ((st = check_device({dYt->data, dYt->scale, Xt->data, Xt->scale, d_m_splits, out, ws,
                          d_status},
                         &dev, &sms)) != MXG_OK)
    return st;
  DeviceGuard g(dev);
  if (!g.ok) return MXG_ERR_CUDA;
  return launch_grouped_bw_gemm(bw_args(MXG_PASS_WGRAD, G, dYt, Xt, d_m_splits, total_rows, N, K,
                                        out, K, out_dtype, accumulate ? 1 : 0, ws, d_status),
                                static_cast<cudaStream_t>(stream), sms);
}

}  // extern "C"
