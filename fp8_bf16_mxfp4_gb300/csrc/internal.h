// Internal launcher declarations shared between the C-ABI layer and kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "mxg.h"

namespace mxg {

uint64_t wait_timeout_ns();
int gemm_cta_group();  // 2: MX and blockwise GEMMs on CTA pairs where possible; 1: one-SM kernels

cudaError_t launch_mx_rowwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int elem,
                              void* q, int64_t ld_q, uint8_t* s, int64_t ld_s,
                              cudaStream_t stream, int num_sms);

cudaError_t launch_mx_rowwise_packed(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int elem,
                                     void* q, int64_t ld_q, uint8_t* sp, const int32_t* splits, int G,
                                     int64_t seg_rows, int64_t rt_bound, int32_t* status,
                                     cudaStream_t stream, int num_sms);

cudaError_t launch_mx_colwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                              const int32_t* splits, int G, int pad, int elem, void* qT,
                              int64_t ld_q, uint8_t* sT, int64_t ld_s, int64_t capacity,
                              int64_t* pad_offsets, int32_t* status, cudaStream_t stream,
                              int num_sms, void* q_row = nullptr, int64_t ld_qr = 0,
                              uint8_t* s_row = nullptr, int64_t ld_sr = 0, int64_t packed_bytes = 0);

cudaError_t launch_bw_rowwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x, void* q,
                              int64_t ld_q, void* s, int64_t ld_s, bool pow2, cudaStream_t stream,
                              int num_sms);
cudaError_t launch_bw_weight(const void* w, int64_t rows, int64_t K, int64_t ld_w, void* q,
                             int64_t ld_q, void* s, int64_t ld_s, void* qT, int64_t ld_qT, void* sT,
                             int64_t ld_sT, bool pow2, cudaStream_t stream, int num_sms);
cudaError_t launch_bw_colwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                              const int32_t* splits, int G, void* qT, int64_t ld_q, void* sT,
                              int64_t ld_s, int64_t capacity, int64_t* pad_offsets,
                              int32_t* status, bool pow2, cudaStream_t stream, int num_sms,
                              void* q_row = nullptr, int64_t ld_qr = 0, void* s_row = nullptr,
                              int64_t ld_sr = 0);

// Grouped MX GEMM (tcgen05 block-scaled).  See gemm_mx.cu.
struct GemmArgs {
  int pass;  // mxg_pass
  int G;
  // operand A (M side) and B (N side): codes, row stride (bytes), plain scales
  const uint8_t* a_data;
  int64_t a_ld;
  const uint8_t* a_scale;
  int64_t a_scale_ld;
  int64_t a_rows, a_cols;
  int a_elem;
  const uint8_t* b_data;
  int64_t b_ld;
  const uint8_t* b_scale;
  int64_t b_scale_ld;
  int64_t b_rows, b_cols;
  int b_elem;
  bool a_packed, b_packed;  // scales already in the GEMM's staging order
  const int32_t* splits;
  int64_t total_rows;  // S
  int64_t N, K;        // fwd: out [S,N] over K; dgrad: out [S,K] over N; wgrad: out [G,N,K]
  int pad;             // wgrad pad multiple
  void* out;
  int64_t ld_out;
  int out_dtype;
  int accumulate;
  void* ws;
  size_t ws_bytes;
  int32_t* status;
};

size_t gemm_workspace_bytes(int pass, int G, int64_t S, int64_t N, int64_t K, int pad);
// Host checks of the forward entry points that precede the workspace check
// (operands, status word, output, G, N, shapes, formats), in their order.
mxg_status fwd_host_checks(const mxg_mx_operand* A, const mxg_mx_operand* W, int32_t G, int64_t N,
                           const void* out, int64_t ld_out, int32_t out_dtype, const int32_t* d_status);
mxg_status launch_grouped_gemm(const GemmArgs& a, cudaStream_t stream, int num_sms);

// Grouped blockwise-FP8 GEMM.  See gemm_bw.cu.
struct BwGemmArgs {
  int pass;
  int G;
  const uint8_t* a_data;
  int64_t a_ld;
  const float* a_scale;  // activation-type: (row, kb) at a_scale[kb * a_scale_ld + row]
  int64_t a_scale_ld;
  int64_t a_rows, a_cols;
  const uint8_t* b_data;
  int64_t b_ld;
  const float* b_scale;  // fwd/dgrad: 128x128 at [rb * ld + kb]; wgrad: activation-type
  int64_t b_scale_ld;
  int64_t b_rows, b_cols;
  const int32_t* splits;
  int64_t total_rows;
  int64_t N, K;
  void* out;
  int64_t ld_out;
  int out_dtype;
  int accumulate;
  void* ws;
  int32_t* status;
};

size_t bw_gemm_workspace_bytes(int G);
mxg_status launch_grouped_bw_gemm(const BwGemmArgs& a, cudaStream_t stream, int num_sms);

}  // namespace mxg
