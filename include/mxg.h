/*
 * mxg.h -- C ABI of the GB300 grouped microscaled GEMM library (libmxg.so).
 *
 * The library computes the hot path of a mixture-of-experts linear layer whose
 * operands use OCP microscaling (MX) formats: BF16 -> MXFP4 (E2M1) / MXFP8
 * (E4M3) quantization with one UE8M0 scale per 32 elements, and the
 * single-launch grouped GEMMs over experts whose row counts (m_splits) live in
 * device memory:
 *
 *   forward (TN)  Y[off_g+i, n]  = sum_k A[off_g+i, k] * W[g*N+n, k]
 *   dgrad   (NN)  dX[off_g+i, k] = sum_n dY[off_g+i, n] * Wt[k, g*N+n]
 *   wgrad   (NT)  dW[g, n, k]   (+)= sum over expert g's padded token segment
 *                                   of dYt[n, j] * Xt[k, j]
 *
 * Sources: "Triton mxfp4 (and a8w4) grouped GEMM kernel" (ROCm
 * TransformerEngine PR #723: the three passes, the split checks, the
 * segment-padded column-wise wgrad operand); PR #745 (the a8w4 mix, fwd only,
 * and the -127 scale-exponent clamp); "Add ROCm Triton blockwise FP8 grouped
 * GEMM" (PR #716: 1x128 / 128x128 blockwise FP8); "Integrate MXFP4 hipblaslt
 * GEMM support" (PR #697: per-pass shapes).  off_g is the exclusive prefix sum
 * of m_splits.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All data pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing, keeps no state between calls (except the wait timeout
 *    and the GEMM CTA-group choice below) and enqueues work on `stream` only,
 *    without synchronising, except
 *    mxg_check_status.  `stream` is a cudaStream_t passed as void* (NULL = the
 *    legacy default stream).
 *  - Matrices are row-major.  Strides (`ld*`) are in BYTES for quantized codes
 *    and scale bytes, and in ELEMENTS for BF16 / FP32 buffers, as stated per
 *    argument.  The quantized code layouts are: E4M3 one byte per element;
 *    E2M1 two per byte, element 2j in the low nibble.  UE8M0 scale byte b
 *    encodes 2^(b-127).
 *  - Host checks run first and do not touch the GPU: null pointers, sizes,
 *    divisibility, 16-byte alignment of pointers and strides, 1 <= G <= 512.
 *    Then the pointers' device and the device architecture (sm_103) are
 *    checked.  A failing check returns its code and enqueues nothing.
 *  - Checks that need device data (m_splits >= 0, sum(m_splits) == rows,
 *    padded rows within capacity) run inside the kernels: the first failure is
 *    written to *d_status (an int32 in device memory, initialised to 0 by the
 *    caller) with an atomic compare-and-swap, and the kernels then write no
 *    output.  mxg_check_status reads and clears it.
 *  - Every in-kernel wait is bounded by a time limit (mxg_set_wait_timeout_ns);
 *    a wait that runs out records MXG_ERR_TIMEOUT in *d_status and the kernel
 *    returns instead of hanging.
 */
#ifndef MXG_H_
#define MXG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mxg_status {
  MXG_OK = 0,
  MXG_ERR_NULL = 1,        /* a required pointer is NULL */
  MXG_ERR_SHAPE = 2,       /* sizes inconsistent or not divisible as required */
  MXG_ERR_ALIGN = 3,       /* pointer or stride not 16-byte aligned */
  MXG_ERR_SPLITS = 4,      /* device-side: negative split or sum != rows */
  MXG_ERR_UNSUPPORTED = 5, /* format combination / option not provided */
  MXG_ERR_DEVICE = 6,      /* pointer not device memory, mixed devices, or not sm_103 */
  MXG_ERR_CUDA = 7,        /* a CUDA runtime call failed */
  MXG_ERR_TIMEOUT = 8,     /* device-side: a bounded wait ran out */
  MXG_ERR_WORKSPACE = 9,   /* workspace missing or smaller than required */
  MXG_ERR_CAPACITY = 10    /* device-side: padded rows exceed the output capacity */
} mxg_status;

typedef enum mxg_elem { MXG_E2M1 = 1, MXG_E4M3 = 2 } mxg_elem;
/* Scale-rule flag, OR'ed into the elem argument of the MX quantizers
 * (mx_quantize_rowwise, _rowwise_packed, _colwise_segment_padded,
 * _dual_segment_padded).  Without it the shared exponent follows the OCP MX
 * rule, e = floor(log2 amax) - emax.  With it, the TransformerEngine recipe
 * described in the review "Clamp tiny block scales to preserve nonzero values"
 * (ROCm TransformerEngine PR #745): e is the smallest integer with
 * maxval * 2^e >= amax (maxval 448 for E4M3, 6 for E2M1), so no element
 * saturates.  Both clamp e to [-127, 127] and give an all-zero block e = -127.
 * Quantized operands carry no trace of the rule: GEMM operands take the plain
 * MXG_E2M1 / MXG_E4M3. */
#define MXG_SCALE_ROUND_UP 0x100
typedef enum mxg_out_dtype { MXG_OUT_BF16 = 1, MXG_OUT_F32 = 2 } mxg_out_dtype;
typedef enum mxg_pass { MXG_PASS_FWD = 0, MXG_PASS_DGRAD = 1, MXG_PASS_WGRAD = 2 } mxg_pass;
/* Where an MX operand's scales are: row-major [rows, cols/32] bytes, or the
 * packed tensor-core staging order written by mx_quantize_rowwise_packed. */
typedef enum mxg_scale_layout { MXG_SCALE_PLAIN = 0, MXG_SCALE_PACKED = 1 } mxg_scale_layout;

/* One MX operand of a grouped GEMM, K-major: `rows` rows of `cols` elements,
 * quantized along `cols` (the contraction dimension).
 *   data         : codes, row r at (uint8*)data + r*ld  (ld >= cols or cols/2 bytes)
 *   scale        : MXG_SCALE_PLAIN: UE8M0 bytes, row r at scale + r*scale_ld,
 *                  entries [0, cols/32);
 *                  MXG_SCALE_PACKED: the tensor-core staging order (16-byte
 *                  aligned; scale_ld is ignored), cut into the same segments
 *                  as the call's experts -- from mx_quantize_rowwise_packed for
 *                  row-segmented operands (forward activations and dgrad
 *                  gradient: the m_splits; forward weights: G segments of N
 *                  rows) and from mx_quantize_colwise_segment_padded_packed for
 *                  k-segmented ones (dgrad weights: G segments of N, pad 32;
 *                  wgrad operands: the m_splits and the call's pad).
 *   elem         : MXG_E2M1 or MXG_E4M3
 *   scale_layout : mxg_scale_layout
 * Requirements: cols % 32 == 0; data 16-byte aligned (32 for E2M1 weights of
 * the a8w4 forward); ld % 16 == 0 (32 for those weights). */
typedef struct mxg_mx_operand {
  const void* data;
  const uint8_t* scale;
  int64_t rows;
  int64_t cols;
  int64_t ld;
  int64_t scale_ld;
  int32_t elem;
  int32_t scale_layout;
} mxg_mx_operand;

/* --------------------------------------------------------------------------
 * MX quantization
 * ------------------------------------------------------------------------ */

/* Row-wise MX quantization (PR #723 `_row_operand`; PR #745 MXFP8 E4M3
 * reference quantizer).  For each row and each block of 32 consecutive BF16
 * values: e = clamp(floor(log2(amax)) - emax, -127, 127) (emax 2 for E2M1,
 * 8 for E4M3; e = -127 for an all-zero block); scale byte = e + 127; element =
 * x * 2^-e rounded to nearest, ties to even, saturating (6 / 448), sign kept.
 *   x      : BF16 [rows, cols], row stride ld_x elements (ld_x % 8 == 0)
 *   q      : codes [rows, cols/2] (E2M1) or [rows, cols] (E4M3), stride ld_q bytes;
 *            q 16-byte aligned and ld_q % 16 == 0 (MXG_ERR_ALIGN otherwise)
 *   s      : scale bytes [rows, cols/32], stride ld_s bytes
 * cols % 32 == 0; rows may be 0 (no launch).  Writes only q and s. */
mxg_status mx_quantize_rowwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                               int32_t elem, void* q, int64_t ld_q, uint8_t* s, int64_t ld_s,
                               void* stream);

/* Bytes of the packed scales of a row-wise MX operand of `rows` x `cols`
 * whose rows are cut into G segments: KC * RTmax * 512, KC = ceil(cols/128),
 * RTmax = floor((rows + min(rows, G) * 127) / 128) -- at least the row tiles
 * of every split of `rows` into G segments.  -1 on invalid input. */
int64_t mx_packed_scale_bytes(int64_t rows, int64_t cols, int32_t G);

/* Row-wise MX quantization (the rule of mx_quantize_rowwise, codes laid out
 * the same way) with the scales written in the tensor-core staging order, so
 * that a grouped GEMM reads them without a repacking pass ("Integrate MXFP4
 * hipblaslt GEMM support", Takeaways: pre-swizzled scales; "Grouped MXFP8
 * GEMMs with HipKittens" PR #661, "fused scale packing kernel").  The rows are cut into segments -- the device
 * d_m_splits (int32[G]; activations and gradients), or, when d_m_splits is
 * NULL, G equal segments of rows/G rows (forward weights, rows % G == 0) --
 * and each segment into tiles of 128 rows, numbered across segments (RT in
 * all).  The scales of a tile's 128 rows and 4 consecutive blocks form one
 * 512-byte chunk; chunk (kc, rt) starts at byte (kc * RT + rt) * 512, and the
 * scale of the tile's row i, block 4*kc + j sits at (i % 32) * 16 + (i / 32) * 4
 * + j in it.  Bytes with no row or block (segment tails, blocks past cols/32)
 * are written as 0.
 *   s_packed : device, 16-byte aligned, s_bytes >= mx_packed_scale_bytes(rows, cols, G)
 *   d_status : required with d_m_splits; a negative split or a sum != rows
 *              sets MXG_ERR_SPLITS and nothing is written.
 * Other arguments and checks as mx_quantize_rowwise. */
mxg_status mx_quantize_rowwise_packed(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                      int32_t elem, void* q, int64_t ld_q, uint8_t* s_packed,
                                      int64_t s_bytes, const int32_t* d_m_splits, int32_t G,
                                      int32_t* d_status, void* stream);

/* Column-wise, segment-padded MX quantization: the wgrad operand of PR #723
 * (`_col_operand_grouped_padded`).  x is BF16 [rows, cols] with the experts'
 * rows concatenated in order.  Expert g's rows [off_g, off_g+m_g) are
 * transposed and written to output columns [poff_g, poff_g + m_g), followed by
 * zero columns up to p_g = ceil(m_g/pad)*pad; 32-blocks start at poff_g, so no
 * block straddles two experts.  poff is the exclusive prefix sum of p_g.
 *   d_m_splits   : int32[G] device
 *   pad_multiple : positive multiple of 32
 *   qT           : codes [cols, capacity(/2)], row stride ld_q bytes
 *   sT           : scale bytes [cols, capacity/32], row stride ld_s bytes
 *   capacity     : columns available in qT (e.g. mx_padded_rows_capacity)
 *   d_pad_offsets: int64[G+1] device, receives poff (may be NULL)
 * Columns beyond poff_G are left untouched.  Device errors: MXG_ERR_SPLITS,
 * MXG_ERR_CAPACITY (poff_G > capacity). */
mxg_status mx_quantize_colwise_segment_padded(const void* x, int64_t rows, int64_t cols,
                                              int64_t ld_x, const int32_t* d_m_splits,
                                              int32_t G, int32_t pad_multiple, int32_t elem,
                                              void* qT, int64_t ld_q, uint8_t* sT, int64_t ld_s,
                                              int64_t capacity, int64_t* d_pad_offsets,
                                              int32_t* d_status, void* stream);

/* Bytes of the packed scales of a column-wise operand of `cols` rows
 * (channels) and `capacity` padded positions over G experts:
 * (capacity / 128 + G) * ceil(cols / 128) * 512 -- at least the k-chunks of
 * every split.  -1 on invalid input. */
int64_t mx_packed_colwise_scale_bytes(int64_t cols, int64_t capacity, int32_t G);

/* mx_quantize_colwise_segment_padded with the scales written in the
 * tensor-core staging order of a k-segmented operand (the dgrad weights, both
 * wgrad operands): the chunk grid restarts at every expert's padded start,
 * expert g's k-chunks being (sum over h < g of ceil(p_h / 128)) + c; chunk
 * (kc, rt) at (kc * RT + rt) * 512 with RT = ceil(cols / 128); channel i of
 * the row tile and block j of the chunk at (i % 32) * 16 + (i / 32) * 4 + j.
 * The first mx_packed_colwise_scale_bytes(cols, capacity, G) bytes of
 * s_packed (16-byte aligned, s_bytes at least that) are zeroed first, so
 * every byte without a channel or block reads as scale 2^-127 (also when the
 * splits turn out invalid; the codes are then left untouched).  Other
 * arguments, checks and device errors as mx_quantize_colwise_segment_padded. */
mxg_status mx_quantize_colwise_segment_padded_packed(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                                     const int32_t* d_m_splits, int32_t G, int32_t pad_multiple,
                                                     int32_t elem, void* qT, int64_t ld_q, uint8_t* s_packed,
                                                     int64_t s_bytes, int64_t capacity, int64_t* d_pad_offsets,
                                                     int32_t* d_status, void* stream);

/* Fused dual MX quantization: one read of x yields both operands of a
 * training step -- the row-wise operand (fwd / dgrad) and the column-wise
 * segment-padded operand (wgrad) -- as the dual activation quantizer of "Add
 * ROCm Triton blockwise FP8 grouped GEMM" (PR #716,
 * `quantize_fp8_blockwise_act_operands`) does for blockwise FP8.  The bytes
 * are identical to mx_quantize_rowwise(x) -> (q, s) followed by
 * mx_quantize_colwise_segment_padded(x, ...) -> (qT, sT, d_pad_offsets).
 *   q, ld_q, s, ld_s      : as in mx_quantize_rowwise (q 16-byte aligned,
 *                           ld_q % 16 == 0)
 *   qT, ld_qT, sT, ld_sT  : as qT, ld_q, sT, ld_s of the column-wise call
 *   other arguments       : as in mx_quantize_colwise_segment_padded
 * Host errors as for the two calls; device errors as for the column-wise call
 * (MXG_ERR_SPLITS, MXG_ERR_CAPACITY), in which case neither operand is
 * written. */
mxg_status mx_quantize_dual_segment_padded(const void* x, int64_t rows, int64_t cols,
                                           int64_t ld_x, const int32_t* d_m_splits, int32_t G,
                                           int32_t pad_multiple, int32_t elem, void* q,
                                           int64_t ld_q, uint8_t* s, int64_t ld_s, void* qT,
                                           int64_t ld_qT, uint8_t* sT, int64_t ld_sT,
                                           int64_t capacity, int64_t* d_pad_offsets,
                                           int32_t* d_status, void* stream);

/* Upper bound of sum_g ceil(m_g/pad)*pad over all splits of `rows` into G
 * experts: floor((rows + k*(pad-1)) / pad) * pad with k = min(G, rows), the
 * most experts that can be non-empty.  -1 on invalid input. */
int64_t mx_padded_rows_capacity(int64_t rows, int32_t G, int32_t pad);

/* --------------------------------------------------------------------------
 * Grouped MX GEMMs (single launch over all experts; tcgen05 block-scaled MMA)
 *
 * Supported element pairs: E2M1 x E2M1 (MXFP4, all passes), E4M3 x E2M1
 * (a8w4: A = MXFP8 activations, W = MXFP4 weights; forward only, K % 128 == 0)
 * and E4M3 x E4M3 (MXFP8, all passes).  Products are exact; accumulation is in
 * fp32; the output is rounded to BF16 (nearest even) or stored as FP32.
 * Only each expert's valid rows/columns are written.
 *
 * ws / ws_bytes: device scratch of at least mxg_gemm_workspace_size(...)
 * bytes, 256-byte aligned; the UE8M0 scales are re-laid out there into the
 * tensor-core staging order before the GEMM kernel runs.
 * ------------------------------------------------------------------------ */

/* Forward (TN).  A: rows = S (sum of m_splits), cols = K.  W: rows = G*N,
 * cols = K (expert g's weight is rows [g*N, g*N+N)).  out: [S, N] with row
 * stride ld_out elements; out is 32-byte aligned and ld_out * element size is
 * a multiple of 32 bytes (the same holds for every GEMM output below).
 * N % 32 == 0. */
mxg_status grouped_gemm_fwd(const mxg_mx_operand* A, const mxg_mx_operand* W,
                            const int32_t* d_m_splits, int32_t G, int64_t N, void* out,
                            int64_t ld_out, int32_t out_dtype, void* ws, size_t ws_bytes,
                            int32_t* d_status, void* stream);

/* Dense (non-grouped) MX GEMM, C[M, N] = A[M, K] * B[N, K]^T with both
 * operands K-major: the dense hipBLASLt MXFP4 GEMM of "Integrate MXFP4
 * hipblaslt GEMM support" (PR #697; its forward TN, dgrad NN and wgrad NT are
 * this call on operands quantized along the respective contraction).  It is
 * grouped_gemm_fwd with one expert of all A->rows rows, and needs no device
 * m_splits.  Operand pairs, output, workspace (mxg_gemm_workspace_size(
 * MXG_PASS_FWD, 1, M, N, K, 32)) and packed scales (one segment) as for
 * grouped_gemm_fwd; d_status receives device-side errors (a wait timeout). */
mxg_status mx_gemm_dense(const mxg_mx_operand* A, const mxg_mx_operand* B, void* out, int64_t ld_out,
                         int32_t out_dtype, void* ws, size_t ws_bytes, int32_t* d_status, void* stream);

/* dgrad (NN).  dY: rows = S, cols = N.  Wt: rows = K, cols = G*N -- W
 * transposed and quantized along N within each expert (mx_quantize_colwise_
 * segment_padded of W [G*N, K] with m_splits = {N, ..., N}, pad 32).
 * out: [S, K], row stride ld_out elements.  K % 32 == 0, N % 32 == 0. */
mxg_status grouped_gemm_dgrad(const mxg_mx_operand* dY, const mxg_mx_operand* Wt,
                              const int32_t* d_m_splits, int32_t G, void* out, int64_t ld_out,
                              int32_t out_dtype, void* ws, size_t ws_bytes, int32_t* d_status,
                              void* stream);

/* wgrad (NT, variable K per expert).  dYt: rows = N, Xt: rows = K, both
 * column-wise segment-padded operands (mx_quantize_colwise_segment_padded with
 * the same m_splits and pad_multiple); cols = their capacity.  The padded
 * offsets are recomputed from d_m_splits and pad_multiple.  total_rows = S
 * (validated against sum(m_splits)).  out: [G, N, K] contiguous; with
 * accumulate != 0 (FP32 only) the result is added in place (fp32 main_grad),
 * otherwise stored.  An empty expert stores zeros (or leaves out unchanged
 * when accumulating). */
mxg_status grouped_gemm_wgrad(const mxg_mx_operand* dYt, const mxg_mx_operand* Xt,
                              const int32_t* d_m_splits, int32_t G, int64_t total_rows,
                              int32_t pad_multiple, void* out, int32_t out_dtype,
                              int32_t accumulate, void* ws, size_t ws_bytes, int32_t* d_status,
                              void* stream);

/* grouped_gemm_fwd for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for code that must not
 * call cudaMalloc at GEMM time -- an inference-engine plugin whose device
 * memory is budgeted and handed out by its host framework, or a
 * latency-critical path that never enters an allocator (an allocation can
 * synchronise the device or wait on the allocator's lock).
 *
 * Same arguments and results as grouped_gemm_fwd minus the workspace: the
 * scratch is a file-scope device array of 32 MiB (33554432 bytes) inside
 * libmxg.so, held on every GPU that loads the library until the process exits.
 * The argument checks of grouped_gemm_fwd run first, in its order; then a
 * problem whose workspace (mxg_gemm_workspace_size(MXG_PASS_FWD, ...))
 * exceeds 32 MiB is rejected with MXG_ERR_WORKSPACE, before anything is
 * enqueued.  Nothing is allocated: no cudaMalloc / cudaFree and no allocating
 * library routine.
 *   - The first call on a device looks up the array's device address (with
 *     that device made current) and keeps it for the life of the process;
 *     make that first call before any stream capture begins.  Do not use this
 *     entry point after a cudaDeviceReset in the same process: the kept
 *     address is not looked up again.
 *   - Every call shares the one array; each call fully rewrites the parts it
 *     reads, so nothing has to be cleared between calls, but calls that may
 *     overlap on the GPU (different streams without ordering) race on it and
 *     must be serialised by the caller. */
mxg_status grouped_gemm_fwd_noalloc(const mxg_mx_operand* A, const mxg_mx_operand* W,
                                    const int32_t* d_m_splits, int32_t G, int64_t N, void* out,
                                    int64_t ld_out, int32_t out_dtype, int32_t* d_status,
                                    void* stream);

/* Scratch bytes needed by a grouped MX GEMM pass (an upper bound valid for
 * every split of S rows into G experts).  For MXG_PASS_FWD and DGRAD the
 * arguments are (G, S, N, K); for MXG_PASS_WGRAD, S is the operands' column
 * capacity.  Returns 0 on invalid input. */
size_t mxg_gemm_workspace_size(int32_t pass, int32_t G, int64_t S, int64_t N, int64_t K,
                               int32_t pad_multiple);

/* --------------------------------------------------------------------------
 * Blockwise FP8 (DeepSeek-style; "Add ROCm Triton blockwise FP8 grouped GEMM",
 * ROCm TransformerEngine PR #716)
 *
 * Per block: a = max(amax, 1e-4), s = a / 448 (fp32, correctly rounded), and
 * each element q = x / s (fp32, correctly rounded) rounded to E4M3 (nearest,
 * ties to even, saturating at 448).  s is the dequantization scale: x ~= q*s.
 * Blocks are 1x128 along the contraction for activations / gradients and for
 * the column-wise wgrad operands, and 128x128 for weights.  All sizes that
 * are block dimensions must be multiples of 128.
 *
 * Scale layouts:
 *   activation-type (1x128): block-column-major, (row r, block kb) at
 *                            s[kb * ld_s + r], ld_s >= rows;
 *   weight-type (128x128):   row-major [rows/128, cols/128], (rb, kb) at
 *                            s[rb * ld_s + kb].
 * ------------------------------------------------------------------------ */

/* A blockwise-FP8 operand, K-major: E4M3 codes [rows, cols] (row r at
 * (uint8*)data + r*ld, ld % 16 == 0) and fp32 scales in the layout the call
 * states (stride scale_ld floats). */
typedef struct mxg_bw_operand {
  const void* data;
  const float* scale;
  int64_t rows;
  int64_t cols;
  int64_t ld;
  int64_t scale_ld;
  int32_t reserved0; /* must be 0 */
  int32_t reserved1; /* must be 0 */
} mxg_bw_operand;

/* 1x128 row-wise quantization of BF16 x [rows, cols] (ld_x elements, % 8):
 * codes q [rows, cols] (ld_q bytes, % 8), activation-type scales s
 * (ld_s >= rows floats).  cols % 128 == 0. */
mxg_status bw_quantize_1x128(const void* x, int64_t rows, int64_t cols, int64_t ld_x, void* q,
                             int64_t ld_q, float* s, int64_t ld_s, void* stream);

/* 128x128 quantization of BF16 weights w [rows, cols] (rows = G*N stacked
 * experts; ld_w elements): codes q [rows, cols] (ld_q bytes), weight-type
 * scales s [rows/128, cols/128] (contiguous).  When qT and sT are given, also
 * writes the dgrad copy: the same blocks transposed, codes qT [cols, rows]
 * (ld_qT bytes) and scales sT [cols/128, rows/128] (contiguous).  rows and
 * cols multiples of 128; qT and sT both NULL or both set. */
mxg_status bw_quantize_128x128(const void* w, int64_t rows, int64_t cols, int64_t ld_w, void* q,
                               int64_t ld_q, float* s, void* qT, int64_t ld_qT, float* sT,
                               void* stream);

/* Column-wise 1x128 quantization along tokens, each expert's segment padded
 * to a multiple of 128 (the variable-K wgrad operand).  x BF16 [rows, cols]
 * with experts concatenated; codes qT [cols, capacity] (ld_q bytes, % 16),
 * activation-type scales sT of the transposed operand: (column c, token
 * block jb) at sT[jb * ld_s + c], ld_s >= cols.  Columns past the last
 * expert's padded end are left untouched.  Device errors as for
 * mx_quantize_colwise_segment_padded. */
mxg_status bw_quantize_colwise_padded(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                      const int32_t* d_m_splits, int32_t G, void* qT,
                                      int64_t ld_q, float* sT, int64_t ld_s, int64_t capacity,
                                      int64_t* d_pad_offsets, int32_t* d_status, void* stream);

/* Blockwise FP8 with power-of-two scales (the `pow2` option of the PR #716
 * quantizers; TE's `power_2_scale` default of its blockwise recipe): for each
 * block, a = max(amax, 1e-4) and s = 2^k, the smallest power of two with
 * 448 * s >= a; codes q = RNE_satfinite_E4M3(x * 2^-k) (exact scaling).  A
 * power-of-two scale is a UE8M0 byte (k + 127), so these quantizers write MX
 * operands: E4M3 codes plus UE8M0 bytes per 32-block, each 128-block's byte
 * repeated over its four 32-blocks.  The results feed grouped_gemm_fwd /
 * _dgrad / _wgrad directly (MXFP8 x MXFP8, elem MXG_E4M3), which compute the
 * same products as the blockwise promotion without it.
 *   1x128:   x [rows, cols] -> q [rows, cols] (ld_q % 8), s [rows, cols/32]
 *            (ld_s % 4, s 4-byte aligned); cols % 128 == 0.
 *   128x128: w [rows, cols] -> q [rows, cols], s [rows, cols/32] and, when
 *            qT != NULL, the dgrad copy qT [cols, rows] (ld_qT % 16), sT
 *            [cols, rows/32]; rows, cols % 128 == 0; ld_q % 16, ld_s % 4.
 *   colwise: as bw_quantize_colwise_padded (segments padded to 128) with
 *            sT [cols, capacity/32] UE8M0 (ld_s % 4). */
mxg_status bw_quantize_1x128_pow2(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                  void* q, int64_t ld_q, uint8_t* s, int64_t ld_s, void* stream);
mxg_status bw_quantize_128x128_pow2(const void* w, int64_t rows, int64_t cols, int64_t ld_w,
                                    void* q, int64_t ld_q, uint8_t* s, int64_t ld_s, void* qT,
                                    int64_t ld_qT, uint8_t* sT, int64_t ld_sT, void* stream);
mxg_status bw_quantize_colwise_padded_pow2(const void* x, int64_t rows, int64_t cols,
                                           int64_t ld_x, const int32_t* d_m_splits, int32_t G,
                                           void* qT, int64_t ld_q, uint8_t* sT, int64_t ld_s,
                                           int64_t capacity, int64_t* d_pad_offsets,
                                           int32_t* d_status, void* stream);

/* Dual blockwise quantization: one read of x [rows, cols] (experts' rows
 * concatenated) writes both activation operands of a training step -- the
 * 1x128 row-wise one (as bw_quantize_1x128 / _pow2) and the column-wise one
 * with every expert's segment padded to 128 (as bw_quantize_colwise_padded /
 * _pow2) -- the fused dual quantizer of "Add ROCm Triton blockwise FP8 grouped
 * GEMM" (PR #716).  Bytes and scales equal those of the two separate calls.
 *   q, ld_q (% 8), s, ld_s : row-wise codes [rows, cols] and scales (fp32
 *                            block-column-major with ld_s >= rows, or UE8M0
 *                            [rows, cols/32] with ld_s % 4 == 0)
 *   qT, ld_qT (% 16), sT, ld_sT : column-wise codes [cols, capacity] and scales
 *                            (fp32 (c, jb) at sT[jb * ld_sT + c], ld_sT >= cols;
 *                            or UE8M0 [cols, capacity/32], ld_sT % 4 == 0)
 * cols % 128 == 0, capacity % 128 == 0.  Device errors as for
 * mx_quantize_colwise_segment_padded; on an error nothing is written. */
mxg_status bw_quantize_dual_padded(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                   const int32_t* d_m_splits, int32_t G, void* q, int64_t ld_q, float* s,
                                   int64_t ld_s, void* qT, int64_t ld_qT, float* sT, int64_t ld_sT,
                                   int64_t capacity, int64_t* d_pad_offsets, int32_t* d_status, void* stream);
mxg_status bw_quantize_dual_padded_pow2(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                                        const int32_t* d_m_splits, int32_t G, void* q, int64_t ld_q,
                                        uint8_t* s, int64_t ld_s, void* qT, int64_t ld_qT, uint8_t* sT,
                                        int64_t ld_sT, int64_t capacity, int64_t* d_pad_offsets,
                                        int32_t* d_status, void* stream);

/* Grouped blockwise-FP8 GEMMs (tcgen05 kind::f8f6f4 + per-128-K promotion in
 * fp32).  Same passes, split validation and output conventions as the MX
 * GEMMs; N and K multiples of 128; the wgrad padding is 128.
 *   fwd:   A [S, K] activation-type scales; W [G*N, K] weight-type scales.
 *   dgrad: dY [S, N] activation-type; Wt [K, G*N] weight-type (the dgrad copy
 *          from bw_quantize_128x128).
 *   wgrad: dYt [N, capacity], Xt [K, capacity] from bw_quantize_colwise_padded
 *          (activation-type scales; Xt's scale pointer 16-byte aligned and its
 *          scale_ld a multiple of 4).
 * ws: at least bw_gemm_workspace_size(G) bytes, 256-byte aligned. */
mxg_status bw_grouped_gemm_fwd(const mxg_bw_operand* A, const mxg_bw_operand* W,
                               const int32_t* d_m_splits, int32_t G, int64_t N, void* out,
                               int64_t ld_out, int32_t out_dtype, void* ws, size_t ws_bytes,
                               int32_t* d_status, void* stream);
mxg_status bw_grouped_gemm_dgrad(const mxg_bw_operand* dY, const mxg_bw_operand* Wt,
                                 const int32_t* d_m_splits, int32_t G, void* out, int64_t ld_out,
                                 int32_t out_dtype, void* ws, size_t ws_bytes, int32_t* d_status,
                                 void* stream);
mxg_status bw_grouped_gemm_wgrad(const mxg_bw_operand* dYt, const mxg_bw_operand* Xt,
                                 const int32_t* d_m_splits, int32_t G, int64_t total_rows,
                                 void* out, int32_t out_dtype, int32_t accumulate, void* ws,
                                 size_t ws_bytes, int32_t* d_status, void* stream);
size_t bw_gemm_workspace_size(int32_t G);

/* --------------------------------------------------------------------------
 * Status and configuration
 * ------------------------------------------------------------------------ */

/* Synchronises `stream`, reads *d_status, resets it to 0 and returns it (the
 * only call that blocks the host). */
mxg_status mxg_check_status(int32_t* d_status, void* stream);

/* Static English description of a status code. */
const char* mxg_status_string(mxg_status s);

/* Time limit for every bounded wait inside the kernels (default 2 s). */
void mxg_set_wait_timeout_ns(uint64_t ns);
uint64_t mxg_get_wait_timeout_ns(void);

/* Which MX GEMM kernel the grouped / dense MX GEMM calls launch (process-wide,
 * read at each call).  2 (the default): clusters of two CTAs on neighbouring
 * SMs share each 256 x 256 output tile through the 2-SM block-scaled MMA
 * (tcgen05.mma.cta_group::2), so that every SM stages half of the tile's B
 * rows; where the device cannot co-schedule such pairs the one-SM kernel runs
 * instead.  1: the one-SM kernel (128 x 256 tiles).  Both give results inside
 * the GEMM tolerance; they differ in speed only.  Any other value returns
 * MXG_ERR_SHAPE and changes nothing.  Not specific to any passage of the
 * pages: a scheduling choice of this implementation. */
mxg_status mxg_set_gemm_cta_group(int32_t n);
int32_t mxg_get_gemm_cta_group(void);

/* Diagnostic for the bounded-wait machinery: launches one CTA that waits on
 * an mbarrier nothing ever arrives at, with the same bounded wait the GEMM
 * kernels use and limit `timeout_ns`.  The wait runs out, MXG_ERR_TIMEOUT is
 * recorded in *d_status and the kernel returns; the CUDA context stays
 * usable.  Returns the launch status (enqueue only). */
mxg_status mxg_diag_bounded_wait(int32_t* d_status, uint64_t timeout_ns, void* stream);

/* ABI version: major*10000 + minor*100 + patch. */
int32_t mxg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXG_H_ */
