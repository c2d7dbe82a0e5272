// BF16 -> MX (E2M1 / E4M3 + UE8M0 per 32) quantization kernels.
//
// Row-wise: the `_row_operand` bridge of "Triton mxfp4 (and a8w4) grouped GEMM
// kernel" (ROCm TransformerEngine PR #723) and the MXFP8 E4M3 reference
// quantizer of PR #745.  Column-wise segment-padded: the wgrad operand
// `_col_operand_grouped_padded` of PR #723.  The scale rule is the OCP MX one
// with the exponent floor at -127 required by the PR #745 review ("Clamp tiny
// block scales to preserve nonzero values").
//
// Both kernels are HBM-bound.  Row-wise: one 32-element block per thread
// (four 16-byte loads, the exponent computed once per block), coalesced
// 16-byte stores.  Column-wise: persistent CTAs stage 128-token x 128-column
// BF16 tiles in shared memory (the next tile's 16-byte loads in flight while
// the current one is quantized); a thread quantizes one column pair down a
// 32-token block and four lanes write 64 (E2M1) / 128 (E4M3) contiguous bytes
// of a transposed output row.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace mxg {

namespace {

template <int kElem>
struct MxFmt;
template <>
struct MxFmt<MXG_E2M1> {
  static constexpr int kEmax = 2;
  static constexpr int kUpMant = 64;  // 6 = (1 + 64/128) * 2^2
};
template <>
struct MxFmt<MXG_E4M3> {
  static constexpr int kEmax = 8;
  static constexpr int kUpMant = 96;  // 448 = (1 + 96/128) * 2^8
};

template <int kElem>
MXG_DEVINL int mx_exponent(uint32_t am, bool round_up) {
  return mx_exponent_from_amax_bits(am, MxFmt<kElem>::kEmax, round_up, MxFmt<kElem>::kUpMant);
}

// Quantize 8 BF16 values (four 32-bit words) with inverse scale `sinv`.
// E2M1 -> one 32-bit word (8 nibbles); E4M3 -> two 32-bit words.
template <int kElem>
MXG_DEVINL void quantize8(const uint32_t* w, float sinv, uint32_t* out) {
  // both values of a word scaled by one packed fp32 multiply (per-lane IEEE
  // round to nearest, subnormals kept: the same results as two scalar products)
  float v[8];
  uint64_t s2;
  asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(sinv));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint64_t p;
    asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%1, %2};\n\tmul.rn.f32x2 %0, t, %3;\n\t}"
        : "=l"(p)
        : "r"(w[i] << 16), "r"(w[i] & 0xFFFF0000u), "l"(s2));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v[2 * i]), "=f"(v[2 * i + 1]) : "l"(p));
  }
  // The hardware conversions keep the sign of a value that rounds to zero
  // (E2M1 0x8, E4M3 0x80), as the OCP rule and the oracle do.
  if constexpr (kElem == MXG_E2M1) {
    out[0] = cvt_e2m1x8(v);
  } else {
    out[0] = cvt_e4m3x4(v[0], v[1], v[2], v[3]);
    out[1] = cvt_e4m3x4(v[4], v[5], v[6], v[7]);
  }
}

constexpr int kRowThreads = 256;

// One 32-element block per thread: four 16-byte loads (the block's 64 bytes),
// amax and exponent computed once, 16 (E2M1) or 32 (E4M3) output bytes and
// one scale byte.  Consecutive threads take consecutive blocks of a row, so
// a warp reads 2 KB and writes 512 B / 1 KB contiguous.
template <int kElem>
__global__ void __launch_bounds__(kRowThreads) mx_rowwise_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld_x,
    uint8_t* __restrict__ q, int64_t ld_q, uint8_t* __restrict__ s, int64_t ld_s, bool round_up) {
  const int64_t blocks_per_row = cols >> 5;
  const int64_t total = rows * blocks_per_row;
  const int64_t step = (int64_t)gridDim.x * kRowThreads;
  for (int64_t t = (int64_t)blockIdx.x * kRowThreads + threadIdx.x; t < total; t += step) {
    const int64_t r = t / blocks_per_row;
    const int64_t b = t - r * blocks_per_row;
    const uint4* src = reinterpret_cast<const uint4*>(x + r * ld_x + b * 32);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldcs(src + i);
      w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
    }
    const uint32_t am = bf16x32_absmax_bits(w);
    const int e = mx_exponent<kElem>(am, round_up);
    const float sinv = pow2_neg(e);
    if constexpr (kElem == MXG_E2M1) {
      uint4 o;
      quantize8<kElem>(&w[0], sinv, &o.x);
      quantize8<kElem>(&w[4], sinv, &o.y);
      quantize8<kElem>(&w[8], sinv, &o.z);
      quantize8<kElem>(&w[12], sinv, &o.w);
      __stcs(reinterpret_cast<uint4*>(q + r * ld_q + b * 16), o);
    } else {
      uint4 o0, o1;
      quantize8<kElem>(&w[0], sinv, &o0.x);
      quantize8<kElem>(&w[4], sinv, &o0.z);
      quantize8<kElem>(&w[8], sinv, &o1.x);
      quantize8<kElem>(&w[12], sinv, &o1.z);
      uint4* dst = reinterpret_cast<uint4*>(q + r * ld_q + b * 32);
      __stcs(dst, o0);
      __stcs(dst + 1, o1);
    }
    s[r * ld_s + b] = (uint8_t)(e + 127);
  }
}

// Row-wise with the scales written straight into the tensor-core staging
// order ("pre-swizzled" scales: "Integrate MXFP4 hipblaslt GEMM support",
// Takeaways; the "fused scale packing kernel" of "Grouped MXFP8 GEMMs with
// HipKittens", ROCm TransformerEngine PR #661).
// The rows are cut into segments (the routing splits, or G equal segments of
// seg_rows rows), each segment into tiles of 128 rows, tiles numbered across
// segments (RT in all); the scales of 128 rows x 4 blocks form a 512-byte
// chunk, chunk (kc, rt) at ((kc * RT + rt) * 512), local row i and block j at
// byte (i % 32) * 16 + (i / 32) * 4 + j; bytes without a row or block are 0.
//
// The loop runs over padded positions (tile row, block rounded up to 4), one
// block per lane as in the plain kernel; the four lanes that share a chunk
// word gather its bytes with shuffles and one of them stores the word.  A
// warp's lanes take consecutive positions, so every group of four is aligned
// to a word and the warp iterates as a whole (the shuffles need all lanes).
template <int kElem, bool kSplits>
__global__ void __launch_bounds__(kRowThreads) mx_rowwise_packed_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld_x,
    uint8_t* __restrict__ q, int64_t ld_q, uint8_t* __restrict__ sp,
    const int32_t* __restrict__ splits, int G, int64_t seg_rows, int32_t* status, bool round_up) {
  __shared__ int64_t s_off[kMaxExperts + 1];  // row offsets of the segments
  __shared__ int32_t s_rtp[kMaxExperts + 1];  // first tile of each segment; [G] = RT
  __shared__ int64_t warp_m[kRowThreads / 32];
  __shared__ int32_t warp_t[kRowThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int64_t RT;
  int tps = 1;  // tiles per segment (equal segments)
  if constexpr (kSplits) {
    // block-wide scan of (rows, tiles) over the G <= 512 splits, two per thread
    static_assert(2 * kRowThreads >= kMaxExperts, "two splits per thread");
    int64_t m0 = 0, m1 = 0;
    if (2 * tid < G) m0 = splits[2 * tid];
    if (2 * tid + 1 < G) m1 = splits[2 * tid + 1];
    const bool neg = m0 < 0 || m1 < 0;
    const int32_t t0 = m0 > 0 ? (int32_t)((m0 + 127) >> 7) : 0;
    const int32_t t1 = m1 > 0 ? (int32_t)((m1 + 127) >> 7) : 0;
    int64_t sm = m0 + m1;
    int32_t st = t0 + t1;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t om = __shfl_up_sync(0xffffffffu, sm, d);
      const int32_t ot = __shfl_up_sync(0xffffffffu, st, d);
      if (lane >= d) { sm += om; st += ot; }
    }
    if (lane == 31) { warp_m[wid] = sm; warp_t[wid] = st; }
    const int any_neg = __syncthreads_or(neg);
    int64_t bm = 0;
    int32_t bt = 0;
    for (int w = 0; w < wid; ++w) { bm += warp_m[w]; bt += warp_t[w]; }
    const int64_t em = bm + sm - (m0 + m1);
    const int32_t et = bt + st - (t0 + t1);
    if (2 * tid <= G) { s_off[2 * tid] = em; s_rtp[2 * tid] = et; }
    if (2 * tid + 1 <= G) { s_off[2 * tid + 1] = em + m0; s_rtp[2 * tid + 1] = et + t0; }
    if (tid == kRowThreads - 1) { s_off[G] = bm + sm; s_rtp[G] = bt + st; }  // totals (G = 512 too)
    __syncthreads();
    if (any_neg || s_off[G] != rows) {  // nothing is written
      if (blockIdx.x == 0 && tid == 0) report(status, MXG_ERR_SPLITS);
      return;
    }
    RT = s_rtp[G];
  } else {
    tps = (int)((seg_rows + 127) >> 7);
    RT = (int64_t)G * tps;
  }
  const int64_t KB = cols >> 5;
  const int64_t KBp = (KB + 3) & ~int64_t(3);
  const int64_t total = RT * 128 * KBp;
  const int64_t step = (int64_t)gridDim.x * kRowThreads;
  // This thread's block t = prow * KBp + b, stepped by the grid stride without
  // dividing; its row tile only grows, so its segment g is found by a forward
  // scan (the last g with a first tile <= rt: non-empty, the next one starts
  // after rt).
  const int64_t t0 = (int64_t)blockIdx.x * kRowThreads + wid * 32 + lane;
  int64_t prow = t0 / KBp, b = t0 - prow * KBp;
  const int64_t sq = step / KBp, sr = step - sq * KBp;
  int g = 0;
  for (int64_t base = (int64_t)blockIdx.x * kRowThreads + wid * 32; base < total; base += step) {
    const int64_t t = base + lane;
    uint32_t sbyte = 0;
    if (t < total) {
      const int rt = (int)(prow >> 7);
      int64_t m, row0;
      if constexpr (kSplits) {
        while (g + 1 < G && s_rtp[g + 1] <= rt) ++g;
        m = s_off[g + 1] - s_off[g];
        row0 = s_off[g];
      } else {
        while ((g + 1) * tps <= rt) ++g;
        m = seg_rows;
        row0 = (int64_t)g * seg_rows;
      }
      const int64_t i = (int64_t)(rt - (kSplits ? s_rtp[g] : g * tps)) * 128 + (prow & 127);
      if (i < m && b < KB) {
        const int64_t r = row0 + i;
        const uint4* src = reinterpret_cast<const uint4*>(x + r * ld_x + b * 32);
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = __ldcs(src + k);
          w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
        }
        const uint32_t am = bf16x32_absmax_bits(w);
        const int e = mx_exponent<kElem>(am, round_up);
        const float sinv = pow2_neg(e);
        if constexpr (kElem == MXG_E2M1) {
          uint4 o;
          quantize8<kElem>(&w[0], sinv, &o.x);
          quantize8<kElem>(&w[4], sinv, &o.y);
          quantize8<kElem>(&w[8], sinv, &o.z);
          quantize8<kElem>(&w[12], sinv, &o.w);
          __stcs(reinterpret_cast<uint4*>(q + r * ld_q + b * 16), o);
        } else {
          uint4 o0, o1;
          quantize8<kElem>(&w[0], sinv, &o0.x);
          quantize8<kElem>(&w[4], sinv, &o0.z);
          quantize8<kElem>(&w[8], sinv, &o1.x);
          quantize8<kElem>(&w[12], sinv, &o1.z);
          uint4* dst = reinterpret_cast<uint4*>(q + r * ld_q + b * 32);
          __stcs(dst, o0);
          __stcs(dst + 1, o1);
        }
        sbyte = (uint32_t)(e + 127);
      }
    }
    // the word of blocks 4c .. 4c+3: lanes (lane & ~3) + j, j = 0..3
    const int l0 = lane & ~3;
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) word |= __shfl_sync(0xffffffffu, sbyte, l0 + j) << (8 * j);
    if (t < total && (lane & 3) == 0) {
      const int64_t rt = prow >> 7;
      const int il = (int)(prow & 127);
      const int64_t kc = b >> 2;
      *reinterpret_cast<uint32_t*>(sp + (kc * RT + rt) * 512 + (il & 31) * 16 + (il >> 5) * 4) = word;
    }
    b += sr;
    prow += sq;
    if (b >= KBp) { b -= KBp; ++prow; }
  }
}

// ---------------------------------------------------------------------------
// Column-wise, segment-padded.
// ---------------------------------------------------------------------------
constexpr int kColTokens = 128;  // padded token positions per CTA (4 blocks)
constexpr int kColCols = 128;    // input columns per CTA
constexpr int kColThreads = 256;

// Per-CTA expert table: splits validated and prefix-summed in shared memory.
struct SegTable {
  int64_t off[kMaxExperts + 1];   // row offsets
  int64_t poff[kMaxExperts + 1];  // padded offsets
};

// Builds the prefix tables with a block-wide scan (blockDim.x == 256, two
// experts per thread).  Returns false -- after reporting when `do_report` --
// if a split is negative, the splits do not sum to `rows`, or the padded
// total exceeds `capacity`.  All threads must call it.
__device__ bool build_seg_table(SegTable& t, const int32_t* __restrict__ splits, int G,
                                int64_t rows, int pad, int64_t capacity, int32_t* status,
                                bool do_report) {
  __shared__ int64_t warp_m[8], warp_p[8];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int64_t m0 = 0, m1 = 0;
  if (2 * tid < G) m0 = splits[2 * tid];
  if (2 * tid + 1 < G) m1 = splits[2 * tid + 1];
  const bool neg = (m0 < 0) || (m1 < 0);
  const int64_t p0 = m0 > 0 ? ((m0 + pad - 1) / pad) * pad : 0;
  const int64_t p1 = m1 > 0 ? ((m1 + pad - 1) / pad) * pad : 0;
  int64_t sm = m0 + m1, sp = p0 + p1;  // inclusive warp scans of the pair sums
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int64_t om = __shfl_up_sync(0xffffffffu, sm, d);
    const int64_t op = __shfl_up_sync(0xffffffffu, sp, d);
    if (lane >= d) { sm += om; sp += op; }
  }
  if (lane == 31) { warp_m[wid] = sm; warp_p[wid] = sp; }
  const int any_neg = __syncthreads_or(neg);
  int64_t bm = 0, bp = 0;
  for (int w = 0; w < wid; ++w) { bm += warp_m[w]; bp += warp_p[w]; }
  // exclusive prefix before this thread's pair
  const int64_t em = bm + sm - (m0 + m1), ep = bp + sp - (p0 + p1);
  if (2 * tid <= G) { t.off[2 * tid] = em; t.poff[2 * tid] = ep; }
  if (2 * tid + 1 <= G) { t.off[2 * tid + 1] = em + m0; t.poff[2 * tid + 1] = ep + p0; }
  if (tid == (int)blockDim.x - 1) {  // the totals, entry G: for G = 512 no pair above reaches it
    t.off[G] = bm + sm;
    t.poff[G] = bp + sp;
  }
  __syncthreads();
  int bad = 0;
  if (any_neg) bad = MXG_ERR_SPLITS;
  else if (t.off[G] != rows) bad = MXG_ERR_SPLITS;
  else if (t.poff[G] > capacity) bad = MXG_ERR_CAPACITY;
  if (bad && do_report && tid == 0) report(status, bad);
  return bad == 0;
}

// Expert owning padded position j (poff[g] <= j < poff[g+1]); -1 if beyond.
__device__ int find_segment(const SegTable& t, int G, int64_t j) {
  if (j >= t.poff[G]) return -1;
  int lo = 0, hi = G - 1;
  while (lo < hi) {  // last g with poff[g] <= j
    const int mid = (lo + hi + 1) >> 1;
    if (t.poff[mid] <= j) lo = mid; else hi = mid - 1;
  }
  return lo;  // the last such g is non-empty since poff[g+1] > j
}

// Blockwise FP8 arithmetic (see the blockwise section below).
constexpr float kBwAmaxFloor = 1e-4f;

MXG_DEVINL float bw_scale(uint32_t amax_bits) {
  const float a = fmaxf(__uint_as_float(amax_bits << 16), kBwAmaxFloor);
  return __fdiv_rn(a, 448.0f);
}

// Power-of-two form: s = 2^k, the smallest power of two with 448 * s >= a,
// a = max(amax, 1e-4f) = m * 2^e with m in [1, 2).  Since 448 = 1.75 * 2^8,
// k = e - 8, plus one when m > 1.75.  k is in [-22, 120] for finite BF16
// input, so the UE8M0 byte k + 127 is an MX scale and x / s = x * 2^-k exactly.
MXG_DEVINL int bw_pow2_exponent(uint32_t amax_bits) {
  const float a = fmaxf(__uint_as_float(amax_bits << 16), kBwAmaxFloor);
  const uint32_t b = __float_as_uint(a);
  return (int)((b >> 23) & 0xFFu) - 127 - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
}
MXG_DEVINL uint32_t ue8m0x4(int k) { return (uint32_t)(k + 127) * 0x01010101u; }

// 8 bf16 (four words) * m (a power of two) -> 8 E4M3 codes (two words).
MXG_DEVINL void bw_quantize8_mul(const uint32_t* w, float m, uint32_t* o) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16lo_to_f32(w[i]) * m;
    v[2 * i + 1] = bf16hi_to_f32(w[i]) * m;
  }
  o[0] = cvt_e4m3x4(v[0], v[1], v[2], v[3]);
  o[1] = cvt_e4m3x4(v[4], v[5], v[6], v[7]);
}

// 8 bf16 (four words) / s -> 8 E4M3 codes (two words).
MXG_DEVINL void bw_quantize8(const uint32_t* w, float s, uint32_t* o) {
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __fdiv_rn(bf16lo_to_f32(w[i]), s);
    v[2 * i + 1] = __fdiv_rn(bf16hi_to_f32(w[i]), s);
  }
  o[0] = cvt_e4m3x4(v[0], v[1], v[2], v[3]);
  o[1] = cvt_e4m3x4(v[4], v[5], v[6], v[7]);
}

// Quantizes one 32-element block (16 words of bf16 pairs, element 2i in the
// low half) and writes its codes and scale.
template <int kElem>
MXG_DEVINL void emit_col_block(const uint32_t* w, uint8_t* qrow, uint8_t* srow, bool round_up) {
  const uint32_t am = bf16x32_absmax_bits(w);
  const int e = mx_exponent<kElem>(am, round_up);
  const float sinv = pow2_neg(e);
  if constexpr (kElem == MXG_E2M1) {
    uint4 o;
    quantize8<kElem>(&w[0], sinv, &o.x);
    quantize8<kElem>(&w[4], sinv, &o.y);
    quantize8<kElem>(&w[8], sinv, &o.z);
    quantize8<kElem>(&w[12], sinv, &o.w);
    __stcs(reinterpret_cast<uint4*>(qrow), o);
  } else {
    uint4 o0, o1;
    quantize8<kElem>(&w[0], sinv, &o0.x);
    quantize8<kElem>(&w[4], sinv, &o0.z);
    quantize8<kElem>(&w[8], sinv, &o1.x);
    quantize8<kElem>(&w[12], sinv, &o1.z);
    __stcs(reinterpret_cast<uint4*>(qrow), o0);
    __stcs(reinterpret_cast<uint4*>(qrow) + 1, o1);
  }
  *srow = (uint8_t)(e + 127);
}

// Column-wise blocks of a column pair straight from the staged tile: T[t] is
// the 32-bit word (column c in the low half, c + 1 in the high half) of token
// t of the block.  Both columns' amax come from one 16-bit SIMD max per word,
// and each value is widened from its half of T[t] in place, so the pair needs
// no byte permutes.  kHi selects column c + 1.  Same results as emit_col_block
// on the column's own words.
template <int kElem, bool kHi>
MXG_DEVINL void quantize8_col(const uint32_t* T, uint64_t s2, uint32_t* out) {
  float v[8];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t a = kHi ? (T[2 * k] & 0xFFFF0000u) : (T[2 * k] << 16);
    const uint32_t b = kHi ? (T[2 * k + 1] & 0xFFFF0000u) : (T[2 * k + 1] << 16);
    uint64_t p;
    asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%1, %2};\n\tmul.rn.f32x2 %0, t, %3;\n\t}" : "=l"(p) : "r"(a), "r"(b), "l"(s2));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v[2 * k]), "=f"(v[2 * k + 1]) : "l"(p));
  }
  if constexpr (kElem == MXG_E2M1) {
    out[0] = cvt_e2m1x8(v);
  } else {
    out[0] = cvt_e4m3x4(v[0], v[1], v[2], v[3]);
    out[1] = cvt_e4m3x4(v[4], v[5], v[6], v[7]);
  }
}

template <int kElem, bool kHi>
MXG_DEVINL uint32_t emit_col_half(const uint32_t* T, uint32_t am, uint8_t* qrow, bool round_up) {
  const int e = mx_exponent<kElem>(am, round_up);
  uint64_t s2;
  const float sinv = pow2_neg(e);
  asm("mov.b64 %0, {%1, %1};" : "=l"(s2) : "f"(sinv));
  if constexpr (kElem == MXG_E2M1) {
    uint4 o;
    quantize8_col<kElem, kHi>(&T[0], s2, &o.x);
    quantize8_col<kElem, kHi>(&T[8], s2, &o.y);
    quantize8_col<kElem, kHi>(&T[16], s2, &o.z);
    quantize8_col<kElem, kHi>(&T[24], s2, &o.w);
    __stcs(reinterpret_cast<uint4*>(qrow), o);
  } else {
    uint4 o0, o1;
    quantize8_col<kElem, kHi>(&T[0], s2, &o0.x);
    quantize8_col<kElem, kHi>(&T[8], s2, &o0.z);
    quantize8_col<kElem, kHi>(&T[16], s2, &o1.x);
    quantize8_col<kElem, kHi>(&T[24], s2, &o1.z);
    __stcs(reinterpret_cast<uint4*>(qrow), o0);
    __stcs(reinterpret_cast<uint4*>(qrow) + 1, o1);
  }
  return (uint32_t)(e + 127);
}

// One column's quarter (32 tokens, 16 words) of a 128-token blockwise block
// whose amax over the four quarters is `am`: E4M3 codes (32 bytes) and, from
// the first quarter, the block's scale -- fp32 at sT[(j0/128)*ld_s + col]
// (kBw 1) or the UE8M0 byte repeated four times at sT + col*ld_s + j0/32 (kBw 2).
template <int kBw>
MXG_DEVINL void emit_bw_col(const uint32_t* w, uint32_t am, uint8_t* q, void* sT, int64_t ld_s,
                            int64_t col, int64_t j0, bool first_quarter) {
  uint32_t o[8];
  if constexpr (kBw == 2) {
    const int k = bw_pow2_exponent(am);
    const float m = pow2_neg(k);
#pragma unroll
    for (int i = 0; i < 4; ++i) bw_quantize8_mul(&w[4 * i], m, &o[2 * i]);
    if (first_quarter) *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(sT) + col * ld_s + j0 / 32) = ue8m0x4(k);
  } else {
    const float sc = bw_scale(am);
#pragma unroll
    for (int i = 0; i < 4; ++i) bw_quantize8(&w[4 * i], sc, &o[2 * i]);
    if (first_quarter) static_cast<float*>(sT)[(j0 / 128) * ld_s + col] = sc;
  }
  __stcs(reinterpret_cast<uint4*>(q), make_uint4(o[0], o[1], o[2], o[3]));
  __stcs(reinterpret_cast<uint4*>(q) + 1, make_uint4(o[4], o[5], o[6], o[7]));
}

// Persistent CTAs over tiles of 128 padded token positions x 128 columns
// (tile = token tile * column tiles + column tile), kColCtasPerSm per SM.
// The expert table is built once per CTA.  For each tile the source row of
// every position is looked up once; the BF16 tile goes through registers
// (each thread's eight 16-byte loads for the next tile are issued before the
// current tile is quantized) into shared memory as 32-bit column pairs,
// token row r at word r*64 + (r/32)*8 (the extra 8 words per 32-row group put
// the four 32-token blocks of a column pair in different banks).  Thread =
// (column pair, 32-token block), the four blocks of a pair on adjacent lanes,
// so each transposed output row is written as 64 (E2M1) / 128 (E4M3)
// contiguous bytes by four lanes.  (A three-buffer cp.async pipeline of the
// same tiles measured ~20% slower on GB300 than this register prefetch.)
//
// kDual: the same pass also writes the row-wise operand (the fused dual
// quantizer, one HBM read of x for both): each real token row of the staged
// tile is quantized along the columns, four 32-blocks per row and tile, and
// written at its source row; padding positions write nothing.
//
// kBw (blockwise FP8 column-wise operand, segments padded to 128, E4M3): a
// tile is one 128-token block; the four lanes of a column pair reduce the
// block's amax with two shuffles and each quantizes its 32 tokens (kBw 1:
// fp32 scales, kBw 2: power-of-two scales as UE8M0, see emit_bw_col).  With
// kDual the same pass writes the 1x128 row-wise operand (the dual blockwise
// quantizer of "Add ROCm Triton blockwise FP8 grouped GEMM"): each token row
// of the tile is one 128-column block, taken by 16 lanes of a warp (one
// 16-byte chunk each, amax over the 16 with four shuffles) so that the row's
// 128 code bytes leave as one contiguous piece.
constexpr int kColCtasPerSm = 2;

// kPacked (MX, not dual): the scales go straight into the tensor-core staging
// order of a k-segmented operand -- chunk (kc, rt) at (kc * RT + rt) * 512 with
// kc = the expert's first k-chunk + local 32-block / 4, RT = ceil(cols / 128),
// channel i of the row tile and block j of the chunk at (i % 32) * 16 +
// (i / 32) * 4 + j -- into a buffer the launcher has zeroed (ld_s unused).
template <int kElem, bool kDual, int kBw = 0, bool kPacked = false>
__global__ void __launch_bounds__(kColThreads, kColCtasPerSm) mx_colwise_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld_x,
    const int32_t* __restrict__ splits, int G, int pad, uint8_t* __restrict__ qT, int64_t ld_q,
    void* __restrict__ sT, int64_t ld_s, int64_t capacity, int64_t* __restrict__ pad_offsets,
    int32_t* status, uint8_t* __restrict__ q_row, int64_t ld_qr, uint8_t* __restrict__ s_row,
    int64_t ld_sr, bool round_up) {
  static_assert(kColTokens == 128 && kColCols == 128 && kColThreads == 256, "thread mapping");
  __shared__ SegTable tab;
  __shared__ __align__(16) uint32_t tile[kColTokens * (kColCols / 2) + 4 * 8];
  __shared__ int64_t src_row[2][kColTokens];  // source row of each position, or -1
  // kPacked: per 32-token block of the tile, its chunk-grid offset
  // (k-chunk * row tiles * 512 + block in the chunk), found once per tile
  __shared__ int64_t blk_off[2][kColTokens / 32];
  __shared__ int32_t kcp[kMaxExperts + 1];     // kPacked: first k-chunk of each expert
  const bool first = blockIdx.x == 0;
  if (!build_seg_table(tab, splits, G, rows, pad, capacity, status, first)) return;
  if constexpr (kPacked) {
    // exclusive prefix of ceil(p_g / 128), two experts per thread
    __shared__ int32_t wsum[kColThreads / 32];
    const int tid = threadIdx.x, ln = tid & 31, wd = tid >> 5;
    const int32_t k0 = 2 * tid < G ? (int32_t)((tab.poff[2 * tid + 1] - tab.poff[2 * tid] + 127) >> 7) : 0;
    const int32_t k1 = 2 * tid + 1 < G ? (int32_t)((tab.poff[2 * tid + 2] - tab.poff[2 * tid + 1] + 127) >> 7) : 0;
    int32_t sc = k0 + k1;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t o = __shfl_up_sync(0xffffffffu, sc, d);
      if (ln >= d) sc += o;
    }
    if (ln == 31) wsum[wd] = sc;
    __syncthreads();
    int32_t base = 0;
    for (int w = 0; w < wd; ++w) base += wsum[w];
    const int32_t ex = base + sc - (k0 + k1);
    if (2 * tid <= G) kcp[2 * tid] = ex;
    if (2 * tid + 1 <= G) kcp[2 * tid + 1] = ex + k0;
    if (tid == kColThreads - 1) kcp[G] = base + sc;  // the total (G = 512 too)
    __syncthreads();
  }
  if (first && pad_offsets != nullptr) {
    for (int g = threadIdx.x; g <= G; g += blockDim.x) pad_offsets[g] = tab.poff[g];
  }
  const int64_t ptot = tab.poff[G];
  const int64_t ntc = (cols + kColCols - 1) / kColCols;
  const int64_t ntiles = (ptot + kColTokens - 1) / kColTokens * ntc;
  int64_t tile_id = blockIdx.x;
  if (tile_id >= ntiles) return;

  // tile = token tile tt * ntc + column tile tc; the pair is advanced by the
  // grid stride without dividing
  const int64_t gq = gridDim.x / ntc, gr = gridDim.x % ntc;
  auto advance = [&](int64_t& tt, int64_t& tc) {
    tt += gq;
    tc += gr;
    if (tc >= ntc) { tc -= ntc; ++tt; }
  };
  auto fill_src = [&](int64_t tt, int buf) {  // threads < kColTokens
    const int64_t j = tt * kColTokens + threadIdx.x;
    int64_t sr = -1;
    const int g = find_segment(tab, G, j);
    if (g >= 0) {
      const int64_t tok = j - tab.poff[g];
      if (tok < tab.off[g + 1] - tab.off[g]) sr = tab.off[g] + tok;
    }
    src_row[buf][threadIdx.x] = sr;
    if constexpr (kPacked) {
      if ((threadIdx.x & 31) == 0 && g >= 0) {
        const int64_t lb = (j - tab.poff[g]) >> 5;  // the expert's local 32-block
        blk_off[buf][threadIdx.x >> 5] = ((int64_t)kcp[g] + (lb >> 2)) * ((cols + 127) >> 7) * 512 + (lb & 3);
      }
    }
  };
  auto load = [&](int64_t tc, int buf, uint4* v) {
    const int64_t c0 = tc * kColCols;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = threadIdx.x + kColThreads * i;
      const int jr = idx >> 4;  // 16 chunks of 8 columns per token row
      const int cc = (idx & 15) * 8;
      const int64_t sr = src_row[buf][jr];
      v[i] = make_uint4(0, 0, 0, 0);
      if (sr >= 0 && c0 + cc < cols) v[i] = __ldcs(reinterpret_cast<const uint4*>(x + sr * ld_x + c0 + cc));
    }
  };

  uint4 v[8];
  int64_t cur_tt = tile_id / ntc, cur_tc = tile_id % ntc;
  if (threadIdx.x < kColTokens) fill_src(cur_tt, 0);
  __syncthreads();
  load(cur_tc, 0, v);
  int buf = 0;
  const int lane = threadIdx.x & 31;
  const int cp = (threadIdx.x >> 5) * 8 + (lane >> 2);  // column pair 0..63
  const int blk = lane & 3;                              // 32-token block 0..3
  constexpr int kBytesPerBlock = kElem == MXG_E2M1 ? 16 : 32;
  for (; tile_id < ntiles; tile_id += gridDim.x) {
    const int64_t next = tile_id + gridDim.x;
    int64_t nxt_tt = cur_tt, nxt_tc = cur_tc;
    advance(nxt_tt, nxt_tc);
    if (next < ntiles && threadIdx.x < kColTokens) fill_src(nxt_tt, buf ^ 1);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int idx = threadIdx.x + kColThreads * i;
      const int jr = idx >> 4;
      const int cc = (idx & 15) * 8;
      *reinterpret_cast<uint4*>(&tile[jr * 64 + (jr >> 5) * 8 + (cc >> 1)]) = v[i];
    }
    __syncthreads();  // tile and the next tile's source rows are visible
    if (next < ntiles) load(nxt_tc, buf ^ 1, v);

    const int64_t jb = cur_tt * kColTokens + 32 * blk;
    const int64_t col = cur_tc * kColCols + 2 * cp;
    const uint32_t* tp = tile + (32 * blk) * 64 + blk * 8 + cp;
    uint32_t T[32];  // token t of the block: column col (low half), col + 1 (high half)
#pragma unroll
    for (int t = 0; t < 32; ++t) T[t] = tp[t * 64];
    if constexpr (kBw == 0) {
      if (jb < ptot && col < cols) {  // beyond the last expert: nothing written
        const int64_t qoff = (jb >> 5) * kBytesPerBlock;
        uint8_t* s8 = static_cast<uint8_t*>(sT);
        uint8_t *sa, *sb;
        if constexpr (kPacked) {
          const int i0 = (int)(col & 127);              // col even: col + 1 is in the same row tile
          uint8_t* cb = s8 + blk_off[buf][blk] + (col >> 7) * 512;
          sa = cb + (i0 & 31) * 16 + (i0 >> 5) * 4;
          sb = cb + ((i0 + 1) & 31) * 16 + ((i0 + 1) >> 5) * 4;
        } else {
          sa = s8 + col * ld_s + (jb >> 5);
          sb = s8 + (col + 1) * ld_s + (jb >> 5);
        }
        uint32_t m = 0;
#pragma unroll
        for (int t = 0; t < 32; ++t) m = __vmaxu2(m, T[t] & 0x7FFF7FFFu);
        *sa = (uint8_t)emit_col_half<kElem, false>(T, m & 0xFFFFu, qT + col * ld_q + qoff, round_up);
        if (col + 1 < cols) *sb = (uint8_t)emit_col_half<kElem, true>(T, m >> 16, qT + (col + 1) * ld_q + qoff, round_up);
      }
    } else {
      uint32_t wa[16], wb[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        wa[i] = __byte_perm(T[2 * i], T[2 * i + 1], 0x5410);  // column col:   tokens 2i, 2i+1
        wb[i] = __byte_perm(T[2 * i], T[2 * i + 1], 0x7632);  // column col+1
      }
      // the 128-token block's amax over the four quarter lanes (all lanes
      // take part; validity is uniform per warp: cols % 32 == 0, ptot % 128 == 0)
      uint32_t m = 0;
#pragma unroll
      for (int t = 0; t < 32; ++t) m = __vmaxu2(m, T[t] & 0x7FFF7FFFu);
      uint32_t ama = m & 0xFFFFu, amb = m >> 16;
      ama = max(ama, __shfl_xor_sync(0xffffffffu, ama, 1));
      ama = max(ama, __shfl_xor_sync(0xffffffffu, ama, 2));
      amb = max(amb, __shfl_xor_sync(0xffffffffu, amb, 1));
      amb = max(amb, __shfl_xor_sync(0xffffffffu, amb, 2));
      if (jb < ptot && col < cols) {
        const int64_t j0 = jb - 32 * blk;
        emit_bw_col<kBw>(wa, ama, qT + col * ld_q + jb, sT, ld_s, col, j0, blk == 0);
        if (col + 1 < cols) emit_bw_col<kBw>(wb, amb, qT + (col + 1) * ld_q + jb, sT, ld_s, col + 1, j0, blk == 0);
      }
    }
    if constexpr (kDual && kBw != 0) {
      // row-wise 1x128 blocks: warp w takes tile rows 16*it + 2w + (lane >> 4);
      // lane & 15 is the row's 16-byte chunk (8 columns)
      const int64_t c0 = cur_tc * kColCols;  // cols % 128 == 0: the block is the whole tile row
      const int sub = lane >> 4, ch = lane & 15, wid = threadIdx.x >> 5;
#pragma unroll 2
      for (int it = 0; it < kColTokens / 16; ++it) {
        const int rr = 16 * it + 2 * wid + sub;
        const int64_t sr = src_row[buf][rr];
        const uint4 v4 = *reinterpret_cast<const uint4*>(tile + rr * 64 + (rr >> 5) * 8 + 4 * ch);
        const uint32_t w[4] = {v4.x, v4.y, v4.z, v4.w};
        uint32_t am = max(max(bf16x2_absmax_bits(w[0]), bf16x2_absmax_bits(w[1])),
                          max(bf16x2_absmax_bits(w[2]), bf16x2_absmax_bits(w[3])));
#pragma unroll
        for (int d = 1; d < 16; d <<= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, d));
        if (sr >= 0) {
          uint32_t o[2];
          if constexpr (kBw == 2) {
            const int k = bw_pow2_exponent(am);
            bw_quantize8_mul(w, pow2_neg(k), o);
            if (ch == 0) *reinterpret_cast<uint32_t*>(s_row + sr * ld_sr + c0 / 32) = ue8m0x4(k);
          } else {
            const float sc = bw_scale(am);
            bw_quantize8(w, sc, o);
            if (ch == 0) reinterpret_cast<float*>(s_row)[(c0 / 128) * ld_sr + sr] = sc;
          }
          *reinterpret_cast<uint2*>(q_row + sr * ld_qr + c0 + 8 * ch) = make_uint2(o[0], o[1]);
        }
      }
    }
    if constexpr (kDual && kBw == 0) {
      // row-wise blocks: thread -> token row tid/2, 32-blocks 2*(tid%2) and +1
      const int rr = threadIdx.x >> 1;
      const int64_t sr = src_row[buf][rr];
      if (sr >= 0) {
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int b = 2 * (threadIdx.x & 1) + bb;
          const int64_t colb = cur_tc * kColCols + 32 * b;
          if (colb < cols) {
            const uint4* rp = reinterpret_cast<const uint4*>(tile + rr * 64 + (rr >> 5) * 8 + 16 * b);
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 v4 = rp[i];
              w[4 * i] = v4.x; w[4 * i + 1] = v4.y; w[4 * i + 2] = v4.z; w[4 * i + 3] = v4.w;
            }
            emit_col_block<kElem>(w, q_row + sr * ld_qr + (colb >> 5) * kBytesPerBlock,
                                  s_row + sr * ld_sr + (colb >> 5), round_up);
          }
        }
      }
    }
    __syncthreads();  // the tile buffer is rewritten next iteration
    buf ^= 1;
    cur_tt = nxt_tt;
    cur_tc = nxt_tc;
  }
}

// ---------------------------------------------------------------------------
// Blockwise FP8 ("Add ROCm Triton blockwise FP8 grouped GEMM", PR #716):
// a = max(amax, 1e-4f), s = a / 448 (fp32, IEEE division), q = RNE_satfinite_
// E4M3(x / s) with x / s an IEEE fp32 division; s is the dequant scale.
// Activation-type scales are stored block-column-major: scale of (row r,
// 128-block kb) at s[kb * ld_s + r], so a GEMM epilogue thread holding row r
// reads its scales with coalesced loads.
// ---------------------------------------------------------------------------
// 1x128 along the row: four lanes per block, 32 values (four 16-byte loads)
// per lane; the block amax is reduced over the four lanes with two shuffles.
// kPow2: power-of-two scales written as UE8M0 bytes [rows, cols/32], each
// block's byte repeated over its four 32-blocks (an MXFP8 operand).
template <bool kPow2>
__global__ void __launch_bounds__(kRowThreads) bw_rowwise_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ld_x,
    uint8_t* __restrict__ q, int64_t ld_q, void* __restrict__ s, int64_t ld_s) {
  const int64_t b32_per_row = cols >> 5;
  const int64_t total = rows * b32_per_row;
  const int64_t step = (int64_t)gridDim.x * kRowThreads;
  for (int64_t base = (int64_t)blockIdx.x * kRowThreads; base < total; base += step) {
    const int64_t t = base + threadIdx.x;
    const bool live = t < total;  // total % 4 == 0: a block's four lanes live or die together
    const int64_t r = live ? t / b32_per_row : 0;
    const int64_t b = live ? t - r * b32_per_row : 0;
    uint32_t w[16];
    if (live) {
      const uint4* src = reinterpret_cast<const uint4*>(x + r * ld_x + b * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldcs(src + i);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = 0;
    }
    uint32_t am = bf16x32_absmax_bits(w);
    am = max(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = max(am, __shfl_xor_sync(0xffffffffu, am, 2));
    if (!live) continue;
    uint32_t o[8];
    const bool first = (b & 3) == 0;
    if constexpr (kPow2) {
      const int k = bw_pow2_exponent(am);
      const float m = pow2_neg(k);
#pragma unroll
      for (int i = 0; i < 4; ++i) bw_quantize8_mul(&w[4 * i], m, &o[2 * i]);
      if (first)
        *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(s) + r * ld_s + b) = ue8m0x4(k);
    } else {
      const float sc = bw_scale(am);
#pragma unroll
      for (int i = 0; i < 4; ++i) bw_quantize8(&w[4 * i], sc, &o[2 * i]);
      if (first) static_cast<float*>(s)[(b >> 2) * ld_s + r] = sc;
    }
    uint2* dst = reinterpret_cast<uint2*>(q + r * ld_q + b * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint2(o[2 * i], o[2 * i + 1]);
  }
}

// 128x128 weight tiles, persistent CTAs of 256 threads (kWCtasPerSm per SM)
// over tiles in row-of-blocks order; thread t holds row t/2, 64 columns, and
// its eight 16-byte loads of the next tile are in flight while the current
// tile is quantized.  Optionally writes the transposed codes (dgrad copy).
// fp32 scales: s [rows/128, K/128], sT [K/128, rows/128] (ld_s, ld_sT unused).
// kPow2: UE8M0 bytes s [rows, K/32] and sT [K, rows/32], the tile's byte in
// every 32-block of its rows (an MXFP8 operand and its transposed copy).
constexpr int kBwTile = 128;
constexpr int kWCtasPerSm = 2;
template <bool kPow2>
__global__ void __launch_bounds__(256, kWCtasPerSm) bw_weight_kernel(
    const uint16_t* __restrict__ w, int64_t rows, int64_t K, int64_t ld_w, uint8_t* __restrict__ q,
    int64_t ld_q, void* __restrict__ s, int64_t ld_s, uint8_t* __restrict__ qT, int64_t ld_qT,
    void* __restrict__ sT, int64_t ld_sT) {
  __shared__ uint32_t warp_max[8];
  __shared__ __align__(16) uint8_t codes[kBwTile][kBwTile + 16];
  const int t = threadIdx.x, r = t >> 1, h = t & 1;
  const int64_t nkb = K / kBwTile;
  const int64_t ntiles = nkb * (rows / kBwTile);
  int64_t id = blockIdx.x;
  if (id >= ntiles) return;
  auto load = [&](int64_t tile, uint32_t* v) {
    const int64_t rb = tile / nkb, kb = tile - rb * nkb;
    const uint4* src = reinterpret_cast<const uint4*>(w + (rb * kBwTile + r) * ld_w + kb * kBwTile + h * 64);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 u = __ldcs(src + i);
      v[4 * i] = u.x; v[4 * i + 1] = u.y; v[4 * i + 2] = u.z; v[4 * i + 3] = u.w;
    }
  };
  uint32_t v[32];
  load(id, v);
  for (; id < ntiles; id += gridDim.x) {
    const int64_t rb = id / nkb, kb = id - rb * nkb;
    uint32_t am = max(bf16x32_absmax_bits(v), bf16x32_absmax_bits(v + 16));
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) am = max(am, __shfl_xor_sync(0xffffffffu, am, d));
    if ((t & 31) == 0) warp_max[t >> 5] = am;
    const int64_t nxt = id + gridDim.x;
    uint32_t pv[32];
    if (nxt < ntiles) load(nxt, pv);
    __syncthreads();
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = max(m, warp_max[i]);  // every thread: the tile amax
    uint32_t o[16];
    int k2 = 0;
    if constexpr (kPow2) {
      k2 = bw_pow2_exponent(m);
      const float mul = pow2_neg(k2);
#pragma unroll
      for (int i = 0; i < 8; ++i) bw_quantize8_mul(&v[4 * i], mul, &o[2 * i]);
      if (h == 0)
        *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(s) + (rb * kBwTile + r) * ld_s + kb * 4) = ue8m0x4(k2);
    } else {
      const float sc = bw_scale(m);
#pragma unroll
      for (int i = 0; i < 8; ++i) bw_quantize8(&v[4 * i], sc, &o[2 * i]);
      if (t == 0) {
        static_cast<float*>(s)[rb * nkb + kb] = sc;
        if (sT != nullptr) static_cast<float*>(sT)[kb * (rows / kBwTile) + rb] = sc;
      }
    }
    uint4* dst = reinterpret_cast<uint4*>(q + (rb * kBwTile + r) * ld_q + kb * kBwTile + h * 64);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    if (qT != nullptr) {  // uniform
      uint4* crow = reinterpret_cast<uint4*>(&codes[r][h * 64]);
#pragma unroll
      for (int i = 0; i < 4; ++i) crow[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      __syncthreads();
      // transposed: thread t writes row kk = t/2 of the [K, rows] copy, 64 codes
      const int kk = t >> 1;
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = h * 64 + 4 * i;
        pk[i] = (uint32_t)codes[j][kk] | ((uint32_t)codes[j + 1][kk] << 8) |
                ((uint32_t)codes[j + 2][kk] << 16) | ((uint32_t)codes[j + 3][kk] << 24);
      }
      uint4* tdst = reinterpret_cast<uint4*>(qT + (kb * kBwTile + kk) * ld_qT + rb * kBwTile + h * 64);
#pragma unroll
      for (int i = 0; i < 4; ++i) tdst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      if constexpr (kPow2) {
        if (h == 0)
          *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(sT) + (kb * kBwTile + kk) * ld_sT + rb * 4) =
              ue8m0x4(k2);
      }
    }
    __syncthreads();  // warp_max and codes are rewritten next iteration
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = pv[i];
  }
}

}  // namespace

cudaError_t launch_mx_rowwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int elem,
                              void* q, int64_t ld_q, uint8_t* s, int64_t ld_s,
                              cudaStream_t stream, int num_sms) {
  const bool round_up = (elem & MXG_SCALE_ROUND_UP) != 0;  // rule flag carried in elem
  elem &= 0xFF;
  const int64_t total = rows * (cols / 32);
  const int threads = kRowThreads;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms * 8 * 4;  // a few full waves, then grid-stride
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(q);
  if (elem == MXG_E2M1)
    mx_rowwise_kernel<MXG_E2M1><<<(unsigned)blocks, threads, 0, stream>>>(xp, rows, cols, ld_x, qp,
                                                                          ld_q, s, ld_s, round_up);
  else
    mx_rowwise_kernel<MXG_E4M3><<<(unsigned)blocks, threads, 0, stream>>>(xp, rows, cols, ld_x, qp,
                                                                          ld_q, s, ld_s, round_up);
  return cudaGetLastError();
}

cudaError_t launch_mx_rowwise_packed(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int elem,
                                     void* q, int64_t ld_q, uint8_t* sp, const int32_t* splits, int G,
                                     int64_t seg_rows, int64_t rt_bound, int32_t* status,
                                     cudaStream_t stream, int num_sms) {
  const bool round_up = (elem & MXG_SCALE_ROUND_UP) != 0;  // rule flag carried in elem
  elem &= 0xFF;
  const int64_t kbp = ((cols / 32) + 3) / 4 * 4;
  const int64_t total = rt_bound * 128 * kbp;
  int64_t blocks = (total + kRowThreads - 1) / kRowThreads;
  // With splits every CTA scans them first: one resident wave (as many CTAs
  // as fit on the SMs at once), each CTA then loops, so the scan is paid once
  // per CTA.  Without splits, a few waves as in the plain kernel.
  int64_t cap = (int64_t)num_sms * 8 * 4;
  if (splits) {
    int per_sm = 0;
    const void* fn = elem == MXG_E2M1 ? (const void*)mx_rowwise_packed_kernel<MXG_E2M1, true>
                                      : (const void*)mx_rowwise_packed_kernel<MXG_E4M3, true>;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kRowThreads, 0) != cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      per_sm = 4;
    }
    cap = (int64_t)num_sms * per_sm;
  }
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(q);
  const dim3 grid((unsigned)blocks);
  if (elem == MXG_E2M1) {
    if (splits)
      mx_rowwise_packed_kernel<MXG_E2M1, true><<<grid, kRowThreads, 0, stream>>>(
          xp, rows, cols, ld_x, qp, ld_q, sp, splits, G, seg_rows, status, round_up);
    else
      mx_rowwise_packed_kernel<MXG_E2M1, false><<<grid, kRowThreads, 0, stream>>>(
          xp, rows, cols, ld_x, qp, ld_q, sp, nullptr, G, seg_rows, status, round_up);
  } else {
    if (splits)
      mx_rowwise_packed_kernel<MXG_E4M3, true><<<grid, kRowThreads, 0, stream>>>(
          xp, rows, cols, ld_x, qp, ld_q, sp, splits, G, seg_rows, status, round_up);
    else
      mx_rowwise_packed_kernel<MXG_E4M3, false><<<grid, kRowThreads, 0, stream>>>(
          xp, rows, cols, ld_x, qp, ld_q, sp, nullptr, G, seg_rows, status, round_up);
  }
  return cudaGetLastError();
}

cudaError_t launch_mx_colwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                              const int32_t* splits, int G, int pad, int elem, void* qT,
                              int64_t ld_q, uint8_t* sT, int64_t ld_s, int64_t capacity,
                              int64_t* pad_offsets, int32_t* status, cudaStream_t stream,
                              int num_sms, void* q_row, int64_t ld_qr, uint8_t* s_row,
                              int64_t ld_sr, int64_t packed_bytes) {
  const bool round_up = (elem & MXG_SCALE_ROUND_UP) != 0;  // rule flag carried in elem
  elem &= 0xFF;
  // persistent: at most kColCtasPerSm CTAs per SM, never more than the tiles
  const int64_t tiles = (capacity + kColTokens - 1) / kColTokens * ((cols + kColCols - 1) / kColCols);
  int64_t ctas = std::min<int64_t>(tiles, (int64_t)num_sms * kColCtasPerSm);
  if (ctas < 1) ctas = 1;
  dim3 grid((unsigned)ctas);
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(qT);
  auto* qr = static_cast<uint8_t*>(q_row);
  const bool dual = q_row != nullptr;
  if (packed_bytes > 0) {  // staging-order scales: slack bytes must read as scale 2^-127
    cudaError_t e = cudaMemsetAsync(sT, 0, (size_t)packed_bytes, stream);
    if (e != cudaSuccess) return e;
    if (elem == MXG_E2M1)
      mx_colwise_kernel<MXG_E2M1, false, 0, true><<<grid, kColThreads, 0, stream>>>(
          xp, rows, cols, ld_x, splits, G, pad, qp, ld_q, sT, 0, capacity, pad_offsets, status, nullptr, 0,
          nullptr, 0, round_up);
    else
      mx_colwise_kernel<MXG_E4M3, false, 0, true><<<grid, kColThreads, 0, stream>>>(
          xp, rows, cols, ld_x, splits, G, pad, qp, ld_q, sT, 0, capacity, pad_offsets, status, nullptr, 0,
          nullptr, 0, round_up);
    return cudaGetLastError();
  }
  if (elem == MXG_E2M1) {
    if (dual)
      mx_colwise_kernel<MXG_E2M1, true><<<grid, kColThreads, 0, stream>>>(
          xp, rows, cols, ld_x, splits, G, pad, qp, ld_q, sT, ld_s, capacity, pad_offsets, status, qr, ld_qr,
          s_row, ld_sr, round_up);
    else
      mx_colwise_kernel<MXG_E2M1, false><<<grid, kColThreads, 0, stream>>>(
          xp, rows, cols, ld_x, splits, G, pad, qp, ld_q, sT, ld_s, capacity, pad_offsets, status, nullptr,
          0, nullptr, 0, round_up);
  } else {
    if (dual)
      mx_colwise_kernel<MXG_E4M3, true><<<grid, kColThreads, 0, stream>>>(
          xp, rows, cols, ld_x, splits, G, pad, qp, ld_q, sT, ld_s, capacity, pad_offsets, status, qr, ld_qr,
          s_row, ld_sr, round_up);
    else
      mx_colwise_kernel<MXG_E4M3, false><<<grid, kColThreads, 0, stream>>>(
          xp, rows, cols, ld_x, splits, G, pad, qp, ld_q, sT, ld_s, capacity, pad_offsets, status, nullptr,
          0, nullptr, 0, round_up);
  }
  return cudaGetLastError();
}

}  // namespace mxg

namespace mxg {

cudaError_t launch_bw_rowwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x, void* q,
                              int64_t ld_q, void* s, int64_t ld_s, bool pow2, cudaStream_t stream,
                              int num_sms) {
  const int64_t total = rows * (cols / 32);
  int64_t blocks = (total + kRowThreads - 1) / kRowThreads;
  const int64_t cap = (int64_t)num_sms * 8 * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(q);
  if (pow2)
    bw_rowwise_kernel<true><<<(unsigned)blocks, kRowThreads, 0, stream>>>(xp, rows, cols, ld_x, qp, ld_q, s, ld_s);
  else
    bw_rowwise_kernel<false><<<(unsigned)blocks, kRowThreads, 0, stream>>>(xp, rows, cols, ld_x, qp, ld_q, s, ld_s);
  return cudaGetLastError();
}

cudaError_t launch_bw_weight(const void* w, int64_t rows, int64_t K, int64_t ld_w, void* q,
                             int64_t ld_q, void* s, int64_t ld_s, void* qT, int64_t ld_qT, void* sT,
                             int64_t ld_sT, bool pow2, cudaStream_t stream, int num_sms) {
  const int64_t tiles = (K / kBwTile) * (rows / kBwTile);
  int64_t ctas = std::min<int64_t>(tiles, (int64_t)num_sms * kWCtasPerSm);
  if (ctas < 1) ctas = 1;
  auto* wp = static_cast<const uint16_t*>(w);
  auto* qp = static_cast<uint8_t*>(q);
  auto* qTp = static_cast<uint8_t*>(qT);
  if (pow2)
    bw_weight_kernel<true><<<(unsigned)ctas, 256, 0, stream>>>(wp, rows, K, ld_w, qp, ld_q, s, ld_s, qTp, ld_qT,
                                                               sT, ld_sT);
  else
    bw_weight_kernel<false><<<(unsigned)ctas, 256, 0, stream>>>(wp, rows, K, ld_w, qp, ld_q, s, ld_s, qTp, ld_qT,
                                                                sT, ld_sT);
  return cudaGetLastError();
}

cudaError_t launch_bw_colwise(const void* x, int64_t rows, int64_t cols, int64_t ld_x,
                              const int32_t* splits, int G, void* qT, int64_t ld_q, void* sT,
                              int64_t ld_s, int64_t capacity, int64_t* pad_offsets,
                              int32_t* status, bool pow2, cudaStream_t stream, int num_sms,
                              void* q_row, int64_t ld_qr, void* s_row, int64_t ld_sr) {
  // the persistent column-wise kernel with one 128-token block per tile
  const int64_t tiles = (capacity + kColTokens - 1) / kColTokens * ((cols + kColCols - 1) / kColCols);
  int64_t ctas = std::min<int64_t>(tiles, (int64_t)num_sms * kColCtasPerSm);
  if (ctas < 1) ctas = 1;
  auto* xp = static_cast<const uint16_t*>(x);
  auto* qp = static_cast<uint8_t*>(qT);
  auto* qr = static_cast<uint8_t*>(q_row);
  auto* sr = static_cast<uint8_t*>(s_row);
  const bool dual = q_row != nullptr;
  if (pow2 && dual)
    mx_colwise_kernel<MXG_E4M3, true, 2><<<(unsigned)ctas, kColThreads, 0, stream>>>(
        xp, rows, cols, ld_x, splits, G, 128, qp, ld_q, sT, ld_s, capacity, pad_offsets, status, qr, ld_qr,
        sr, ld_sr, false);
  else if (pow2)
    mx_colwise_kernel<MXG_E4M3, false, 2><<<(unsigned)ctas, kColThreads, 0, stream>>>(
        xp, rows, cols, ld_x, splits, G, 128, qp, ld_q, sT, ld_s, capacity, pad_offsets, status, nullptr, 0,
        nullptr, 0, false);
  else if (dual)
    mx_colwise_kernel<MXG_E4M3, true, 1><<<(unsigned)ctas, kColThreads, 0, stream>>>(
        xp, rows, cols, ld_x, splits, G, 128, qp, ld_q, sT, ld_s, capacity, pad_offsets, status, qr, ld_qr,
        sr, ld_sr, false);
  else
    mx_colwise_kernel<MXG_E4M3, false, 1><<<(unsigned)ctas, kColThreads, 0, stream>>>(
        xp, rows, cols, ld_x, splits, G, 128, qp, ld_q, sT, ld_s, capacity, pad_offsets, status, nullptr, 0,
        nullptr, 0, false);
  return cudaGetLastError();
}

}  // namespace mxg
