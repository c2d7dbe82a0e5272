// Single-launch grouped blockwise-FP8 GEMM for sm_103a ("Add ROCm Triton
// blockwise FP8 grouped GEMM", ROCm TransformerEngine PR #716): E4M3 operands
// with fp32 scales per 1x128 (activations, gradients, column-wise wgrad
// operands) or 128x128 (weights) block, and per-128-K promotion:
//
//     C[m, n] = sum_kb ( sum_{k in kb} qa[m, k] * qb[n, k] ) * sa[m, kb] * sb[n, kb]
//
// The passes and their per-expert geometry are those of the MX kernels
// (gemm_common.cuh).  Tile 128x128, one 128-element K block per stage:
//   warp 0     TMA producer: A and B tiles (128-byte swizzle), and for wgrad the
//              stage's 128 column scales of B (1-D bulk copy), 6-stage ring;
//   warp 1     owns TMEM (512 columns) and issues 4 tcgen05.mma kind::f8f6f4
//              (no block scaling) per stage into one of four 128-column
//              partial accumulators, in turn, each started fresh, and makes
//              one commit per stage (to the partial's barrier);
//   warps 2-9  promotion: each thread owns one row and 64 columns; it reads
//              the stage's partial from TMEM, hands it back, frees the
//              stage's shared memory for the producer (the partial being
//              complete means its MMAs have read the stage), and adds
//              partial * sa[row, kb] * sb[., kb] into fp32 registers; at the
//              end of the tile the registers go out through a shared-memory
//              box per warp by TMA tiled stores (bulk reduce-adds for +=).
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace mxg {
namespace {

constexpr int BN = 128;
constexpr int kStages = 6;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr int kTileBytes = 128 * 128;  // one operand tile per stage: 128 rows x 128 B
constexpr int kSbBytes = 128 * 4;      // wgrad: 128 fp32 column scales per stage
constexpr int kTmemCols = 512;
constexpr int kPBufs = 4;  // 128-column partial accumulators in TMEM
// Output staging: one box of 16 rows x 128 bytes (64 BF16 / 32 FP32 columns,
// TMA 128-byte swizzle) per promotion warp.
constexpr int kBoxRows = 16;
constexpr int kBoxBytes = kBoxRows * 128;

struct BwParams {
  Params p;
  const float* sA;   // activation-type scales: (row r, block kb) at sA[kb * sA_ld + r]
  int64_t sA_ld;
  int64_t a_rows;    // rows of A (scale reads beyond it are skipped)
  const float* sB;   // fwd / dgrad: 128x128 weight scales at sB[rb * sB_ld + kb];
  int64_t sB_ld;     // wgrad: activation-type like sA
};

struct BwSmem {
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSbOff = kStages * kStageBytes;
  static constexpr int kBarOff = kSbOff + kStages * kSbBytes;
  static constexpr int kNumBars = 2 * kStages + 2 * kPBufs + 1;  // full, empty, pfull, pempty, drain
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kEpiOff = (kMiscOff + 16 + 1023) & ~1023;  // 1024-byte aligned (swizzle atoms)
  static constexpr int kTotal = kEpiOff + kEpiWarps * kBoxBytes + 1024;
};

__global__ void __launch_bounds__(kThreads, 1)
    grouped_bw_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmOut, const BwParams bp) {
  using L = BwSmem;
  const Params& p = bp.p;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  const bool wg = p.pass == MXG_PASS_WGRAD;

  const PlanView pv = plan_view(const_cast<int32_t*>(p.plan), G);
  if (pv.hdr[0] == 0) return;
  const int total_tiles = pv.hdr[1];
  if ((int)blockIdx.x >= total_tiles) return;

  // per-expert tables: read in place from the plan
  const int32_t* t_off = pv.off;
  const int32_t* t_rt = pv.rt;
  const int32_t* t_poff = pv.poff;
  const int32_t* t_kc = pv.kc;
  const int32_t* t_tiles = pv.tiles;
  const uint32_t bar0 = sbase + L::kBarOff;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto pfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto pempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + kPBufs + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 2 * kPBufs);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      // freed by the promotion warps once the stage's partial is complete
      // (and, for wgrad, once they have read its column scales)
      ptx::mbar_init(empty_bar(s), kEpiWarps);
    }
    for (int b = 0; b < kPBufs; ++b) {
      ptx::mbar_init(pfull_bar(b), 1);
      ptx::mbar_init(pempty_bar(b), kEpiWarps);
    }
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmOut);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto locate = [&](int tile, int& g, int& mt, int& nt, Geo& e) {
    g = find_prefix(t_tiles, G, tile);
    e = group_geo(p, t_off, t_rt, t_poff, t_kc, g);
    const int ntn = cdiv_d(e.Nn, BN);
    tile_mn(tile - t_tiles[g], t_tiles[g + 1] - t_tiles[g], ntn, p.group_m, mt, nt);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed_phase[kStages];
      bool armed[kStages];
      for (int s = 0; s < kStages; ++s) { armed[s] = false; armed_phase[s] = 0; }
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        int g, mt, nt;
        Geo e;
        locate(tile, g, mt, nt, e);
        const int nk = e.Kc / 128;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          const uint32_t fb = full_bar(stage);
          ptx::mbar_arrive_expect_tx(fb, 2 * kTileBytes + (wg ? kSbBytes : 0));
          armed[stage] = true;
          armed_phase[stage] = phase;
          const uint32_t sA = sbase + stage * L::kStageBytes;
          ptx::tma_load_2d(sA, &tmA, (int)(e.a_k0 + kb * 128), (int)(e.a_row0 + (int64_t)mt * 128), fb);
          ptx::tma_load_2d(sA + kTileBytes, &tmB, (int)(e.b_k0 + kb * 128),
                           (int)(e.b_row0 + (int64_t)nt * BN), fb);
          if (wg) {
            const float* src = bp.sB + (e.b_k0 / 128 + kb) * bp.sB_ld + (int64_t)nt * BN;
            ptx::bulk_load(sbase + L::kSbOff + stage * kSbBytes, src, kSbBytes, fb);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < kStages; ++s)
        if (armed[s]) {
          volatile int no_abort = 0;
          ptx::mbar_wait(full_bar(s), armed_phase[s], &no_abort, p.status, p.drain_ns);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t kcount = 0;  // stages consumed so far (selects the partial buffer)
      bool ok = true, issued = false;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        int g, mt, nt;
        Geo e;
        locate(tile, g, mt, nt, e);
        const int nk = e.Kc / 128;
        for (int kb = 0; kb < nk; ++kb, ++kcount) {
          const uint32_t buf = kcount % kPBufs;
          if (!ptx::mbar_wait(full_bar(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          if (!ptx::mbar_wait(pempty_bar(buf), ((kcount / kPBufs) & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t sA = sbase + stage * L::kStageBytes;
          const uint64_t adesc0 = ptx::smem_desc(sA, 16, 1024, 2);
          const uint64_t bdesc0 = ptx::smem_desc(sA + kTileBytes, 16, 1024, 2);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            ptx::mma_f8f6f4(tmem + buf * BN, adesc0 + 2 * j, bdesc0 + 2 * j, p.idesc, j != 0);
          issued = true;
          ptx::tc_commit(pfull_bar(buf));  // the promotion warps free the stage
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (issued) {
        ptx::tc_commit(drain_bar);
        volatile int no_abort = 0;
        ptx::mbar_wait(drain_bar, 0, &no_abort, p.status, p.drain_ns);
      }
    }
  } else {
    // ------------------------------------------------------------ promotion / epilogue
    const int quarter = warp & 3;
    const int chalf = (warp - 2) >> 2;  // columns [64*chalf, 64*chalf + 64)
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(chalf * 64);
    // this warp's staging box; lane l's row of it is l % 16 (lanes 0-15 fill it for
    // rows 0-15 of the warp, then lanes 16-31 for rows 16-31)
    const uint32_t box = sbase + (uint32_t)(L::kEpiOff + (warp - 2) * kBoxBytes);
    const int brow = lane & 15;
    bool pending = false;  // lane 0: bulk groups issued from the box
    // stage the 128-byte row pieces v of lanes (lane >> 4) == half and, when
    // the half's 16 rows are all inside the expert, send them as one box
    auto send_half = [&](int half, const uint32_t* v, int64_t x, int64_t y, bool full, bool reduce) {
      if (lane == 0 && pending) ptx::bulk_wait_group_read<0>();  // the box has been read
      __syncwarp();
      if ((lane >> 4) == half) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          ptx::st_shared_v4(box + (uint32_t)(brow * 128 + ((k ^ (brow & 7)) << 4)), v[4 * k], v[4 * k + 1],
                            v[4 * k + 2], v[4 * k + 3]);
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && full) {
        if (reduce) ptx::tma_reduce_add_2d(&tmOut, box, (int)x, (int)y);
        else ptx::tma_store_2d(&tmOut, box, (int)x, (int)y);
        ptx::bulk_commit_group();
        pending = true;
      }
    };
    uint32_t kcount = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
      int g, mt, nt;
      Geo e;
      locate(tile, g, mt, nt, e);
      const int nk = e.Kc / 128;
      const int row = mt * 128 + quarter * 32 + lane;
      const bool row_ok = row < e.M;
      const int64_t arow = e.a_row0 + row;
      const bool arow_ok = arow < bp.a_rows;
      const int64_t akb0 = e.a_k0 / 128, bkb0 = e.b_k0 / 128;
      const float* sa_col = bp.sA + arow;
      const float* sb_row = bp.sB + (e.b_row0 / 128 + nt) * bp.sB_ld + bkb0;  // fwd / dgrad
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.f;
      float sa_next = (nk > 0 && arow_ok) ? __ldg(sa_col + akb0 * bp.sA_ld) : 0.f;
      float sb_next = (nk > 0 && !wg) ? __ldg(sb_row) : 0.f;
      for (int kb = 0; kb < nk; ++kb, ++kcount) {
        const float sa = sa_next, sb = sb_next;
        if (kb + 1 < nk) {  // prefetch the next block's scales
          sa_next = arow_ok ? __ldg(sa_col + (akb0 + kb + 1) * bp.sA_ld) : 0.f;
          if (!wg) sb_next = __ldg(sb_row + kb + 1);
        }
        const uint32_t buf = kcount % kPBufs;
        const bool landed = ptx::mbar_wait(pfull_bar(buf), (kcount / kPBufs) & 1u, abort_flag, p.status, p.timeout_ns);
        if (!__all_sync(0xffffffffu, landed)) { ok = false; break; }  // the warp leaves together
        ptx::tc_fence_after();
        // every MMA of this stage has completed: its shared memory may be refilled
        if (!wg && lane == 0) ptx::mbar_arrive(empty_bar((int)(kcount % kStages)));
        uint32_t r[64];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(tl + buf * BN, r);
        ptx::tmem_ld_32x32b_x32(tl + buf * BN + 32, r + 32);
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(pempty_bar(buf));
        if (!wg) {
          const float f = sa * sb;
#pragma unroll
          for (int i = 0; i < 64; ++i) acc[i] = fmaf(__uint_as_float(r[i]), f, acc[i]);
        } else {
          const int st = (int)(kcount % kStages);
          // acquire the stage's bulk-copied column scales directly
          const bool sb_ok = ptx::mbar_wait(full_bar(st), (kcount / kStages) & 1u, abort_flag, p.status, p.timeout_ns);
          if (!__all_sync(0xffffffffu, sb_ok)) { ok = false; break; }
          const float4* sbv = reinterpret_cast<const float4*>(smem + L::kSbOff + st * kSbBytes) + chalf * 16;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 b = sbv[i];
            acc[4 * i] = fmaf(__uint_as_float(r[4 * i]), sa * b.x, acc[4 * i]);
            acc[4 * i + 1] = fmaf(__uint_as_float(r[4 * i + 1]), sa * b.y, acc[4 * i + 1]);
            acc[4 * i + 2] = fmaf(__uint_as_float(r[4 * i + 2]), sa * b.z, acc[4 * i + 2]);
            acc[4 * i + 3] = fmaf(__uint_as_float(r[4 * i + 3]), sa * b.w, acc[4 * i + 3]);
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(empty_bar(st));  // column scales consumed
        }
      }
      if (!ok) break;
      const int row0 = mt * 128 + quarter * 32;  // the warp's first row inside the expert
      const int vrows = e.M - row0;
      if (vrows <= 0 || (nk == 0 && p.accumulate)) continue;  // warp-uniform: nothing to write
      const bool full[2] = {vrows >= kBoxRows, vrows >= 2 * kBoxRows};
      const bool direct = row_ok && !full[lane >> 4];  // partial box: the lane stores its own row
      const int64_t col = (int64_t)nt * BN + chalf * 64;
      const int64_t oy0 = e.out_row0 + row0;
      if (p.out_dtype == MXG_OUT_BF16) {
        uint32_t h[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
          h[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) send_half(half, h, col, oy0 + half * kBoxRows, full[half], false);
        if (direct) {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + (e.out_row0 + row) * p.ld_out + col;
#pragma unroll
          for (int i = 0; i < 4; ++i) ptx::st_global_v8(dst + 16 * i, h + 8 * i);
        }
      } else {
#pragma unroll
        for (int piece = 0; piece < 2; ++piece) {  // 32 fp32 columns each
          const uint32_t* v = reinterpret_cast<const uint32_t*>(acc + 32 * piece);
#pragma unroll
          for (int half = 0; half < 2; ++half)
            send_half(half, v, col + 32 * piece, oy0 + half * kBoxRows, full[half], p.accumulate != 0);
        }
        if (direct) {
          float* dst = static_cast<float*>(p.out) + (e.out_row0 + row) * p.ld_out + col;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t v[8];
            if (p.accumulate) {
              ptx::ld_global_v8(dst + 8 * i, v);
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + acc[8 * i + j]);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) v[j] = __float_as_uint(acc[8 * i + j]);
            }
            ptx::st_global_v8(dst + 8 * i, v);
          }
        }
      }
    }
    // every bulk store has completed before the CTA ends
    if (lane == 0 && pending) ptx::bulk_wait_group0();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t bw_gemm_workspace_bytes(int G) { return plan_bytes(G); }

mxg_status launch_grouped_bw_gemm(const BwGemmArgs& a, cudaStream_t stream, int num_sms) {
  if (a.total_rows > 0x7FFFFFFF || a.N > 0x7FFFFFFF || a.K > 0x7FFFFFFF) return MXG_ERR_SHAPE;
  BwParams bp{};
  Params& p = bp.p;
  p.pass = a.pass;
  p.G = a.G;
  p.bn = BN;
  p.accumulate = a.accumulate;
  p.out_dtype = a.out_dtype;
  p.S = a.total_rows;
  p.N = a.N;
  p.K = a.K;
  p.cap = a.a_cols;
  p.pad = 128;
  p.plan = static_cast<const int32_t*>(a.ws);
  p.out = a.out;
  p.ld_out = a.ld_out;
  p.status = a.status;
  p.timeout_ns = wait_timeout_ns();
  p.drain_ns = std::max<uint64_t>(p.timeout_ns, 200000000ull);
  p.group_m = tile_group_m(a.pass == MXG_PASS_FWD ? (double)a.K
                           : a.pass == MXG_PASS_DGRAD ? (double)a.N : (double)a.a_cols / a.G);
  // kind::f8f6f4 descriptor: fp32 accumulate, E4M3 x E4M3, K-major, N = 128, M = 128
  p.idesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
  bp.sA = a.a_scale;
  bp.sA_ld = a.a_scale_ld;
  bp.a_rows = a.a_rows;
  bp.sB = a.b_scale;
  bp.sB_ld = a.b_scale_ld;

  plan_kernel<<<1, kPlanThreads, 0, stream>>>(a.splits, p, static_cast<int32_t*>(a.ws));
  if (cudaGetLastError() != cudaSuccess) return MXG_ERR_CUDA;
  if (a.pass != MXG_PASS_WGRAD && a.total_rows == 0) return MXG_OK;

  CUtensorMap tmA, tmB;
  bool ok;
  if (a.a_cols == 0) {
    ok = make_tmap(&tmA, a.ws, CU_TENSOR_MAP_DATA_TYPE_UINT8, 16, 1, 16, 128, 128) &&
         make_tmap(&tmB, a.ws, CU_TENSOR_MAP_DATA_TYPE_UINT8, 16, 1, 16, 128, BN);
  } else {
    ok = make_tmap(&tmA, a.a_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a_cols, a.a_rows, a.a_ld, 128, 128) &&
         make_tmap(&tmB, a.b_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.b_cols, a.b_rows, a.b_ld, 128, BN);
  }
  if (!ok) return MXG_ERR_CUDA;
  // the output as tiled-store destination (see gemm_mx.cu): boxes of 16 rows x 128 bytes
  CUtensorMap tmOut;
  {
    const bool f32 = a.out_dtype == MXG_OUT_F32;
    const int64_t ocols = a.pass == MXG_PASS_FWD ? a.N : a.K;
    const int64_t orows = a.pass == MXG_PASS_WGRAD ? (int64_t)a.G * a.N : a.total_rows;
    if (!make_tmap(&tmOut, a.out, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ocols,
                   orows, a.ld_out * (f32 ? 4 : 2), f32 ? 32 : 64, kBoxRows))
      return MXG_ERR_CUDA;
  }

  int dev = 0;
  cudaGetDevice(&dev);
  static std::mutex mu;
  static bool attr_set[64] = {};
  {
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 64 && !attr_set[dev]) {
      if (cudaFuncSetAttribute(grouped_bw_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               BwSmem::kTotal) != cudaSuccess) {
        cudaGetLastError();
        return MXG_ERR_CUDA;
      }
      attr_set[dev] = true;
    }
  }
  grouped_bw_gemm_kernel<<<num_sms, kThreads, BwSmem::kTotal, stream>>>(tmA, tmB, tmOut, bp);
  if (cudaGetLastError() != cudaSuccess) return MXG_ERR_CUDA;
  return MXG_OK;
}

}  // namespace mxg
