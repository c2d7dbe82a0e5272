// Single-launch grouped blockwise-FP8 GEMM for sm_103a ("Add ROCm Triton
// blockwise FP8 grouped GEMM", ROCm TransformerEngine PR #716): E4M3 operands
// with fp32 scales per 1x128 (activations, gradients, column-wise wgrad
// operands) or 128x128 (weights) block, and per-128-K promotion:
//
//     C[m, n] = sum_kb ( sum_{k in kb} qa[m, k] * qb[n, k] ) * sa[m, kb] * sb[n, kb]
//
// The passes and their per-expert geometry are those of the MX kernels
// (gemm_common.cuh).  Two kernels: by default clusters of two CTAs run the
// 2-SM MMA on 256 x 256 tiles (grouped_bw_gemm_pair_kernel, described below
// it); mxg_set_gemm_cta_group(1), or a device that cannot co-schedule pairs,
// selects the one-SM kernel.  The one-SM kernel: tile 128x128, one
// 128-element K block per stage:
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

// ---------------------------------------------------------------------------
// The CTA-pair kernel (the default).  Clusters of two CTAs on neighbouring
// SMs own a 256 x 256 output tile: the even CTA issues tcgen05.mma.cta_group::2
// kind::f8f6f4 (M = 256, N = 256, no block scaling) for both, each CTA stages
// its own 128 A rows and one 128-row half of the B tile, and each CTA's TMEM
// receives its 128 rows x 256 columns of every K block's partial product.
// Two 256-column partials alternate in TMEM.  The promotion runs on eight
// warps per CTA whose threads each own one row and 128 columns of the tile in
// registers: per K block they read the partial from TMEM, hand it back, and
// fold it in with packed fp32 pairs (fma.rn.f32x2):
//   fwd / dgrad  acc += P * fl(sa[row, kb] * sb[128-column block, kb])
//   wgrad        acc += fl(P * sa[row, kb]) * sb[column, kb]
// (one rounding before the fused multiply-add; the one-SM kernel rounds the
// scale product in both cases -- either order is one of the evaluations the
// error bound of the promoted sum allows).  The accumulator stays in
// registers until the tile's last K block, so there is no per-tile hand-over
// of TMEM: the next tile's first two K blocks run while the promotion warps
// write the finished tile out.
//   warp 0      TMA producer (each CTA): its A rows and its half of B into a
//               4-stage ring and, for wgrad, the K block's 256 column scales
//               into an 8-slot ring of their own (freed by the promotion
//               warps once folded, so a stage is refilled as soon as its MMAs
//               have read it);
//   warp 1      TMEM owner (512 columns, both CTAs) and, in the even CTA, the
//               MMA issuer: per K block it waits until both CTAs' stages have
//               landed and the partial is free, issues 4 MMAs and commits the
//               stage's barrier and then the partial's barrier in both CTAs;
//   warp 2      relay (each CTA): a landed stage is reported to the issuer's
//               barrier of the even CTA;
//   warps 4-11  promotion and epilogue (TMA tiled stores from a two-box ring
//               per warp; bulk reduce-adds for +=).
// Every wait of the main loops lets the thread sleep in try_wait (a suspend-time
// hint) instead of spinning, so that waiting warps do not take issue slots
// from the promotion warps that share their SM sub-partition.
// Register split: the first warpgroup gives up registers (setmaxnreg) so that
// the two promotion warpgroups can hold 128 fp32 accumulators per thread.
constexpr int kPBN = 256;                 // tile columns
constexpr int kPThreads = 384;            // three warpgroups
constexpr int kPStages = 4;
constexpr int kPPromoWarps = 8;
constexpr int kPRegsLow = 40;             // warpgroup 0 after setmaxnreg.dec
constexpr int kPRegsHigh = 232;          // promotion warpgroups after setmaxnreg.inc
static_assert(kPRegsLow * 128 + kPRegsHigh * 256 <= ((65536 / kPThreads) & ~7) * kPThreads,
              "the register split fits what the block is launched with");
constexpr int kPEpiBoxes = 2;             // per promotion warp: a ring of 32-row x 128-byte boxes
constexpr int kPEpiBytes = kPEpiBoxes * 32 * 128;
constexpr int kPScaleAhead = 4;           // K blocks between a scale's load and its use
constexpr int kPSbSlots = 8;              // wgrad column-scale ring (outlives the operand stage)

struct PairSmem {
  static constexpr int kATile = 128 * 128;
  static constexpr int kBTile = (kPBN / 2) * 128;
  static constexpr int kStageBytes = kATile + kBTile;
  static constexpr int kSbBytes = kPBN * 4;  // wgrad: the tile's 256 column scales per K block
  static constexpr int kSbOff = kPStages * kStageBytes;
  static constexpr int kBarOff = kSbOff + kPSbSlots * kSbBytes;
  // full, empty, sready per stage; pfull, pempty per partial; drain; sbempty per scale slot
  static constexpr int kNumBars = 3 * kPStages + 2 * 2 + 1 + kPSbSlots;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kEpiOff = (kMiscOff + 16 + 1023) & ~1023;
  static constexpr int kTotal = kEpiOff + kPPromoWarps * kPEpiBytes + 1024;
  static_assert(kStageBytes % 1024 == 0, "stage tiles keep the swizzle-atom alignment");
  static_assert(kTotal <= 232448, "fits the dynamic shared memory of one CTA");
};

// Two fp32 values packed in a 64-bit word (low first) -> BF16x2, round to nearest even.
MXG_DEVINL uint32_t pack_bf16x2_u64(uint64_t a) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float((uint32_t)a), __uint_as_float((uint32_t)(a >> 32)));
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <bool kWgrad>
__global__ void __launch_bounds__(kPThreads, 1)
    grouped_bw_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                                const __grid_constant__ CUtensorMap tmB,
                                const __grid_constant__ CUtensorMap tmOut,
                                const __grid_constant__ CUtensorMap tmOut32, const BwParams bp) {
  using L = PairSmem;
  const Params& p = bp.p;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  constexpr bool wg = kWgrad;  // column scales per stage (wgrad) or per 128x128 weight block
  const uint32_t rank = ptx::cluster_ctarank();
  const int unit = (int)ptx::cluster_id_x();
  const int units = (int)ptx::nclusters_x();

  const PlanView pv = plan_view(const_cast<int32_t*>(p.plan), G);
  if (pv.hdr[0] == 0) return;  // invalid splits: nothing is written (both CTAs)
  const int total_tiles = pv.hdr[1];
  if (unit >= total_tiles) return;

  const int32_t* t_off = pv.off;
  const int32_t* t_rt = pv.rt;
  const int32_t* t_poff = pv.poff;
  const int32_t* t_kc = pv.kc;
  const int32_t* t_tiles = pv.tiles;
  const uint32_t bar0 = sbase + L::kBarOff;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kPStages + s); };
  auto sready_bar = [&](int s) { return bar0 + 8u * (2 * kPStages + s); };
  auto pfull_bar = [&](int b) { return bar0 + 8u * (3 * kPStages + b); };
  auto pempty_bar = [&](int b) { return bar0 + 8u * (3 * kPStages + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (3 * kPStages + 4);
  auto sbempty_bar = [&](int j) { return bar0 + 8u * (3 * kPStages + 5 + j); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  auto arrive_issuer = [&](uint32_t bar) { ptx::mbar_arrive_cluster(ptx::mapa_shared(bar, 0)); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);             // the K block's MMAs have read the stage (both CTAs)
      ptx::mbar_init(sready_bar(s), 2);            // the relays of both CTAs
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(pfull_bar(b), 1);
      ptx::mbar_init(pempty_bar(b), 2 * kPPromoWarps);  // the promotion warps of both CTAs
    }
    ptx::mbar_init(drain_bar, 1);
    for (int j = 0; j < kPSbSlots; ++j) ptx::mbar_init(sbempty_bar(j), kPPromoWarps);  // this CTA's promotion warps
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmOut);
    ptx::prefetch_tmap(&tmOut32);
  }
  if (warp == 1) {
    ptx::tmem_alloc_g<2>(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish_g<2>();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the peer's barriers exist before any remote arrival or commit
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto locate = [&](int tile, int& g, int& mt, int& nt, Geo& e) {
    g = find_prefix(t_tiles, G, tile);
    e = group_geo(p, t_off, t_rt, t_poff, t_kc, g);
    const int ntn = cdiv_d(e.Nn, kPBN);
    int mg;
    tile_mn(tile - t_tiles[g], t_tiles[g + 1] - t_tiles[g], ntn, p.group_m, mg, nt);
    mt = mg * 2 + (int)rank;
  };

  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPRegsLow));
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0, kcount = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += units) {
        int g, mt, nt;
        Geo e;
        locate(tile, g, mt, nt, e);
        const int nk = e.Kc / 128;
        // the odd CTA past the expert's rows loads no A (its rows are never stored)
        const bool a_in = mt * 128 < e.M;
        const int ya = (int)(e.a_row0 + (int64_t)mt * 128);
        const int yb = (int)(e.b_row0 + (int64_t)nt * kPBN + (int64_t)rank * (kPBN / 2));
        const uint32_t sb_bytes = wg ? (uint32_t)min(kPBN, e.Nn - nt * kPBN) * 4u : 0u;
        for (int kb = 0; kb < nk; ++kb, ++kcount) {
          if (!ptx::mbar_wait_quiet(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          // wgrad: the column-scale slot's previous K block has been folded
          const int sj = (int)(kcount % kPSbSlots);
          if (wg && !ptx::mbar_wait_quiet(sbempty_bar(sj), ((kcount / kPSbSlots) & 1u) ^ 1u, abort_flag, p.status,
                                          p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          ptx::mbar_arrive_expect_tx(fb, (a_in ? L::kATile : 0) + L::kBTile + sb_bytes);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          const uint32_t sA = sbase + stage * L::kStageBytes;
          if (a_in) ptx::tma_load_2d(sA, &tmA, (int)(e.a_k0 + kb * 128), ya, fb);
          ptx::tma_load_2d(sA + L::kATile, &tmB, (int)(e.b_k0 + kb * 128), yb, fb);
          if (wg) {
            const float* src = bp.sB + (e.b_k0 / 128 + kb) * bp.sB_ld + (int64_t)nt * kPBN;
            ptx::bulk_load(sbase + L::kSbOff + sj * L::kSbBytes, src, sb_bytes, fb);
          }
          if (++stage == kPStages) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < kPStages; ++s)
        if ((armed >> s) & 1u) {
          volatile int no_abort = 0;
          ptx::mbar_wait(full_bar(s), (armed_phase >> s) & 1u, &no_abort, p.status, p.drain_ns);
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t phase = 0, kcount = 0;
      bool ok = true, issued = false;
      for (int tile = unit; tile < total_tiles && ok; tile += units) {
        int g, mt, nt;
        Geo e;
        locate(tile, g, mt, nt, e);
        const int nk = e.Kc / 128;
        for (int kb = 0; kb < nk; ++kb, ++kcount) {
          const uint32_t b = kcount & 1u;
          // both CTAs' stages have landed, and both CTAs have read the partial's previous use
          if (!ptx::mbar_wait_quiet(sready_bar(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          if (!ptx::mbar_wait_quiet(pempty_bar(b), ((kcount >> 1) & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sA = sbase + stage * L::kStageBytes;
          const uint64_t adesc0 = ptx::smem_desc(sA, 16, 1024, 2);
          const uint64_t bdesc0 = ptx::smem_desc(sA + L::kATile, 16, 1024, 2);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            ptx::mma_f8f6f4_g<2>(tmem + b * kPBN, adesc0 + 2 * j, bdesc0 + 2 * j, p.idesc, j != 0);
          issued = true;
          ptx::tc_commit_pair<2>(empty_bar(stage));  // both CTAs' stages have been read
          ptx::tc_commit_pair<2>(pfull_bar(b));      // the partial is complete in both CTAs
          if (++stage == kPStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (issued) {
        ptx::tc_commit_g<2>(drain_bar);
        volatile int no_abort = 0;
        ptx::mbar_wait(drain_bar, 0, &no_abort, p.status, p.drain_ns);
      }
    } else if (warp == 2 && lane == 0) {
      // ---------------------------------------------------------- relay
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += units) {
        int g, mt, nt;
        Geo e;
        locate(tile, g, mt, nt, e);
        const int nk = e.Kc / 128;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait_quiet(full_bar(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          arrive_issuer(sready_bar(stage));
          if (++stage == kPStages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPRegsHigh));
    // ------------------------------------------------------------ promotion / epilogue
    const int quarter = warp & 3;
    const int chalf = (warp - 4) >> 2;  // columns [128 * chalf, 128 * chalf + 128) of the tile
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(chalf * 128);
    const uint32_t box = sbase + (uint32_t)(L::kEpiOff + (warp - 4) * kPEpiBytes);
    uint32_t nsent = 0;  // boxes sent by this warp (one bulk group each)
    // stage 32 words (128 bytes) of this lane's row in the next box of the
    // ring and send the box's valid 16- or 32-row part; a box with fewer than
    // 16 valid rows is not staged (its lanes store their rows themselves)
    auto send = [&](const uint32_t* v, int64_t x, int64_t y0, bool full0, bool full1, bool reduce) {
      if (!full0) return;  // warp-uniform
      const uint32_t bx = box + (nsent % kPEpiBoxes) * (32 * 128);
      // the box's previous bulk store (kPEpiBoxes sends ago) has read it
      if (lane == 0 && nsent >= kPEpiBoxes) ptx::bulk_wait_group_read<kPEpiBoxes - 1>();
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 8; ++k)
        ptx::st_shared_v4(bx + (uint32_t)(lane * 128 + ((k ^ (lane & 7)) << 4)), v[4 * k], v[4 * k + 1],
                          v[4 * k + 2], v[4 * k + 3]);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const void* map = full1 ? (const void*)&tmOut32 : (const void*)&tmOut;
        if (reduce) ptx::tma_reduce_add_2d(map, bx, (int)x, (int)y0);
        else ptx::tma_store_2d(map, bx, (int)x, (int)y0);
        ptx::bulk_commit_group();
      }
      ++nsent;
    };
    uint32_t kcount = 0;
    bool ok = true;
    for (int tile = unit; tile < total_tiles && ok; tile += units) {
      int g, mt, nt;
      Geo e;
      locate(tile, g, mt, nt, e);
      const int nk = e.Kc / 128;
      const int row0 = mt * 128 + quarter * 32;  // the warp's first row inside the expert
      const int col0 = nt * kPBN + chalf * 128;  // the warp's first column
      const bool col_ok = col0 < e.Nn;           // the last tile of an odd 128-column count is half wide
      const int64_t akb0 = e.a_k0 / 128;
      const int64_t oy0 = e.out_row0 + row0;
      const int vrows = e.M - row0;              // the warp's rows inside the expert (may be <= 0)
      uint64_t acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0;
      // thread = row of the tile, 128 columns of it per warp
      const int row = row0 + lane;
      const int64_t arow = e.a_row0 + row;
      const bool arow_ok = row < e.M && arow < bp.a_rows;
      const float* sa_col = bp.sA + arow;
      const float* sb_row = bp.sB + (e.b_row0 / 128 + col0 / 128) * bp.sB_ld + e.b_k0 / 128;  // fwd / dgrad
      // the scales of K blocks kb .. kb + kPScaleAhead - 1, loaded that many
      // blocks ahead of their use (a global load outlasts one K block)
      float saq[kPScaleAhead], sbq[kPScaleAhead];
      auto load_scales = [&](int k, float& a, float& bsc) {
        a = (k < nk && arow_ok) ? __ldg(sa_col + (akb0 + k) * bp.sA_ld) : 0.f;
        bsc = (!wg && k < nk && col_ok) ? __ldg(sb_row + k) : 0.f;
      };
#pragma unroll
      for (int j = 0; j < kPScaleAhead; ++j) load_scales(j, saq[j], sbq[j]);
      for (int kb = 0; kb < nk; ++kb, ++kcount) {
        const float sa = saq[0], sb = sbq[0];
#pragma unroll
        for (int j = 0; j + 1 < kPScaleAhead; ++j) { saq[j] = saq[j + 1]; sbq[j] = sbq[j + 1]; }
        load_scales(kb + kPScaleAhead, saq[kPScaleAhead - 1], sbq[kPScaleAhead - 1]);
        const uint32_t b = kcount & 1u;
        const uint64_t sa2 = ptx::f32x2_pack(sa, sa);
        const uint64_t f2 = ptx::f32x2_pack(sa * sb, sa * sb);
        // wgrad: the K block's column scales of this warp's 128 columns, as fp32 pairs
        const int sj = (int)(kcount % kPSbSlots);
        const ulonglong2* sbc =
            reinterpret_cast<const ulonglong2*>(smem + L::kSbOff + sj * L::kSbBytes + chalf * 128 * 4);
        const bool landed =
            ptx::mbar_wait_quiet(pfull_bar(b), (kcount >> 1) & 1u, abort_flag, p.status, p.timeout_ns);
        if (!__all_sync(0xffffffffu, landed)) { ok = false; break; }
        ptx::tc_fence_after();
        // fwd / dgrad: acc += P * fl(sa * sb); wgrad: acc += fl(P * sa) * sb[column]
        auto fold = [&](const uint32_t* r, int c0) {  // 64 columns starting at c0 of the warp's 128
          if constexpr (!wg) {
#pragma unroll
            for (int i = 0; i < 32; ++i) ptx::fma_f32x2(acc[c0 / 2 + i], ptx::u32x2_pack(r[2 * i], r[2 * i + 1]), f2);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const ulonglong2 c = sbc[c0 / 4 + i];  // column scales (c, c+1) and (c+2, c+3)
              ptx::fma_f32x2(acc[c0 / 2 + 2 * i], ptx::mul_f32x2(ptx::u32x2_pack(r[4 * i], r[4 * i + 1]), sa2), c.x);
              ptx::fma_f32x2(acc[c0 / 2 + 2 * i + 1], ptx::mul_f32x2(ptx::u32x2_pack(r[4 * i + 2], r[4 * i + 3]), sa2),
                             c.y);
            }
          }
        };
        uint32_t r[64];
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(tl + b * kPBN, r);
        ptx::tmem_ld_32x32b_x32(tl + b * kPBN + 32, r + 32);
        ptx::tmem_ld_wait();
        if (col_ok) fold(r, 0);
        __syncwarp();
        ptx::tmem_ld_32x32b_x32(tl + b * kPBN + 64, r);
        ptx::tmem_ld_32x32b_x32(tl + b * kPBN + 96, r + 32);
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_issuer(pempty_bar(b));
        if (col_ok) fold(r, 64);
        if constexpr (wg) {  // every read of the slot's column scales is done
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(sbempty_bar(sj));
        }
      }
      if (!ok) break;
      if (!col_ok || vrows <= 0 || (nk == 0 && p.accumulate)) continue;  // warp-uniform: nothing to write
      const bool full0 = vrows >= 16, full1 = vrows >= 32;
      const bool direct = row < e.M && !((lane >> 4) == 0 ? full0 : full1);
      const int64_t orow = e.out_row0 + row;
      if (p.out_dtype == MXG_OUT_BF16) {
        uint32_t h[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) h[i] = pack_bf16x2_u64(acc[i]);
#pragma unroll
        for (int c = 0; c < 2; ++c) send(h + 32 * c, col0 + 64 * c, oy0, full0, full1, false);
        if (direct) {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + orow * p.ld_out + col0;
#pragma unroll
          for (int i = 0; i < 8; ++i) ptx::st_global_v8(dst + 16 * i, h + 8 * i);
        }
      } else {
        const uint32_t* v = reinterpret_cast<const uint32_t*>(acc);
        const bool reduce = wg && p.accumulate != 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) send(v + 32 * c, col0 + 32 * c, oy0, full0, full1, reduce);
        if (direct) {
          float* dst = static_cast<float*>(p.out) + orow * p.ld_out + col0;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            uint32_t w[8];
            if (reduce) {
              ptx::ld_global_v8(dst + 8 * i, w);
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = __float_as_uint(__uint_as_float(w[j]) + __uint_as_float(v[8 * i + j]));
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = v[8 * i + j];
            }
            ptx::st_global_v8(dst + 8 * i, w);
          }
        }
      }
    }
    if (lane == 0 && nsent > 0) ptx::bulk_wait_group0();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // neither CTA releases TMEM or leaves while the peer may still signal it
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_g<2>(tmem, kTmemCols);
  }
}

}  // namespace

size_t bw_gemm_workspace_bytes(int G) { return plan_bytes(G); }

namespace {
constexpr int kMaxDev = 64;
std::mutex g_bw_mu;

bool bw_smem_attr(const void* fn, int smem, int which, int dev) {
  static bool done[kMaxDev][3] = {};
  std::lock_guard<std::mutex> lk(g_bw_mu);
  if (dev >= 0 && dev < kMaxDev && done[dev][which]) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (dev >= 0 && dev < kMaxDev) done[dev][which] = true;
  return true;
}

// CTA pairs of the pair kernel that the device holds at once (0: clusters of
// two cannot be scheduled), looked up once per device.
int bw_pair_clusters(int dev) {
  static int cached[kMaxDev];
  static bool have[kMaxDev] = {};
  if (dev < 0 || dev >= kMaxDev) return 0;
  {
    std::lock_guard<std::mutex> lk(g_bw_mu);
    if (have[dev]) return cached[dev];
  }
  int n = 0;
  // setmaxnreg.inc waits until the block's registers allow the split: the
  // kernel must be launched with at least the split's total
  cudaFuncAttributes fa{}, fb{};
  const bool regs_ok =
      cudaFuncGetAttributes(&fa, (const void*)grouped_bw_gemm_pair_kernel<false>) == cudaSuccess &&
      cudaFuncGetAttributes(&fb, (const void*)grouped_bw_gemm_pair_kernel<true>) == cudaSuccess &&
      fa.numRegs * kPThreads >= kPRegsLow * 128 + kPRegsHigh * 256 &&
      fb.numRegs * kPThreads >= kPRegsLow * 128 + kPRegsHigh * 256;
  if (!regs_ok) cudaGetLastError();
  if (regs_ok && bw_smem_attr((const void*)grouped_bw_gemm_pair_kernel<false>, PairSmem::kTotal, 1, dev) &&
      bw_smem_attr((const void*)grouped_bw_gemm_pair_kernel<true>, PairSmem::kTotal, 2, dev)) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3((unsigned)std::max(2, sms - (sms & 1)));
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = (size_t)PairSmem::kTotal;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, (const void*)grouped_bw_gemm_pair_kernel<false>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
  }
  std::lock_guard<std::mutex> lk(g_bw_mu);
  cached[dev] = n;
  have[dev] = true;
  return n;
}
}  // namespace

mxg_status launch_grouped_bw_gemm(const BwGemmArgs& a, cudaStream_t stream, int num_sms) {
  if (a.total_rows > 0x7FFFFFFF || a.N > 0x7FFFFFFF || a.K > 0x7FFFFFFF) return MXG_ERR_SHAPE;
  int dev = 0;
  cudaGetDevice(&dev);
  // CTA pairs unless the caller chose the one-SM kernel or the device cannot co-schedule pairs
  const int pair_clusters = gemm_cta_group() == 2 ? bw_pair_clusters(dev) : 0;
  const bool pair = pair_clusters > 0;
  const int bn = pair ? kPBN : BN;
  BwParams bp{};
  Params& p = bp.p;
  p.pass = a.pass;
  p.G = a.G;
  p.bn = bn;
  p.tile_m = pair ? 256 : 128;
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
  p.group_m = std::max(1, tile_group_m(a.pass == MXG_PASS_FWD ? (double)a.K
                                       : a.pass == MXG_PASS_DGRAD ? (double)a.N : (double)a.a_cols / a.G) /
                              (pair ? 2 : 1));
  // kind::f8f6f4 descriptor: fp32 accumulate, E4M3 x E4M3, K-major; N = bn, M = 128 per CTA
  p.idesc = (1u << 4) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(p.tile_m >> 4) << 24);
  bp.sA = a.a_scale;
  bp.sA_ld = a.a_scale_ld;
  bp.a_rows = a.a_rows;
  bp.sB = a.b_scale;
  bp.sB_ld = a.b_scale_ld;

  plan_kernel<<<1, kPlanThreads, 0, stream>>>(a.splits, p, static_cast<int32_t*>(a.ws));
  if (cudaGetLastError() != cudaSuccess) return MXG_ERR_CUDA;
  if (a.pass != MXG_PASS_WGRAD && a.total_rows == 0) return MXG_OK;

  // operand maps; a CTA of a pair loads one 128-row half of the B tile
  const int b_box = pair ? kPBN / 2 : BN;
  CUtensorMap tmA, tmB;
  bool ok;
  if (a.a_cols == 0) {
    ok = make_tmap(&tmA, a.ws, CU_TENSOR_MAP_DATA_TYPE_UINT8, 16, 1, 16, 128, 128) &&
         make_tmap(&tmB, a.ws, CU_TENSOR_MAP_DATA_TYPE_UINT8, 16, 1, 16, 128, b_box);
  } else {
    ok = make_tmap(&tmA, a.a_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a_cols, a.a_rows, a.a_ld, 128, 128) &&
         make_tmap(&tmB, a.b_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.b_cols, a.b_rows, a.b_ld, 128, b_box);
  }
  if (!ok) return MXG_ERR_CUDA;
  // the output as tiled-store destination: boxes of 16 (and, for the pair
  // kernel, 32) rows x 128 bytes
  CUtensorMap tmOut, tmOut32;
  {
    const bool f32 = a.out_dtype == MXG_OUT_F32;
    const int64_t ocols = a.pass == MXG_PASS_FWD ? a.N : a.K;
    const int64_t orows = a.pass == MXG_PASS_WGRAD ? (int64_t)a.G * a.N : a.total_rows;
    const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_tmap(&tmOut, a.out, dt, ocols, orows, a.ld_out * (f32 ? 4 : 2), f32 ? 32 : 64, kBoxRows) ||
        !make_tmap(&tmOut32, a.out, dt, ocols, orows, a.ld_out * (f32 ? 4 : 2), f32 ? 32 : 64, 2 * kBoxRows))
      return MXG_ERR_CUDA;
  }

  cudaError_t err;
  if (pair) {
    void* args[] = {(void*)&tmA, (void*)&tmB, (void*)&tmOut, (void*)&tmOut32, (void*)&bp};
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * pair_clusters));
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = (size_t)PairSmem::kTotal;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const void* fn = a.pass == MXG_PASS_WGRAD ? (const void*)grouped_bw_gemm_pair_kernel<true>
                                              : (const void*)grouped_bw_gemm_pair_kernel<false>;
    err = cudaLaunchKernelExC(&cfg, fn, args);
  } else {
    if (!bw_smem_attr((const void*)grouped_bw_gemm_kernel, BwSmem::kTotal, 0, dev)) return MXG_ERR_CUDA;
    grouped_bw_gemm_kernel<<<num_sms, kThreads, BwSmem::kTotal, stream>>>(tmA, tmB, tmOut, bp);
    err = cudaGetLastError();
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return MXG_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return MXG_ERR_CUDA;
  return MXG_OK;
}

}  // namespace mxg
