// Single-launch grouped MX GEMM for sm_103a (tcgen05 block-scaled MMA).
//
// The three passes of an MoE expert layer ("Triton mxfp4 (and a8w4) grouped
// GEMM kernel", ROCm TransformerEngine PR #723; per-pass shapes from
// "Integrate MXFP4 hipblaslt GEMM support", PR #697) are one problem: for each
// expert g, C_g[M_g x N_g] = A_g[M_g x Kc_g] * B_g[N_g x Kc_g]^T with both
// operands K-major and MX-quantized along Kc:
//
//   pass   A (rows)        B (rows)         contraction           output rows
//   fwd    X  rows off_g   W  rows g*N      K, from 0             off_g + i
//   dgrad  dY rows off_g   Wt rows 0..K-1   N, B from col g*N     off_g + i
//   wgrad  dYt rows 0..N   Xt rows 0..K     p_g, from col poff_g  g*N + n
//
// Launch sequence on the caller's stream (all device-side, no host sync):
//   1. plan kernel (1 CTA): validates m_splits (>= 0, sum == rows, padded
//      total <= capacity) and writes per-expert prefix tables to the
//      workspace.  A failure is reported in *status and disables 2 and 3.
//   2. scale-pack kernel: UE8M0 bytes from the plain [rows, cols/32] layout
//      into 512-byte chunks (128 rows x 4 blocks, the order tcgen05.cp
//      32x128b.warpx4 expects: byte (r%32)*16 + (r/32)*4 + block), one chunk
//      per (row tile, 128-element k chunk) with every expert's rows (or k
//      range) starting on a fresh chunk -- the "scale packing" step that the
//      HipKittens grouped MXFP8 kernel (PR #661) also performs.  Skipped for
//      an operand whose quantizer already wrote that order (packed scales).
//   3. the persistent GEMM kernel, one CTA per SM, 352 threads:
//        warp 0    TMA producer: A/B data tiles (128-byte swizzle) into a
//                  4-stage shared-memory ring (mbarriers);
//        warp 1    TMEM owner and MMA issuer (one thread): 4 tcgen05.mma per
//                  stage (kind::mxf4 for MXFP4, kind::mxf8f6f4 for MXFP8 /
//                  a8w4) accumulating a 128x256 fp32 tile in TMEM;
//        warps 2-5 epilogue: tcgen05.ld, fp32 -> BF16/FP32, staged through
//                  shared memory and written by TMA tiled stores (bulk
//                  reduce-adds for +=), only the expert's valid rows;
//        warps 6-9 scale feeders, one per 32-lane quarter of TMEM: each
//                  stage's scale chunks go from shared memory to registers
//                  and on into that stage's TMEM scale slot (tcgen05.st),
//                  then the stage is handed to the MMA issuer;
//        warp 10   second producer: the stage's scale chunks (TMA / bulk
//                  copies onto the same barrier).
//      The feeders keep every tcgen05.cp out of the MMA issuer's stream:
//      measured on GB300, a scale copy issued between MMAs (3 per FP8 stage,
//      6 per FP4 stage) slowed the MMA stream by a third to two thirds, and
//      more again when the issuer also waited on an mbarrier.
//      Tiles (expert, m-tile, n-tile) are enumerated expert-major and strided
//      over the CTAs; inside an expert, m-tiles run in groups (tile_mn) so
//      that a group's A rows stay in L2 while the n-tiles sweep over them.
//   By default the kernel runs as clusters of two CTAs on neighbouring SMs
//   (kCta = 2): a pair owns a 256 x 256 tile, the even CTA issues the 2-SM
//   block-scaled MMA (tcgen05.mma.cta_group::2, M = 256) for both, and each
//   CTA stages its own 128 A rows and one 128-row half of the B tile (5-6
//   stage ring), fills its own TMEM scale slots (its A rows, all 256 B rows)
//   and writes its own 128 output rows.  mxg_set_gemm_cta_group(1) selects
//   the one-SM form (kCta = 1: 128 x 256 tiles, 4 stages).
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "gemm_common.cuh"
#include "sm100_ptx.cuh"

namespace mxg {
namespace {

constexpr int BM = 128;           // tile rows of one CTA (TMEM lanes)
constexpr int BN = 256;           // tile columns (TMEM fp32 columns)
constexpr int kThreads = 352;
constexpr int kATileBytes = BM * 128;  // 128 bytes of K per row per stage
constexpr int kChunkBytes = 512;       // 128 rows x 4 scale bytes
constexpr int kTmemCols = 512;
// Epilogue output staging: per epilogue warp (32 tile rows), two boxes of 16
// rows x 128 bytes (64 BF16 or 32 FP32 columns) in the TMA 128-byte swizzle.
constexpr int kEpiWarps = 4;
constexpr int kEpiBoxRows = 16;
constexpr int kEpiBoxBytes = kEpiBoxRows * 128;
constexpr int kEpiWarpBytes = 2 * kEpiBoxBytes;
constexpr int kSfTmemCol0 = BN;        // scale slots start after the accumulator
constexpr int kStashCol = 384;         // FP32 epilogue: accumulator columns 128..255, copied here

enum Kind { KIND_MXF4 = 0, KIND_A8W4 = 1, KIND_MXF8 = 2 };

template <int kKind>
struct KindCfg {
  static constexpr int kMmaK = kKind == KIND_MXF4 ? 64 : 32;      // elements per MMA
  static constexpr int kStageK = kKind == KIND_MXF4 ? 256 : 128;  // elements per stage
  static constexpr int kKPS = kStageK / 128;                      // scale k-chunks per stage
  static constexpr int kSlotCols = kKPS * 12;                     // TMEM scale slot: A 4 + B 8 columns per k-chunk
};
static_assert(kStashCol + BN / 2 <= kTmemCols, "the FP32 stash lies inside the allocation");

// ---------------------------------------------------------------------------
// 2. Scale packing.  blockIdx.y selects the operand (0 = A, 1 = B).
// ---------------------------------------------------------------------------
struct PackSrc {
  const uint8_t* src;
  int64_t ld;
  uint8_t* dst;
};

constexpr int kPackKc = 8;  // k-chunks per CTA (eight 4-byte words per 32-byte row segment)
static_assert(kPackKc == 8, "the pack kernel maps 8 threads to a row");

// grid = (row tiles, k-chunk groups of kPackKc, operand), 128 threads.  A CTA
// repacks one 128-row tile over kPackKc chunks (32 scale bytes per row): the
// rows are read as 4-byte words, eight threads per row (one chunk each), into
// a shared-memory tile, and every 512-byte chunk is then written with one
// coalesced 4-byte store per thread.  Words whose four blocks are not all
// inside the expert's contraction range, or are not 4-byte aligned, are
// assembled from byte loads; blocks outside the range are zero.
__global__ void __launch_bounds__(128) pack_scales_kernel(Params p, PackSrc sa, PackSrc sb) {
  const PlanView pv = plan_view(const_cast<int32_t*>(p.plan), p.G);
  if (pv.hdr[0] == 0) return;
  const bool isA = blockIdx.z == 0;
  const PackSrc ps = isA ? sa : sb;
  if (ps.dst == nullptr) return;  // this operand's scales arrive packed
  const int G = p.G;
  const int nrt = (int)((p.N + 127) / 128);
  int RT, KC;
  if (p.pass == MXG_PASS_FWD) {
    RT = isA ? pv.rt[G] : p.rtB;
    KC = p.kcA_fixed;
  } else if (p.pass == MXG_PASS_DGRAD) {
    RT = isA ? pv.rt[G] : p.rtB;
    KC = isA ? p.kcA_fixed : p.kcB_fixed;
  } else {
    RT = isA ? p.rtA_fixed : p.rtB;
    KC = pv.kc[G];
  }
  const int rt = blockIdx.x;
  const int kc0 = blockIdx.y * kPackKc;
  if (rt >= RT || kc0 >= KC) return;
  const bool wg = p.pass == MXG_PASS_WGRAD;
  const bool kseg = wg || (p.pass == MXG_PASS_DGRAD && !isA);
  __shared__ int32_t pre[kMaxExperts + 1];
  __shared__ int32_t pof[kMaxExperts + 1];
  __shared__ uint32_t tile[128][kPackKc + 1];
  const int tid = threadIdx.x;
  if ((isA && !kseg) || wg) {
    for (int i = tid; i <= G; i += blockDim.x) {
      pre[i] = wg ? pv.kc[i] : pv.rt[i];
      if (wg) pof[i] = pv.poff[i];
    }
    __syncthreads();
  }
  // rows of this tile: [row0 + t*128, row0 + min(R, t*128 + 128))
  int t, R;
  int64_t row0;
  if (!kseg) {
    if (isA) {
      const int g = find_prefix(pre, G, rt);
      t = rt - pre[g];
      row0 = pv.off[g];
      R = pv.off[g + 1] - pv.off[g];
    } else {  // forward weights: G blocks of N rows
      const int g = rt / nrt;
      t = rt - g * nrt;
      row0 = (int64_t)g * p.N;
      R = (int)p.N;
    }
  } else {
    t = rt;
    row0 = 0;
    R = (int)(isA ? p.N : p.K);
  }
  // load phase: thread -> (chunk j = tid % 8, rows tid / 8 + 16 i)
  const int j = tid & (kPackKc - 1);
  const int kcg = kc0 + j;
  int nb = 0;        // valid blocks of the word (0..4)
  int64_t boff = 0;  // byte offset of the word's first block in the row
  if (kcg < KC) {
    int c, KB;
    int64_t kb0;
    if (!kseg) {
      c = kcg;
      kb0 = 0;
      KB = (int)((p.pass == MXG_PASS_FWD ? p.K : p.N) / 32);
    } else if (wg) {
      const int g = find_prefix(pre, G, kcg);
      c = kcg - pre[g];
      kb0 = pof[g] >> 5;
      KB = (pof[g + 1] - pof[g]) >> 5;
    } else {  // dgrad weights: expert g's contraction is columns [g*N, g*N+N)
      const int g = kcg / nrt;
      c = kcg - g * nrt;
      kb0 = (int64_t)g * (p.N >> 5);
      KB = (int)(p.N >> 5);
    }
    nb = max(0, min(4, KB - 4 * c));
    boff = kb0 + 4 * (int64_t)c;
  }
  const bool vec = nb == 4 && ((boff | ps.ld | (int64_t)reinterpret_cast<uintptr_t>(ps.src)) & 3) == 0;
#pragma unroll 4
  for (int i = 0; i < 128 / 16; ++i) {
    const int r = i * 16 + (tid >> 3);
    const int rr = t * 128 + r;
    uint32_t w = 0;
    if (rr < R && nb > 0) {
      const uint8_t* src = ps.src + (row0 + rr) * ps.ld + boff;
      if (vec) {
        w = __ldg(reinterpret_cast<const uint32_t*>(src));
      } else {
        for (int b = 0; b < nb; ++b) w |= (uint32_t)__ldg(src + b) << (8 * b);
      }
    }
    tile[r][j] = w;
  }
  __syncthreads();
  // store phase: chunk word tid holds rows 32*(tid%4) + tid/4 (byte (r%32)*16 + (r/32)*4 + block)
  const int r_of = 32 * (tid & 3) + (tid >> 2);
  const int kc_n = min(KC - kc0, kPackKc);
  for (int jj = 0; jj < kc_n; ++jj) {
    uint32_t* dst = reinterpret_cast<uint32_t*>(ps.dst + ((int64_t)(kc0 + jj) * RT + rt) * kChunkBytes);
    dst[tid] = tile[r_of][jj];
  }
}

// ---------------------------------------------------------------------------
// 3. The GEMM kernel.
// ---------------------------------------------------------------------------
// Shared-memory layout of one CTA.  kCta = 1: the CTA stages a 128-row A tile
// and the whole 256-row B tile of its 128x256 output tile.  kCta = 2: a CTA
// pair computes a 256x256 tile with one MMA stream; each CTA stages its own
// 128 rows of A and one 128-row half of B, so a stage is 32 KB instead of 48
// KB and the ring is deeper.  TMEM: the 256-column accumulator, then one scale
// slot per stage (per 128-element k-chunk, 4 columns for the CTA's 128 A rows
// and 8 for all 256 B rows, in the 32x128b.warpx4 replicated layout).
template <int kKind, int kCta>
struct Cfg {
  using K = KindCfg<kKind>;
  static constexpr int kStages = kCta == 1 ? 4 : (kKind == KIND_MXF4 ? 5 : 6);  // operand ring depth
  static constexpr int kBRows = BN / kCta;  // B rows staged by this CTA
  static constexpr int kBBytes = kBRows * 128;
  static constexpr int kStageBytes = kATileBytes + kBBytes;
  static constexpr int kBChunks = 2;        // 128-row scale chunks of the B tile
  static constexpr int kSfBytes = K::kKPS * kChunkBytes * (1 + kBChunks);
  static constexpr int kDataBytes = kStages * kStageBytes;
  static constexpr int kSfOff = kDataBytes;
  static constexpr int kBarOff = kSfOff + kStages * kSfBytes;
  static constexpr int kNumBars = 4 * kStages + 3;  // full, empty, sready, sgo per stage; tmem_full, tmem_empty, drain
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem addr, abort flag
  // epilogue staging: one buffer per epilogue warp, 1024-byte aligned (swizzle atoms)
  static constexpr int kEpiOff = (kMiscOff + 16 + 1023) & ~1023;
  static constexpr int kTotal = kEpiOff + kEpiWarps * kEpiWarpBytes + 1024;  // + alignment slack
  static_assert(kStageBytes % 1024 == 0, "stage tiles keep the 1024-byte swizzle-atom alignment");
  static_assert(kSfBytes % 512 == 0, "scale stages keep chunk (and 128-byte TMA) alignment");
  static_assert(kTotal <= 232448, "fits the 227 KB of dynamic shared memory of one CTA");
  static_assert(kSfTmemCol0 + kStages * K::kSlotCols <= kStashCol, "the scale slots end before the FP32 stash columns");
};

// FP32 output: one 32-column chunk of a row, stored with 32-byte accesses,
// or added in place with 16-byte reductions at L2 (the thread does not wait
// for the old values, so the accumulator is released sooner).
MXG_DEVINL void store_row_chunk_f32(const Params& p, int64_t row, int64_t col, uint32_t* r) {
  float* dst = static_cast<float*>(p.out) + row * p.ld_out + col;
  if (p.accumulate) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      ptx::red_add_v4_f32(dst + 4 * i, __uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                          __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) ptx::st_global_v8(dst + 8 * i, r + 8 * i);
}

MXG_DEVINL uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<const uint32_t*>(&b);
}

// kCta = 2 (launched as clusters of two CTAs): the even CTA of the pair
// issues tcgen05.mma.cta_group::2 with M = 256 (its TMEM and A rows hold tile
// rows 0-127, the odd CTA's rows 128-255) over B rows split between the two
// CTAs' stages; both CTAs load their own operands and scales, their feeders
// fill their own TMEM scale slots (A: the CTA's 128 rows; B: all 256 rows),
// and their epilogues write their own 128 rows.  Hand-over: the even CTA's
// issuer waits for the feeders and epilogues of both CTAs (remote arrivals on
// its own sready / tmem_empty barriers) and commits every stage and every
// accumulator to the barriers of both CTAs at once.
template <int kKind, int kCta>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_mx_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmOut,
                           const __grid_constant__ CUtensorMap tmOut32,
                           const __grid_constant__ CUtensorMap tmSA,
                           const __grid_constant__ CUtensorMap tmSB, const Params p) {
  using KC = KindCfg<kKind>;
  using L = Cfg<kKind, kCta>;
  constexpr int kStages = L::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.G;
  // the CTA's rank in its pair, and the tile walker's index / count (a pair walks together)
  const uint32_t rank = kCta == 2 ? ptx::cluster_ctarank() : 0u;
  const int unit = kCta == 2 ? (int)ptx::cluster_id_x() : (int)blockIdx.x;
  const int units = kCta == 2 ? (int)ptx::nclusters_x() : (int)gridDim.x;

  const PlanView pv = plan_view(const_cast<int32_t*>(p.plan), G);
  if (pv.hdr[0] == 0) return;  // invalid splits: nothing is written
  const int total_tiles = pv.hdr[1];
  if (unit >= total_tiles) return;  // the same decision in both CTAs of a pair

  // per-expert tables: read in place from the plan (a few loads per tile and role)
  const int32_t* t_off = pv.off;
  const int32_t* t_rt = pv.rt;
  const int32_t* t_poff = pv.poff;
  const int32_t* t_kc = pv.kc;
  const int32_t* t_tiles = pv.tiles;
  const uint32_t bar0 = sbase + L::kBarOff;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto sready_bar = [&](int s) { return bar0 + 8u * (2 * kStages + s); };  // scales in TMEM
  auto sgo_bar = [&](int s) { return bar0 + 8u * (3 * kStages + s); };     // stage armed: load its scales
  const uint32_t tmem_full = bar0 + 8u * (4 * kStages);
  const uint32_t tmem_empty = tmem_full + 8;
  const uint32_t drain_bar = tmem_full + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  // arrive on the issuing CTA's barrier (the even CTA of a pair)
  auto arrive_issuer = [&](uint32_t bar) {
    if constexpr (kCta == 2) ptx::mbar_arrive_cluster(ptx::mapa_shared(bar, 0));
    else ptx::mbar_arrive(bar);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(full_bar(s), 1);
      ptx::mbar_init(empty_bar(s), 1);
      ptx::mbar_init(sready_bar(s), 4 * kCta);  // the feeder warps of every CTA of the group
      ptx::mbar_init(sgo_bar(s), 1);
    }
    ptx::mbar_init(tmem_full, 1);
    ptx::mbar_init(tmem_empty, 4 * kCta);       // the epilogue warps of every CTA of the group
    ptx::mbar_init(drain_bar, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    ptx::prefetch_tmap(&tmOut);
    ptx::prefetch_tmap(&tmOut32);
    ptx::prefetch_tmap(&tmSB);
    if (p.a_scale_tma) ptx::prefetch_tmap(&tmSA);
  }
  if (warp == 1) {
    ptx::tmem_alloc_g<kCta>(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish_g<kCta>();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // the peer's barriers are initialised before any remote arrival or commit reaches them
  if constexpr (kCta == 2) ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // tile -> expert g, this CTA's 128-row m-tile mt, n-tile nt
  auto locate = [&](int tile, int& g, int& mt, int& nt, Geo& e) {
    g = find_prefix(t_tiles, G, tile);
    e = group_geo(p, t_off, t_rt, t_poff, t_kc, g);
    const int ntn = cdiv_d(e.Nn, BN);
    int mg;
    tile_mn(tile - t_tiles[g], t_tiles[g + 1] - t_tiles[g], ntn, p.group_m, mg, nt);
    mt = mg * kCta + (int)rank;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Per stage: the A and B tiles (TMA), and the expected byte count of the
    // whole stage -- tiles and scale chunks, which warp 10 loads onto the same
    // barrier (a copy issue costs the issuing thread ~100 clocks, and five of
    // them per stage took one thread longer than the stage's MMAs).
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_phase = 0;  // per stage: a load was issued / its phase
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += units) {
        int g, mt, nt;
        Geo e;
        locate(tile, g, mt, nt, e);
        const int nk = cdiv_d(e.Kc, KC::kStageK);
        // The odd CTA of a pair whose rows lie past the expert loads no A
        // (its rows are computed from stale data and never stored; their
        // scale chunk may not exist).
        const bool a_in = mt * BM < e.M;
        const int ya = (int)(e.a_row0 + (int64_t)mt * BM);
        const int yb = (int)(e.b_row0 + (int64_t)nt * BN + (int64_t)rank * L::kBRows);
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          const int kc_valid = min(KC::kKPS, cdiv_d(e.Kc - kb * KC::kStageK, 128));
          // The 4-bit-unpacking load of the a8w4 weight tile counts the packed
          // source bytes (64 per row), although it fills 128 bytes per row.
          constexpr uint32_t kBTx = kKind == KIND_A8W4 ? L::kBBytes / 2 : L::kBBytes;
          const uint32_t a_sf = !a_in ? 0u : p.a_scale_tma ? KC::kKPS * kChunkBytes : kc_valid * kChunkBytes;
          const uint32_t bytes = (a_in ? kATileBytes : 0) + kBTx + a_sf + KC::kKPS * L::kBChunks * kChunkBytes;
          const uint32_t fb = full_bar(stage);
          ptx::mbar_arrive_expect_tx(fb, bytes);
          ptx::mbar_arrive(sgo_bar(stage));  // warp 10 loads the stage's scales
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          const uint32_t sA = sbase + stage * L::kStageBytes;
          const uint32_t sB = sA + kATileBytes;
          const int64_t ka = e.a_k0 + (int64_t)kb * KC::kStageK;
          const int64_t kbk = e.b_k0 + (int64_t)kb * KC::kStageK;
          const int xa = kKind == KIND_MXF4 ? (int)(ka >> 1) : (int)ka;
          const int xb = kKind == KIND_MXF4 ? (int)(kbk >> 1) : (int)kbk;
          if (a_in) ptx::tma_load_2d(sA, &tmA, xa, ya, fb);
          ptx::tma_load_2d(sB, &tmB, xb, yb, fb);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // do not leave copies in flight: wait (bounded) for every armed stage
      for (int s = 0; s < kStages; ++s)
        if ((armed >> s) & 1u) {
          volatile int no_abort = 0;
          ptx::mbar_wait(full_bar(s), (armed_phase >> s) & 1u, &no_abort, p.status, p.drain_ns);
        }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && rank == 0) {
      int stage = 0, tcount = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool issued = false;
      for (int tile = unit; tile < total_tiles && ok; tile += units) {
        int g, mt, nt;
        Geo e;
        locate(tile, g, mt, nt, e);
        // every epilogue warp of the group has read the previous accumulator
        if (!ptx::mbar_wait(tmem_empty, (uint32_t)(tcount & 1) ^ 1u, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t dacc = tmem;
        const int nk = cdiv_d(e.Kc, KC::kStageK);
        for (int kb = 0; kb < nk; ++kb) {
          // the stage's data has landed and the feeders have put its scales in TMEM (every CTA)
          if (!ptx::mbar_wait(sready_bar(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          ptx::tc_fence_after();
          const int rem = e.Kc - kb * KC::kStageK;
          const int steps = min(4, cdiv_d(rem, KC::kMmaK));
          const uint32_t sA = sbase + stage * L::kStageBytes;
          const uint32_t sB = sA + kATileBytes;
          const uint32_t tsf = tmem + kSfTmemCol0 + stage * KC::kSlotCols;  // A: kKPS*4 cols, then B
          const uint64_t adesc0 = ptx::smem_desc(sA, 16, 1024, 2);
          const uint64_t bdesc0 = ptx::smem_desc(sB, 16, 1024, 2);
          // unrolled (straight-line issue); the steps past a K tail are skipped
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (j < steps) {
              constexpr int kMmaK = KC::kMmaK;
              const int kel = j * kMmaK;  // element offset inside the stage
              const int c = kel >> 7;
              const uint32_t sfid = (uint32_t)((kel & 127) >> 5);
              const uint32_t idesc = p.idesc | (sfid << 4) | (sfid << 29);
              const uint64_t adv = (uint64_t)((j * 32) >> 4);  // 32 bytes of K per MMA
              const uint32_t sfa = tsf + 4 * c;
              const uint32_t sfb = tsf + KC::kKPS * 4 + 8 * c;
              if constexpr (kKind == KIND_MXF4)
                ptx::mma_mxf4_g<kCta>(dacc, adesc0 + adv, bdesc0 + adv, idesc, sfa, sfb, (kb | j) != 0);
              else
                ptx::mma_mxf8f6f4_g<kCta>(dacc, adesc0 + adv, bdesc0 + adv, idesc, sfa, sfb, (kb | j) != 0);
            }
          }
          issued = true;
          ptx::tc_commit_pair<kCta>(empty_bar(stage));
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        ptx::tc_commit_pair<kCta>(tmem_full);
        ++tcount;
      }
      if (issued) {  // every MMA (both CTAs' halves) has retired before TMEM is released
        ptx::tc_commit_g<kCta>(drain_bar);
        volatile int no_abort = 0;
        ptx::mbar_wait(drain_bar, 0, &no_abort, p.status, p.drain_ns);
      }
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------ scale loads
    // Per stage, once warp 0 has armed the stage's full barrier with the
    // stage's whole byte count (so that warp 0's final wait on every armed
    // stage covers these copies too): the B scale chunks of the stage's k-chunks (one TMA load of
    // whole 512-byte chunks through a map over the packed scales), and the A
    // scale chunks -- one TMA load when the A operand's row-tile count is
    // fixed (wgrad), otherwise one bulk copy per k-chunk (the row-tile count
    // of a row-segmented A is only known on the device).  Chunks past the
    // operand are zero-filled; chunks of a neighbouring expert or a k tail
    // carry scales that no stored output uses.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      const int rtA = p.pass == MXG_PASS_WGRAD ? p.rtA_fixed : pv.rt[G];
      bool ok = true;
      for (int tile = unit; tile < total_tiles && ok; tile += units) {
        int g, mt, nt;
        Geo e;
        locate(tile, g, mt, nt, e);
        const int nk = cdiv_d(e.Kc, KC::kStageK);
        const bool a_in = mt * BM < e.M;
        const int qb = e.b_rt0 + ((nt * BN) >> 7);  // the B tile's first 128-row scale chunk
        const uint8_t* srcA0 = p.packA + ((int64_t)e.a_kc0 * rtA + e.a_rt0 + mt) * kChunkBytes;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(sgo_bar(stage), phase, abort_flag, p.status, p.timeout_ns)) { ok = false; break; }
          const int kc_valid = min(KC::kKPS, cdiv_d(e.Kc - kb * KC::kStageK, 128));
          const uint32_t fb = full_bar(stage);
          const uint32_t sf = sbase + L::kSfOff + stage * L::kSfBytes;
          const int kc0 = kb * KC::kKPS;
          // B scales: chunks (kc, qb .. qb+1) for the stage's k-chunks, kc-major
          ptx::tma_load_3d(sf + KC::kKPS * kChunkBytes, &tmSB, 0, qb, e.b_kc0 + kc0, fb);
          if (a_in) {
            if (p.a_scale_tma) {
              ptx::tma_load_3d(sf, &tmSA, 0, e.a_rt0 + mt, e.a_kc0 + kc0, fb);
            } else {
              for (int c = 0; c < kc_valid; ++c)
                ptx::bulk_load(sf + c * kChunkBytes, srcA0 + (int64_t)(kc0 + c) * rtA * kChunkBytes, kChunkBytes, fb);
            }
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ scale feeders
    // A stage's scale chunks (the A chunk of each k-chunk, then the two B
    // chunks of each k-chunk) go to the stage's TMEM scale slot, every lane of
    // this warp's quarter receiving the 16 bytes that tcgen05.cp
    // 32x128b.warpx4 would have given it: A chunk c to columns 4c..4c+3, the
    // two B chunks of k-chunk c to the next 8 columns.  Words of chunks past
    // the operand, a neighbouring expert or a k tail carry scales into columns
    // that no MMA reads for a stored output.
    const int quarter = warp & 3;
    const uint32_t tq = tmem + ((uint32_t)(quarter * 32) << 16) + kSfTmemCol0;
    const uint8_t* sf_lane = smem + L::kSfOff + lane * 16;
    int stage = 0;
    uint32_t phase = 0;
    for (int tile = unit; tile < total_tiles; tile += units) {
      int g, mt, nt;
      Geo e;
      locate(tile, g, mt, nt, e);
      const int nk = cdiv_d(e.Kc, KC::kStageK);
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        const bool landed = ptx::mbar_wait(full_bar(stage), phase, abort_flag, p.status, p.timeout_ns);
        if (!__all_sync(0xffffffffu, landed)) { ok = false; break; }
        const uint8_t* src = sf_lane + stage * L::kSfBytes;
        const uint32_t dst = tq + stage * KC::kSlotCols;
#pragma unroll
        for (int c = 0; c < KC::kKPS; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(src + c * kChunkBytes);
          ptx::tmem_st_32x32b_x4(dst + 4 * c, v.x, v.y, v.z, v.w);
        }
#pragma unroll
        for (int c = 0; c < KC::kKPS; ++c) {
          const uint8_t* bsrc = src + (KC::kKPS + c * L::kBChunks) * kChunkBytes;
          const uint4 v0 = *reinterpret_cast<const uint4*>(bsrc);
          const uint4 v1 = *reinterpret_cast<const uint4*>(bsrc + kChunkBytes);
          const uint32_t o[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          ptx::tmem_st_32x32b_x8(dst + 4 * KC::kKPS + 8 * c, o);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_issuer(sready_bar(stage));
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5)
    // Warp q owns TMEM lane quarter q: rows q*32 .. q*32+31 of the tile.  The
    // output goes out through the warp's staging buffer: two 16-row boxes of
    // 128 bytes per row (64 BF16 / 32 FP32 columns) in the TMA 128-byte
    // swizzle, written to global memory by tiled bulk stores -- bulk
    // reduce-adds when accumulating -- issued by lane 0, so that the tile
    // leaves the SM as whole lines instead of one 32-byte piece per row and
    // lane.  A box only partly inside the expert's rows is written by the
    // lanes of its valid rows directly; columns past the output's last are
    // clipped by the map.  TMEM is handed back right after its last read:
    // BF16 copies the second half of its row into TMEM columns that no MMA or
    // scale slot uses and reads the first half into registers as packed
    // pairs; FP32 copies the second half the same way and keeps the first
    // half in registers; either then hands back and writes both halves out
    // while the next tile's MMAs run.
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const uint32_t tlane0 = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t ebuf = sbase + (uint32_t)(L::kEpiOff + quarter * kEpiWarpBytes);
    const int brow = lane & 15;                                  // row inside this lane's box
    const uint32_t my_off = (uint32_t)((lane >> 4) * kEpiBoxBytes + brow * 128);
    int tcount = 0;
    bool pending = false;  // lane 0: bulk groups issued
    // stage this lane's 128-byte row piece v[0..31] and send the full boxes
    auto send = [&](const uint32_t* v, int64_t x, int64_t y0, bool full0, bool full1, bool reduce) {
      // the buffer's previous contents have been read
      if (lane == 0 && pending) ptx::bulk_wait_group_read<0>();
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 8; ++k)
        ptx::st_shared_v4(ebuf + my_off + (uint32_t)((k ^ (brow & 7)) << 4), v[4 * k], v[4 * k + 1],
                          v[4 * k + 2], v[4 * k + 3]);
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0 && (full0 || full1)) {
        // both boxes inside the expert: one 32-row box (the same rows in the same swizzle)
        const void* map = full1 ? (const void*)&tmOut32 : (const void*)&tmOut;
        if (reduce) ptx::tma_reduce_add_2d(map, ebuf, (int)x, (int)y0);
        else ptx::tma_store_2d(map, ebuf, (int)x, (int)y0);
        ptx::bulk_commit_group();
        pending = true;
      }
    };
    for (int tile = unit; tile < total_tiles; tile += units) {
      int g, mt, nt;
      Geo e;
      locate(tile, g, mt, nt, e);
      const bool ready = ptx::mbar_wait(tmem_full, (uint32_t)(tcount & 1), abort_flag, p.status, p.timeout_ns);
      if (!__all_sync(0xffffffffu, ready)) break;  // the warp leaves together (.aligned TMEM loads)
      ptx::tc_fence_after();
      const uint32_t tlane = tlane0;
      auto release = [&]() {
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_issuer(tmem_empty);
      };
      const int row0 = mt * BM + quarter * 32;  // the warp's first row inside the expert
      const int row = row0 + lane;
      const bool row_ok = row < e.M;
      const int64_t orow = e.out_row0 + row;
      const int64_t oy0 = e.out_row0 + row0;
      const int ncols = min(BN, e.Nn - nt * BN);  // multiple of 32
      const int64_t col0 = (int64_t)nt * BN;
      const int vrows = e.M - row0;               // the warp's rows inside the expert (may be <= 0)
      const bool full0 = vrows >= kEpiBoxRows, full1 = vrows >= 2 * kEpiBoxRows;
      const bool direct = row_ok && !((lane >> 4) == 0 ? full0 : full1);  // partial box: own store
      const bool skip_out = vrows <= 0 || (e.Kc == 0 && p.accumulate);   // nothing of this warp to write
      const int nch = ncols / 32;
      // 32 fp32 columns c of the accumulator (zeros for an empty contraction)
      auto read_chunk = [&](uint32_t taddr, uint32_t* r) {
        if (e.Kc > 0) {
          __syncwarp();
          ptx::tmem_ld_32x32b_x32(taddr, r);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0;
        }
      };
      if (p.out_dtype == MXG_OUT_BF16) {
        // Hand-off: accumulator columns 128..255 are copied to the stash columns
        // and columns 0..127 read and packed into registers, 64 columns (two
        // loads) per load wait; TMEM is then handed back and the write-out
        // overlaps the next tile's MMAs.  The store wait sits before the
        // second half's loads: the compiler holds a tcgen05.st's source
        // registers until it, and after the hand-back they would spill.  An
        // empty contraction never wrote the accumulator: its output is zeros
        // and the stash is unused.
        constexpr int kHalf = BN / 2;
        uint32_t hb[kHalf / 2];  // columns 0..127 of this lane's row as packed BF16 pairs
        if (e.Kc > 0) {
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t f[64];
            ptx::tmem_ld_32x32b_x32(tlane + (uint32_t)(kHalf + q * 64), f);
            ptx::tmem_ld_32x32b_x32(tlane + (uint32_t)(kHalf + q * 64 + 32), f + 32);
            ptx::tmem_ld_wait();
            ptx::tmem_st_32x32b_x32(tlane0 + (uint32_t)(kStashCol + q * 64), f);
            ptx::tmem_st_32x32b_x32(tlane0 + (uint32_t)(kStashCol + q * 64 + 32), f + 32);
          }
          ptx::tmem_st_wait();
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t f[64];
            ptx::tmem_ld_32x32b_x32(tlane + (uint32_t)(q * 64), f);
            ptx::tmem_ld_32x32b_x32(tlane + (uint32_t)(q * 64 + 32), f + 32);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) hb[q * 32 + i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < kHalf / 2; ++i) hb[i] = 0;
        }
        release();
        if (!skip_out) {
          __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + orow * p.ld_out + col0;
          auto out64 = [&](int c4, const uint32_t* h) {  // 64 columns as packed BF16 pairs, staged and sent
            send(h, col0 + c4 * 64, oy0, full0, full1, false);
            if (direct) {  // this lane's row, written by the lane itself
              ptx::st_global_v8(dst + c4 * 64, h);
              ptx::st_global_v8(dst + c4 * 64 + 16, h + 8);
              if (c4 * 64 + 32 < ncols) {
                ptx::st_global_v8(dst + c4 * 64 + 32, h + 16);
                ptx::st_global_v8(dst + c4 * 64 + 48, h + 24);
              }
            }
          };
#pragma unroll
          for (int c4 = 0; c4 < kHalf / 64; ++c4)
            if (c4 * 64 < ncols) out64(c4, hb + c4 * 32);  // warp-uniform
#pragma unroll 1
          for (int c4 = kHalf / 64; c4 < BN / 64; ++c4) {
            if (c4 * 64 < ncols) {
              uint32_t r[64];
              if (e.Kc > 0) {
                __syncwarp();
                ptx::tmem_ld_32x32b_x32(tlane0 + (uint32_t)(kStashCol + (2 * c4 - kHalf / 32) * 32), r);
                ptx::tmem_ld_32x32b_x32(tlane0 + (uint32_t)(kStashCol + (2 * c4 + 1 - kHalf / 32) * 32), r + 32);
                ptx::tmem_ld_wait();
              } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) r[i] = 0;
              }
              uint32_t h[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) h[i] = pack_bf16x2(r[2 * i], r[2 * i + 1]);
              out64(c4, h);
            }
          }
        }
      } else {
        // Columns 128..255 are copied into the spare TMEM columns, 0..127 are
        // read into registers, and the accumulator is handed back before any
        // output is written: the next tile's MMAs overlap the write-out.
        uint32_t h[BN / 2];
#pragma unroll
        for (int c = BN / 64; c < BN / 32; ++c) {
          if (c < nch && e.Kc > 0) {  // warp-uniform
            uint32_t r[32];
            read_chunk(tlane + (uint32_t)(c * 32), r);
            ptx::tmem_st_32x32b_x32(tlane0 + (uint32_t)(kStashCol + (c - BN / 64) * 32), r);
          }
        }
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) {
          if (c < nch) {
            uint32_t r[32];
            read_chunk(tlane + (uint32_t)(c * 32), r);
#pragma unroll
            for (int i = 0; i < 32; ++i) h[c * 32 + i] = r[i];
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) h[c * 32 + i] = 0;
          }
        }
        release();
        if (nch > BN / 64 && e.Kc > 0) ptx::tmem_st_wait();  // the stash is complete before it is read
        if (!skip_out) {
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) {
            if (c < nch) {
              send(&h[c * 32], col0 + c * 32, oy0, full0, full1, p.accumulate != 0);
              if (direct) store_row_chunk_f32(p, orow, col0 + c * 32, &h[c * 32]);
            }
          }
          for (int c = BN / 64; c < nch; ++c) {
            uint32_t r[32];
            if (e.Kc > 0) {
              __syncwarp();
              ptx::tmem_ld_32x32b_x32(tlane0 + (uint32_t)(kStashCol + (c - BN / 64) * 32), r);
              ptx::tmem_ld_wait();
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = 0;
            }
            send(r, col0 + c * 32, oy0, full0, full1, p.accumulate != 0);
            if (direct) store_row_chunk_f32(p, orow, col0 + c * 32, r);
          }
        }
      }
      ++tcount;
    }
    // every bulk store has completed before the CTA ends
    if (lane == 0 && pending) ptx::bulk_wait_group0();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  // Neither CTA of a pair leaves (or releases TMEM) while the other may still
  // arrive on its barriers; the issuer's drain above has retired every MMA.
  if constexpr (kCta == 2) ptx::cluster_sync();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc_g<kCta>(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
struct PackSizes {
  int64_t rtA, kcA, rtB, kcB;  // upper bounds (chunks)
};

PackSizes pack_sizes(int pass, int G, int64_t S, int64_t N, int64_t K, int pad) {
  PackSizes s;
  const int64_t rt_rows = (S + (int64_t)G * (BM - 1)) / BM;  // >= sum ceil(m_g/128)
  if (pass == MXG_PASS_FWD) {
    s.rtA = rt_rows; s.kcA = cdiv(K, 128);
    s.rtB = G * cdiv(N, 128); s.kcB = cdiv(K, 128);
  } else if (pass == MXG_PASS_DGRAD) {
    s.rtA = rt_rows; s.kcA = cdiv(N, 128);
    s.rtB = cdiv(K, 128); s.kcB = G * cdiv(N, 128);
  } else {  // S = column capacity of the padded operands
    const int64_t kc = S / 128 + G;  // >= sum ceil(p_g/128) whenever sum p_g <= S
    s.rtA = cdiv(N, 128); s.kcA = kc;
    s.rtB = cdiv(K, 128); s.kcB = kc;
  }
  (void)pad;
  return s;
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct KernelInfo {
  const void* fn;
  int smem;
};

template <int kKind>
KernelInfo kernel_info_kind(int cta) {
  if (cta == 2) return {(const void*)grouped_mx_gemm_kernel<kKind, 2>, Cfg<kKind, 2>::kTotal};
  return {(const void*)grouped_mx_gemm_kernel<kKind, 1>, Cfg<kKind, 1>::kTotal};
}

KernelInfo kernel_info(int kind, int cta) {
  switch (kind) {
    case KIND_MXF4: return kernel_info_kind<KIND_MXF4>(cta);
    case KIND_A8W4: return kernel_info_kind<KIND_A8W4>(cta);
    default: return kernel_info_kind<KIND_MXF8>(cta);
  }
}

constexpr int kMaxDevices = 64;
std::mutex g_attr_mu;

// The dynamic shared-memory opt-in, once per (device, kind, CTA group).
bool ensure_smem_attr(const KernelInfo& ki, int kind, int cta, int dev) {
  static bool done[kMaxDevices][3][2] = {};
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (dev >= 0 && dev < kMaxDevices && done[dev][kind][cta - 1]) return true;
  if (cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (dev >= 0 && dev < kMaxDevices) done[dev][kind][cta - 1] = true;
  return true;
}

// Number of CTA pairs of the 2-SM kernel that the device holds at once (one
// CTA per SM), looked up once per (device, kind); 0 when clusters of two
// cannot be scheduled there.
int pair_cluster_count(int kind, int dev) {
  static int cached[kMaxDevices][3];
  static bool have[kMaxDevices][3] = {};
  if (dev < 0 || dev >= kMaxDevices) return 0;
  {
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (have[dev][kind]) return cached[dev][kind];
  }
  const KernelInfo ki = kernel_info(kind, 2);
  int n = 0;
  if (ensure_smem_attr(ki, kind, 2, dev)) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cfg.gridDim = dim3((unsigned)std::max(2, sms - (sms & 1)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)ki.smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, ki.fn, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
  }
  std::lock_guard<std::mutex> lk(g_attr_mu);
  cached[dev][kind] = n;
  have[dev][kind] = true;
  return n;
}

}  // namespace

size_t gemm_workspace_bytes(int pass, int G, int64_t S, int64_t N, int64_t K, int pad) {
  const PackSizes s = pack_sizes(pass, G, S, N, K, pad);
  return plan_bytes(G) + align256((size_t)(s.rtA * s.kcA) * kChunkBytes) +
         align256((size_t)(s.rtB * s.kcB) * kChunkBytes) + 1024;
}

mxg_status launch_grouped_gemm(const GemmArgs& a, cudaStream_t stream, int num_sms) {
  int kind;
  if (a.a_elem == MXG_E2M1 && a.b_elem == MXG_E2M1) kind = KIND_MXF4;
  else if (a.a_elem == MXG_E4M3 && a.b_elem == MXG_E2M1) kind = KIND_A8W4;
  else if (a.a_elem == MXG_E4M3 && a.b_elem == MXG_E4M3) kind = KIND_MXF8;
  else return MXG_ERR_UNSUPPORTED;
  if (a.total_rows > 0x7FFFFFFF || a.N > 0x7FFFFFFF || a.K > 0x7FFFFFFF) return MXG_ERR_SHAPE;

  const int64_t S = a.pass == MXG_PASS_WGRAD ? a.a_cols : a.total_rows;
  const PackSizes ps = pack_sizes(a.pass, a.G, S, a.N, a.K, a.pad);
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  uint8_t* packA = ws + plan_bytes(a.G);
  uint8_t* packB = packA + align256((size_t)(ps.rtA * ps.kcA) * kChunkBytes);
  // operands quantized with packed scales are read in place
  if (a.a_packed) packA = const_cast<uint8_t*>(a.a_scale);
  if (a.b_packed) packB = const_cast<uint8_t*>(a.b_scale);

  Params p{};
  p.pass = a.pass;
  p.G = a.G;
  p.accumulate = a.accumulate;
  p.out_dtype = a.out_dtype;
  p.S = a.total_rows;
  p.N = a.N;
  p.K = a.K;
  p.cap = a.a_cols;
  p.pad = a.pad;
  p.rtA_fixed = (int)cdiv(a.N, 128);
  p.rtB = (int)ps.rtB;
  p.kcA_fixed = (int)(a.pass == MXG_PASS_FWD ? cdiv(a.K, 128) : cdiv(a.N, 128));
  p.kcB_fixed = (int)(a.pass == MXG_PASS_FWD ? cdiv(a.K, 128) : a.G * cdiv(a.N, 128));
  p.plan = reinterpret_cast<const int32_t*>(ws);
  p.packA = packA;
  p.packB = packB;
  p.out = a.out;
  p.ld_out = a.ld_out;
  p.status = a.status;
  p.timeout_ns = wait_timeout_ns();
  p.drain_ns = std::max<uint64_t>(p.timeout_ns, 200000000ull);
  int dev = 0;
  cudaGetDevice(&dev);
  // contraction length of the A rows (wgrad: the mean expert's padded tokens)
  const int64_t kc_len = a.pass == MXG_PASS_FWD ? a.K : a.pass == MXG_PASS_DGRAD ? a.N : a.a_cols / a.G;
  // CTA pairs (2-SM MMA) unless the caller chose the one-SM kernel or the
  // device cannot co-schedule pairs
  const int pair_clusters = gemm_cta_group() == 2 ? pair_cluster_count(kind, dev) : 0;
  const int cta = pair_clusters > 0 ? 2 : 1;
  p.bn = BN;
  p.tile_m = BM * cta;
  {  // bytes of one A row along the contraction
    const double eb = kind == KIND_MXF4 ? 0.5 : 1.0;
    p.group_m = std::max(1, tile_group_m((double)kc_len * eb) / cta);  // in scheduled tiles of BM * cta rows
  }

  // instruction descriptor: dense, K-major A and B, UE8M0 scales, M = 128 per
  // CTA (256 for a pair), N = 256
  uint32_t at = kind == KIND_MXF4 ? 1u : 0u;
  uint32_t bt = kind == KIND_MXF4 ? 1u : (kind == KIND_A8W4 ? 5u : 0u);
  p.idesc = (at << 7) | (bt << 10) | ((uint32_t)(BN >> 3) << 17) | (1u << 23) |
            ((uint32_t)((BM * cta) >> 4) << 24);

  // 1. plan
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(a.splits, p, reinterpret_cast<int32_t*>(ws));
  if (cudaGetLastError() != cudaSuccess) return MXG_ERR_CUDA;

  // An empty forward / dgrad batch needs only the split validation.
  if (a.pass != MXG_PASS_WGRAD && a.total_rows == 0) return MXG_OK;

  // 2. scale packing (both operands in one launch; none for packed operands)
  if (!(a.a_packed && a.b_packed)) {
    PackSrc sa{a.a_scale, a.a_scale_ld, a.a_packed ? nullptr : packA};
    PackSrc sb{a.b_scale, a.b_scale_ld, a.b_packed ? nullptr : packB};
    const int64_t gx = std::max<int64_t>(1, std::max(a.a_packed ? 0 : ps.rtA, a.b_packed ? 0 : ps.rtB));
    const int64_t gy = std::max<int64_t>(
        1, cdiv(std::max(a.a_packed ? 0 : ps.kcA, a.b_packed ? 0 : ps.kcB), kPackKc));
    if (gy > 65535) return MXG_ERR_SHAPE;
    pack_scales_kernel<<<dim3((unsigned)gx, (unsigned)gy, 2), 128, 0, stream>>>(p, sa, sb);
    if (cudaGetLastError() != cudaSuccess) return MXG_ERR_CUDA;
  }

  // 3. tensor maps + GEMM (each CTA of a pair loads one 128-row half of the B tile)
  const int b_box = BN / cta;
  CUtensorMap tmA, tmB;
  bool ok;
  if (a.a_cols == 0) {
    // wgrad with zero capacity: every expert is empty and no tile loads data;
    // the maps only need to be well formed (over the workspace).
    ok = make_tmap(&tmA, ws, CU_TENSOR_MAP_DATA_TYPE_UINT8, 16, 1, 16, 128, BM) &&
         make_tmap(&tmB, ws, CU_TENSOR_MAP_DATA_TYPE_UINT8, 16, 1, 16, 128, b_box);
  } else if (kind == KIND_MXF4) {
    ok = make_tmap(&tmA, a.a_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a_cols / 2, a.a_rows, a.a_ld, 128, BM) &&
         make_tmap(&tmB, a.b_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.b_cols / 2, a.b_rows, a.b_ld, 128, b_box);
  } else if (kind == KIND_A8W4) {
    ok = make_tmap(&tmA, a.a_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a_cols, a.a_rows, a.a_ld, 128, BM) &&
         make_tmap(&tmB, a.b_data, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, a.b_cols, a.b_rows, a.b_ld, 128, b_box);
  } else {
    ok = make_tmap(&tmA, a.a_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.a_cols, a.a_rows, a.a_ld, 128, BM) &&
         make_tmap(&tmB, a.b_data, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.b_cols, a.b_rows, a.b_ld, 128, b_box);
  }
  if (!ok) return MXG_ERR_CUDA;
  // the output as tiled-store destination: columns = N (fwd) or K, rows = S
  // (fwd, dgrad) or G*N (wgrad); boxes of 16 rows x 128 bytes
  // the packed scales as chunk grids: B always (its row-tile count is fixed),
  // A for wgrad (likewise); a row-segmented A's scales go by bulk copies
  const int kps = kind == KIND_MXF4 ? 2 : 1;  // scale k-chunks per stage
  p.a_scale_tma = a.pass == MXG_PASS_WGRAD ? 1 : 0;
  CUtensorMap tmSA, tmSB;
  if (!make_scale_tmap(&tmSB, packB, ps.rtB, ps.kcB, 2, kps)) return MXG_ERR_CUDA;
  if (p.a_scale_tma) {
    if (!make_scale_tmap(&tmSA, packA, ps.rtA, ps.kcA, 1, kps)) return MXG_ERR_CUDA;
  } else {
    tmSA = tmSB;  // not read
  }
  CUtensorMap tmOut, tmOut32;  // 16-row boxes, and 32-row boxes for warps whose rows are all valid
  {
    const bool f32 = a.out_dtype == MXG_OUT_F32;
    const int64_t ocols = a.pass == MXG_PASS_FWD ? a.N : a.K;
    const int64_t orows = a.pass == MXG_PASS_WGRAD ? (int64_t)a.G * a.N : a.total_rows;
    const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_tmap(&tmOut, a.out, dt, ocols, orows, a.ld_out * (f32 ? 4 : 2), f32 ? 32 : 64, kEpiBoxRows) ||
        !make_tmap(&tmOut32, a.out, dt, ocols, orows, a.ld_out * (f32 ? 4 : 2), f32 ? 32 : 64, 2 * kEpiBoxRows))
      return MXG_ERR_CUDA;
  }

  const KernelInfo ki = kernel_info(kind, cta);
  if (!ensure_smem_attr(ki, kind, cta, dev)) return MXG_ERR_CUDA;
  void* args[] = {(void*)&tmA, (void*)&tmB, (void*)&tmOut, (void*)&tmOut32, (void*)&tmSA, (void*)&tmSB, (void*)&p};
  cudaError_t err;
  if (cta == 1) {
    err = cudaLaunchKernel(ki.fn, dim3((unsigned)num_sms), dim3(kThreads), args, (size_t)ki.smem, stream);
  } else {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(2 * pair_clusters));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)ki.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelExC(&cfg, ki.fn, args);
  }
  if (err != cudaSuccess) {
    cudaGetLastError();
    return MXG_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return MXG_ERR_CUDA;
  return MXG_OK;
}

}  // namespace mxg
