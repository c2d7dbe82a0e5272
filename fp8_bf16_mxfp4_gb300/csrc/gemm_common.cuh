// Pieces shared by the grouped GEMM kernels (MX block-scaled and blockwise
// FP8): per-call plan (split validation + per-expert prefix tables, computed
// on the device), per-expert pass geometry, and tensor-map construction.
#pragma once

#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace mxg {
namespace {

constexpr int kTileM = 128;  // tile rows = TMEM lanes (all GEMM kernels)

// Offsets of the per-expert tables inside the plan (int32 arrays of G+1).
struct PlanView {
  int32_t* hdr;  // [0] valid, [1] total tiles
  int32_t* off;  // prefix of m_g
  int32_t* rt;   // prefix of ceil(m_g/128)
  int32_t* poff; // prefix of p_g = ceil(m_g/pad)*pad
  int32_t* kc;   // prefix of ceil(p_g/128)
  int32_t* tiles;// prefix of tiles per expert
};

constexpr int kPlanHdrInts = 16;
inline size_t plan_bytes(int G) {
  size_t b = (kPlanHdrInts + 5 * (size_t)(G + 1)) * sizeof(int32_t);
  return (b + 255) & ~(size_t)255;
}
__host__ __device__ inline PlanView plan_view(void* ws, int G) {
  PlanView v;
  int32_t* p = static_cast<int32_t*>(ws);
  v.hdr = p;
  v.off = p + kPlanHdrInts;
  v.rt = v.off + (G + 1);
  v.poff = v.rt + (G + 1);
  v.kc = v.poff + (G + 1);
  v.tiles = v.kc + (G + 1);
  return v;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
MXG_DEVINL int cdiv_d(int a, int b) { return (a + b - 1) / b; }

struct Params {
  int pass, G, accumulate, out_dtype;
  int bn;         // tile columns (plan: tiles per expert)
  int64_t S, N, K, cap;
  int pad;
  int rtA_fixed;  // A row tiles when fixed (wgrad: ceil(N/128))
  int rtB;        // B row tiles total (fwd: G*ceil(N/128); dgrad/wgrad: ceil(K/128))
  int kcA_fixed;  // A k-chunks when fixed (fwd: ceil(K/128); dgrad: ceil(N/128))
  int kcB_fixed;  // B k-chunks when fixed (fwd: ceil(K/128); dgrad: G*ceil(N/128))
  const int32_t* plan;
  const uint8_t* packA;
  const uint8_t* packB;
  void* out;
  int64_t ld_out;
  int32_t* status;
  uint64_t timeout_ns;  // every wait of the main loops
  uint64_t drain_ns;    // teardown waits for copies / MMAs still in flight (>= 200 ms)
  uint32_t idesc;
  int group_m;          // m-tiles per group of the tile order (see tile_mn)
  int tile_m;           // rows of one scheduled tile: 128, or 256 for a CTA pair (0 = 128)
  int a_scale_tma;      // A's packed scales have a fixed row-tile count: loaded through a tensor map
};

// Per-expert geometry of one pass (see the table at the top of the file).
struct Geo {
  int64_t a_row0, b_row0, a_k0, b_k0, out_row0;
  int M, Nn, Kc;
  int a_rt0, b_rt0, a_kc0, b_kc0;
};

MXG_DEVINL Geo group_geo(const Params& p, const int32_t* off, const int32_t* rt,
                         const int32_t* poff, const int32_t* kc, int g) {
  Geo e;
  const int nrt = (int)((p.N + 127) / 128);
  if (p.pass == MXG_PASS_FWD) {
    e.a_row0 = off[g]; e.b_row0 = (int64_t)g * p.N; e.a_k0 = 0; e.b_k0 = 0;
    e.M = off[g + 1] - off[g]; e.Nn = (int)p.N; e.Kc = (int)p.K;
    e.a_rt0 = rt[g]; e.b_rt0 = g * nrt; e.a_kc0 = 0; e.b_kc0 = 0;
    e.out_row0 = off[g];
  } else if (p.pass == MXG_PASS_DGRAD) {
    e.a_row0 = off[g]; e.b_row0 = 0; e.a_k0 = 0; e.b_k0 = (int64_t)g * p.N;
    e.M = off[g + 1] - off[g]; e.Nn = (int)p.K; e.Kc = (int)p.N;
    e.a_rt0 = rt[g]; e.b_rt0 = 0; e.a_kc0 = 0; e.b_kc0 = g * nrt;
    e.out_row0 = off[g];
  } else {
    e.a_row0 = 0; e.b_row0 = 0; e.a_k0 = poff[g]; e.b_k0 = poff[g];
    e.M = (int)p.N; e.Nn = (int)p.K; e.Kc = poff[g + 1] - poff[g];
    e.a_rt0 = 0; e.b_rt0 = 0; e.a_kc0 = kc[g]; e.b_kc0 = kc[g];
    e.out_row0 = (int64_t)g * p.N;
  }
  return e;
}

// ---------------------------------------------------------------------------
// 1. Plan: split validation + prefix tables (one CTA of 256 threads, two
//    experts per thread).
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 256;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ splits,
                                                            Params p, int32_t* plan_ws) {
  PlanView pv = plan_view(plan_ws, p.G);
  __shared__ int64_t wsum[8][5];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int G = p.G;
  const int nt_n = p.pass == MXG_PASS_FWD ? (int)cdiv_d((int)p.N, p.bn) : (int)cdiv_d((int)p.K, p.bn);
  const int tm = p.tile_m > 0 ? p.tile_m : kTileM;  // scheduled tile rows (scale row tiles stay 128)
  const int wg_tiles = (int)(cdiv_d((int)p.N, tm) * cdiv_d((int)p.K, p.bn));
  int64_t v[2][5];
  bool neg = false;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int g = 2 * tid + i;
    // no splits: one expert of all S rows (the dense entry point)
    const int64_t m = g < G ? (splits ? (int64_t)splits[g] : p.S) : 0;
    neg |= m < 0;
    const int64_t mm = m > 0 ? m : 0;
    const int64_t pg = p.pass == MXG_PASS_WGRAD ? ((mm + p.pad - 1) / p.pad) * p.pad : 0;
    v[i][0] = m;
    v[i][1] = (mm + kTileM - 1) / kTileM;
    v[i][2] = pg;
    v[i][3] = (pg + 127) / 128;
    if (g >= G) v[i][4] = 0;
    else if (p.pass == MXG_PASS_WGRAD) v[i][4] = (pg > 0 || !p.accumulate) ? wg_tiles : 0;
    else v[i][4] = ((mm + tm - 1) / tm) * nt_n;
  }
  int64_t incl[5];
#pragma unroll
  for (int q = 0; q < 5; ++q) {
    int64_t s = v[0][q] + v[1][q];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t o = __shfl_up_sync(0xffffffffu, s, d);
      if (lane >= d) s += o;
    }
    incl[q] = s;
    if (lane == 31) wsum[wid][q] = s;
  }
  const int any_neg = __syncthreads_or(neg);
  int32_t* tabs[5] = {pv.off, pv.rt, pv.poff, pv.kc, pv.tiles};
  __shared__ int64_t totals[5];
#pragma unroll
  for (int q = 0; q < 5; ++q) {
    int64_t base = 0;
    for (int w = 0; w < wid; ++w) base += wsum[w][q];
    const int64_t ex = base + incl[q] - (v[0][q] + v[1][q]);
    if (2 * tid <= G) tabs[q][2 * tid] = (int32_t)ex;
    if (2 * tid + 1 <= G) tabs[q][2 * tid + 1] = (int32_t)(ex + v[0][q]);
    if (tid == kPlanThreads - 1) {
      // the total, entry G: for G = 2 * kPlanThreads no pair above reaches it
      totals[q] = base + incl[q];
      tabs[q][G] = (int32_t)(base + incl[q]);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int bad = 0;
    if (any_neg || totals[0] != p.S) bad = MXG_ERR_SPLITS;
    else if (p.pass == MXG_PASS_WGRAD && totals[2] > p.cap) bad = MXG_ERR_CAPACITY;
    else if (totals[4] > 0x7FFFFFFF) bad = MXG_ERR_SHAPE;
    if (bad) report(p.status, bad);
    pv.hdr[0] = bad ? 0 : 1;
    pv.hdr[1] = bad ? 0 : (int32_t)totals[4];
  }
}

// Tile order inside an expert: groups of `group_m` m-tiles; inside a group m
// runs fastest and n outer, so CTAs running at the same time share a B tile
// and the group's A rows stay in L2 across all of its n-tiles (B is then read
// once per group instead of once per m-tile).
MXG_DEVINL void tile_mn(int local, int expert_tiles, int ntn, int group_m, int& mt, int& nt) {
  const int mtn = expert_tiles / ntn;
  const int span = group_m * ntn;
  const int grp = local / span;
  const int first = grp * group_m;
  const int rows = min(group_m, mtn - first);
  const int idx = local - grp * span;
  mt = first + idx % rows;
  nt = idx / rows;
}

// Host: group size that keeps about 32 MiB of A rows (128-row strips of
// `a_row_bytes` each) resident.
inline int tile_group_m(double a_row_bytes) {
  const double strip = 128.0 * (a_row_bytes > 1.0 ? a_row_bytes : 1.0);
  const double g = (32.0 * 1024 * 1024) / strip;
  return g < 1.0 ? 1 : (g > 4096.0 ? 4096 : (int)g);
}

MXG_DEVINL int find_prefix(const int32_t* pre, int G, int x) {  // last g with pre[g] <= x
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}


// ---------------------------------------------------------------------------
// Host: tensor maps (driver entry point looked up through the runtime, so the
// library does not link libcuda).
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

// 3-D map over a packed scale buffer: chunks of 128 32-bit words (512 bytes),
// `rt` chunks per k-chunk row, `kc` k-chunk rows; box = `box_rt` x `box_kc`
// whole chunks; no swizzle.
bool make_scale_tmap(CUtensorMap* m, const void* base, int64_t rt, int64_t kc, int box_rt, int box_kc) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, (cuuint64_t)(rt > 0 ? rt : 1), (cuuint64_t)(kc > 0 ? kc : 1)};
  cuuint64_t strides[2] = {512, (cuuint64_t)(rt > 0 ? rt : 1) * 512};
  cuuint32_t box[3] = {128, (cuuint32_t)box_rt, (cuuint32_t)box_kc};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D K-major operand map: inner extent `inner` (in elements of `dt`), `rows`
// rows at `ld_bytes`; box = `box_inner` x `box_rows`; 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int64_t inner,
               int64_t rows, int64_t ld_bytes, int box_inner, int box_rows) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)(rows > 0 ? rows : 1)};
  cuuint64_t strides[1] = {(cuuint64_t)ld_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


}  // namespace
}  // namespace mxg
