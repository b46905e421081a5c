// Tiled GEMM on the 5th-generation tensor cores for token counts that make
// the products bound by the tensor cores rather than by the weight stream
// (the whole-prompt context projection; the LM head of a large batch).
//
// Y[rows, N] = A[rows, K] W[N, K]^T.  Persistent CTAs (one per SM) in
// clusters of two walk pairs of 128 x BN output tiles (token rows x
// features) that share their feature range, in a banded raster order (8 pairs
// of row tiles per band, so the clusters of one wave share weight and token
// tiles in L2).  The cluster only places the two CTAs of a pair on one GPC:
// each CTA's TMA pipeline stages its own 128 x 64 token box and the whole
// BN x 64 weight box (two boxes of BN/2 rows), so the pair's second read of
// the weight box is an L2 hit.  One thread issues tcgen05.mma (M = 128
// tokens, N = BN features, K = 16) into one of two TMEM accumulators while
// four epilogue warps drain the other.  TMEM lane = token row, so an
// epilogue's row-wise work stays inside one thread.
//
// The epilogue is a policy class Epi with
//   using Params = ...;                        (passed as a grid constant)
//   static void setup(const Params&, float* tab, int i);   i = 0..127: fill
//                                              128 floats of shared tables
//   static void prologue(const TileCore&, const Params&);  CTA 0, once
//   static void tile(const TileCore&, const Params&, int n, uint32_t tacc,
//                    int row, const float* tab);  one row of feature tile n
// Token rows past `rows` and features past the weight matrix are read as
// zeros by the TMA; the epilogue decides what to do with them.
#pragma once

#include "common.cuh"
#include "host.h"

namespace dflash {

constexpr int kTileThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kTileM = 128;
constexpr int kTileABytes = kTileM * 128;  // 128 rows x 64 bf16
constexpr int kBand = 8;                   // pairs of row tiles per raster band
constexpr int kTileSmemBudget = 220 * 1024;

struct TileCore {
  int rows;          // token rows (M)
  int m_tiles, n_tiles, k_tiles;
  int bn;            // features per tile: 128 or 256
  int layer_cols;    // token map l holds columns [l * layer_cols, (l + 1) * layer_cols)
  int b_split;       // feature tiles below it read weight map 0, the others map 1
  int b_split2;      // > 0: feature tiles from it on read weight map 2
  int b_cols;        // > 0: weight columns; k-tile kt reads weight column (64 kt) % b_cols
                     // (the same weights against two token operands summed along K)
  int b_paired;      // 1: half h of feature tile n's weight box comes from weight map h,
                     // rows n * BN/2 ..: accumulator columns [0, BN/2) are map 0's
                     // features, [BN/2, BN) map 1's same features (b_split unused)
  int n_stages, stage_bytes;
  uint32_t* status;
};

struct TokenMaps {
  CUtensorMap m[kMaxCtxLayers];
};

struct WeightMaps {
  CUtensorMap m[3];
};

// Pair tile t of the raster (row-tile pair mp = rows 256 mp .. 256 mp + 255,
// feature tile n): bands of kBand pairs; inside a band the pair varies
// fastest, so consecutive pair tiles (the clusters of one wave) share weights.
__device__ __forceinline__ void tile_coords(int mp_tiles, int n_tiles, int t, int* mp, int* n) {
  const int per_band = kBand * n_tiles;
  const int band = t / per_band, r = t - band * per_band;
  const int bm = min(kBand, mp_tiles - band * kBand);
  *n = r / bm;
  *mp = band * kBand + (r - *n * bm);
}

// Shared memory after the stages: full[n], empty[n], tfull[2], tempty[2],
// mdrain, the TMEM address, the abort flag, two spare words, then 128 floats
// of tables the epilogue may load (Epi::setup).
constexpr int kTileTailFixed = 5 * 8 + 4 * 4 + 128 * 4;

template <class Epi>
__global__ void __launch_bounds__(kTileThreads, 1)
tile_gemm_kernel(const __grid_constant__ TokenMaps tm_a, const __grid_constant__ WeightMaps tm_b,
                 const TileCore p, const __grid_constant__ typename Epi::Params ep) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.n_stages * p.stage_bytes);
  uint64_t* empty = full + p.n_stages;
  uint64_t* tfull = empty + p.n_stages;   // [2] accumulator ready
  uint64_t* tempty = tfull + 2;           // [2] accumulator drained
  uint64_t* mdrain = tempty + 2;          // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdrain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* tab = reinterpret_cast<float*>(tmem_slot + 4);  // the epilogue's tables
  const int crank = static_cast<int>(cluster_ctarank());   // 0 or 1: which tile of the pair
  const int cid = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int mp_tiles = (p.m_tiles + 1) >> 1;
  const int n_total = mp_tiles * p.n_tiles;                // pair tiles
  const uint32_t acc_cols = static_cast<uint32_t>(p.bn);
  const int half_rows = p.bn >> 1;                         // rows of one weight box

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.n_stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(mdrain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * acc_cols);
    tmem_relinquish();
  }
  if (threadIdx.x >= 64) Epi::setup(ep, tab, threadIdx.x - 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_normal();
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      for (int t = cid; ok && t < n_total; t += n_clusters) {
        int mp, n;
        tile_coords(mp_tiles, p.n_tiles, t, &mp, &n);
        const int m = 2 * mp + crank;
        const bool third = !p.b_paired && p.b_split2 > 0 && n >= p.b_split2;
        const bool second = !p.b_paired && !third && n >= p.b_split;
        const CUtensorMap* mb = third ? &tm_b.m[2] : (second ? &tm_b.m[1] : &tm_b.m[0]);
        const int n_local = third ? n - p.b_split2 : (second ? n - p.b_split : n);
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* a = smem + stage * p.stage_bytes;
          mbar_arrive_expect_tx(&full[stage], kTileABytes + p.bn * 128);
          const int l = (kt * 64) / p.layer_cols;
          tma_load_2d(a, &tm_a.m[l], &full[stage], kt * 64 - l * p.layer_cols, m * kTileM, pol);
          const int bcol = p.b_cols > 0 ? (kt * 64) % p.b_cols : kt * 64;
          // the weight box in two halves of BN/2 rows (a box has at most 256 rows)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const CUtensorMap* mh = p.b_paired ? &tm_b.m[h] : mb;
            const int brow = p.b_paired ? n * half_rows : n_local * p.bn + h * half_rows;
            tma_load_2d(a + kTileABytes + h * half_rows * 128, mh, &full[stage], bcol, brow, pol);
          }
          ++issued;
          if (++stage == static_cast<uint32_t>(p.n_stages)) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // no copy may still be landing when the CTA exits
      for (int st = 0; st < p.n_stages && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / p.n_stages) * p.n_stages;
        mbar_wait_drain(&full[st], static_cast<uint32_t>((last / p.n_stages) & 1), p.status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t base = smem_u32(smem);
      const uint32_t idesc = umma_idesc_bf16(kTileM, p.bn);
      uint32_t stage = 0, phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = cid; ok && t < n_total; t += n_clusters, ++it) {
        const int slot = it & 1;
        if (it >= 2 && !mbar_wait(&tempty[slot], static_cast<uint32_t>(((it >> 1) - 1) & 1),
                                  abort_flag, p.status))
          break;
        tc_fence_after();
        const uint32_t acc = tmem_base + slot * acc_cols;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = base + stage * p.stage_bytes;
          const uint64_t adesc = umma_sdesc_sw128(a_addr);
          const uint64_t bdesc = umma_sdesc_sw128(a_addr + kTileABytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(acc, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kt | kk) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == static_cast<uint32_t>(p.n_stages)) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) umma_commit(&tfull[slot]);
      }
      umma_commit(mdrain);
      mbar_wait_drain(mdrain, 0, p.status);
    }
  } else {
    if (blockIdx.x == 0) Epi::prologue(p, ep);
    const int q = warp & 3;  // TMEM lane quadrant this warp may read
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int it = 0;
    for (int t = cid; t < n_total; t += n_clusters, ++it) {
      int mp, n;
      tile_coords(mp_tiles, p.n_tiles, t, &mp, &n);
      const int m = 2 * mp + crank;
      const int slot = it & 1;
      if (!mbar_wait(&tfull[slot], static_cast<uint32_t>((it >> 1) & 1), abort_flag, p.status))
        break;
      tc_fence_after();
      Epi::tile(p, ep, n, tmem_base + slot * acc_cols + lane_base, m * kTileM + q * 32 + lane,
                tab);
      tc_fence_before();
      mbar_arrive(&tempty[slot]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * acc_cols);
  }
  griddep_launch_dependents();
}

// Pipeline shape and launch: as many stages as the shared-memory budget
// holds, one cluster of two per pair of SMs that can hold it, at most one per
// pair tile, and at most max_ctas / 2 clusters when max_ctas >= 2 (below that
// the whole device: a cluster needs two SMs).  The clusters stride over the
// pair tiles, so any cluster count covers the work.
template <class Epi>
int run_tile_gemm(TileCore& g, const TokenMaps& am, const WeightMaps& bm,
                  const typename Epi::Params& ep, cudaStream_t st, int max_ctas = 0) {
  g.stage_bytes = kTileABytes + g.bn * 128;
  const int tail = 2 * 8 + kTileTailFixed;  // per-stage barriers counted below
  g.n_stages = (kTileSmemBudget - 1024 - tail) / (g.stage_bytes + 16);
  if (g.n_stages > 8) g.n_stages = 8;
  const int smem = 1024 + g.n_stages * (g.stage_bytes + 16) + tail;
  // once per process and instantiation (thread-safe static initialisation):
  // the shared-memory limit (it covers any stage count) and how many clusters
  // of two fit on the device at once (at most one CTA per SM)
  static const int limit_rc = set_smem_limit(
      reinterpret_cast<const void*>(tile_gemm_kernel<Epi>), kTileSmemBudget);
  if (limit_rc) return limit_rc;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kTileThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static const int max_clusters = [&cfg] {
    const int nsm = current_num_sms();
    if (nsm <= 0) return 0;
    cudaLaunchConfig_t q = cfg;
    q.gridDim = dim3(nsm & ~1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tile_gemm_kernel<Epi>, &q) != cudaSuccess) return 0;
    return n;
  }();
  if (max_clusters < 1) return DFLASH_E_CUDA;
  const int pairs = ((g.m_tiles + 1) / 2) * g.n_tiles;
  int clusters = pairs < max_clusters ? pairs : max_clusters;
  if (max_ctas >= 2 && clusters > max_ctas / 2) clusters = max_ctas / 2;
  cfg.gridDim = dim3(2 * clusters);
  cfg.numAttrs = 2;
  return cuda_err(cudaLaunchKernelEx(&cfg, tile_gemm_kernel<Epi>, am, bm, g, ep));
}

}  // namespace dflash
