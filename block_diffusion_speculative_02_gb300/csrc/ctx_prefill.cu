// Next: the context projection of a whole prompt, for the prefill.
//
// "dflash-mlx" (dpshk.com) 单次前向验证 ①: the target prefills the prompt in
// chunks, which initialises the caches; "DFlash双实现对比" (hotelren.com) §4:
// the drafter's context K/V are projected from the target's selected-layer
// hidden states.  So at prefill every prompt token needs the same projection
// as the per-cycle one (a1), over thousands of rows at once:
//   Y  = [h_1 | ... | h_nL] W_fc^T,   Y^ = RMSNorm(Y) g_h,
//   K  = RoPE(RMSNorm_head(Y^ W_k^T) g_k),   V = Y^ W_v^T.
// With that many rows the GEMMs are bound by the tensor cores, not by the
// weight stream, so this is a tiled GEMM rather than the stream-K one:
// persistent CTAs (one per SM) in clusters of two walk pairs of 128 x BN
// output tiles (token rows x features) that share their feature range, in a
// banded raster order (8 pairs of row tiles per band, so the clusters of one
// wave share weight and token tiles in L2).  A TMA pipeline stages each CTA's
// own 128 x 64 token box, and each CTA loads one half of the BN x 64 weight
// box multicast to both CTAs of the pair, so every weight byte leaves L2 once
// per pair (the L2-to-SM traffic per MMA drops by a third); a stage is
// refilled only when the MMAs of both CTAs have released it (their commits
// arrive on both CTAs' empty barriers).  One thread issues tcgen05.mma
// (M = 128 tokens, N = BN features, K = 16) into one of two TMEM accumulators
// while four epilogue warps drain the other.  TMEM lane = token row, so the
// row-wise work of the epilogues (sums of squares, head norms, the RoPE
// partner at d + D/2) stays inside one thread.
//  1. fc GEMM.  The token operand of k-tile kt is read from layer
//     floor(64 kt / H) through its own tensor map (the concatenation is never
//     built).  Epilogue: bf16(g_h * Y) and the tile's sum of Y^2 per row.
//     CTA 0 first snapshots the write positions, maps the pages the rows need
//     and moves the lengths.
//  2. K/V GEMM on bf16(g_h * Y).  Epilogue: the row's RMSNorm factor (one per
//     row, so it commutes with the GEMM), per-head RMSNorm and RoPE for K,
//     bf16 stores into the cache rows.
#include "common.cuh"
#include "host.h"

namespace dflash {
namespace {

constexpr int kTileThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kTileM = 128;
constexpr int kATileBytes = kTileM * 128;  // 128 rows x 64 bf16
constexpr int kBand = 8;                   // pairs of row tiles per raster band
constexpr uint16_t kPairMask = 0x3;        // both CTAs of the cluster
constexpr int kPrefillSmemBudget = 220 * 1024;

struct TileCore {
  int rows;          // token rows (M)
  int m_tiles, n_tiles, k_tiles;
  int bn;            // features per tile: 128 or 256
  int layer_cols;    // token map l holds columns [l * layer_cols, (l + 1) * layer_cols)
  int b_split;       // feature tiles below it read weight map 0, the others map 1
  int n_stages, stage_bytes;
  uint32_t* status;
};

struct TokenMaps {
  CUtensorMap m[kMaxCtxLayers];
};

struct WeightMaps {
  CUtensorMap m[2];
};

struct PrefillParams {
  int hidden, fc_n_tiles, tokens_per_seq, batch;
  float rms_eps;
  const uint16_t* hidden_norm_w;  // [H] or null
  uint16_t* yhat;                 // [rows][H]: bf16(g_h * Y)
  float* ss;                      // [fc_n_tiles][rows]: partial sums of Y^2
  const int32_t* write_pos;
  int32_t* pos_snapshot;          // [B]; -1: the sequence's rows are skipped
  dflash_kv_view cache;
  int n_kv_heads, head_dim;
  const uint16_t* k_norm_w;       // [D] or null
  RopeTable rope;
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

__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  return static_cast<uint32_t>(float_to_bf16_bits(a)) |
         (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
}

// Shared memory after the stages: full[n], empty[n], tfull[2], tempty[2],
// mdrain, the TMEM address, the abort flag, two spare words, then the RoPE
// table (hi[64], lo[64]).
constexpr int kTileTailFixed = 5 * 8 + 4 * 4 + 128 * 4;

template <class Epi>
__global__ void __launch_bounds__(kTileThreads, 1)
tile_gemm_kernel(const __grid_constant__ TokenMaps tm_a, const __grid_constant__ WeightMaps tm_b,
                 const TileCore p, const __grid_constant__ PrefillParams ep) {
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
  float* rope_tab = reinterpret_cast<float*>(tmem_slot + 4);
  const int crank = static_cast<int>(cluster_ctarank());   // 0 or 1: which tile of the pair
  const int cid = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  const int mp_tiles = (p.m_tiles + 1) >> 1;
  const int n_total = mp_tiles * p.n_tiles;                // pair tiles
  const uint32_t acc_cols = static_cast<uint32_t>(p.bn);
  const int half_rows = p.bn >> 1;                         // weight rows this CTA loads

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.n_stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 2);  // the MMAs of both CTAs of the pair
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
  if (threadIdx.x >= 64) {
    const int i = threadIdx.x - 64;
    if (i < 64) {
      rope_tab[i] = ep.rope.hi[i];
      rope_tab[64 + i] = ep.rope.lo[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before anything lands in them
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
        const bool second = n >= p.b_split;
        const CUtensorMap* mb = second ? &tm_b.m[1] : &tm_b.m[0];
        const int brow = (second ? n - p.b_split : n) * p.bn + crank * half_rows;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* a = smem + stage * p.stage_bytes;
          mbar_arrive_expect_tx(&full[stage], kATileBytes + p.bn * 128);
          const int l = (kt * 64) / p.layer_cols;
          tma_load_2d(a, &tm_a.m[l], &full[stage], kt * 64 - l * p.layer_cols, m * kTileM, pol);
          tma_load_2d_mc(a + kATileBytes + crank * half_rows * 128, mb, &full[stage], kt * 64,
                         brow, kPairMask, pol);
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
          const uint64_t bdesc = umma_sdesc_sw128(a_addr + kATileBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(acc, adesc + 2 * kk, bdesc + 2 * kk, idesc, (kt | kk) ? 1u : 0u);
          umma_commit_mc(&empty[stage], kPairMask);  // frees the stage in both CTAs' eyes
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
                rope_tab);
      tc_fence_before();
      mbar_arrive(&tempty[slot]);
    }
  }
  __syncthreads();
  // the peer may still be releasing stages of this CTA (its MMA commits
  // arrive here): neither CTA leaves before both have drained
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * acc_cols);
  }
  griddep_launch_dependents();
}

// Per sequence: snapshot the write position, map the pages rows pos..pos+T-1
// need and set seq_len = pos + T.
__device__ void reserve_prompt_rows(const PrefillParams& e, uint32_t* status, int b) {
  const int pos = e.write_pos[b];
  const dflash_kv_view& v = e.cache;
  const int limit = v.page_table ? v.max_pages * v.page_size : v.capacity;
  if (pos < 0 || pos > limit - e.tokens_per_seq) {
    e.pos_snapshot[b] = -1;
    set_status(status, DFLASH_ST_CAPACITY);
    return;
  }
  e.pos_snapshot[b] = pos;
  if (v.page_table) map_rows(v, b, pos, e.tokens_per_seq, status);
  v.seq_len[b] = pos + e.tokens_per_seq;
}

// fc epilogue: thread = token row; Y of the tile's bn features in 16-column
// pieces: bf16(g_h * Y) to yhat and the row's sum of Y^2 over the tile.
struct FcEpi {
  static __device__ void prologue(const TileCore& p, const PrefillParams& e) {
    for (int b = threadIdx.x - 64; b < e.batch; b += 128) reserve_prompt_rows(e, p.status, b);
  }
  static __device__ void tile(const TileCore& p, const PrefillParams& e, int n, uint32_t tacc,
                              int row, const float*) {
    const int n0 = n * p.bn;
    const bool live = row < p.rows;
    uint16_t* dst = e.yhat + static_cast<size_t>(row) * e.hidden + n0;
    float ss = 0.f;
    for (int c0 = 0; c0 < p.bn; c0 += 16) {
      uint32_t v[16];
      tmem_ld_32x32b_x16(tacc + c0, v);
      float g[16];
      if (e.hidden_norm_w) {
        const uint4* gp = reinterpret_cast<const uint4*>(e.hidden_norm_w + n0 + c0);
        const uint4 g0 = __ldg(gp), g1 = __ldg(gp + 1);
        const uint32_t w[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          g[2 * j] = __uint_as_float(w[j] << 16);
          g[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) g[j] = 1.f;
      }
      tmem_ld_wait();
      uint32_t out[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float y0 = __uint_as_float(v[2 * j]), y1 = __uint_as_float(v[2 * j + 1]);
        ss = fmaf(y0, y0, fmaf(y1, y1, ss));
        out[j] = pack2_bf16(y0 * g[2 * j], y1 * g[2 * j + 1]);
      }
      if (live) {
        uint4* d = reinterpret_cast<uint4*>(dst + c0);
        d[0] = make_uint4(out[0], out[1], out[2], out[3]);
        d[1] = make_uint4(out[4], out[5], out[6], out[7]);
      }
    }
    if (live) e.ss[static_cast<size_t>(n) * p.rows + row] = ss;
  }
};

// K/V epilogue: thread = token row; the tile holds bn / D heads of K (tiles
// below b_split) or of V.  The row's RMSNorm factor of Y, then for K the head
// RMSNorm (a first pass over the head's columns for the sum of squares) and
// RoPE with the partner dimension d + D/2 loaded beside d; bf16 stores into
// the cache row write_pos + t.
struct KvEpi {
  static __device__ void prologue(const TileCore&, const PrefillParams&) {}
  static __device__ void tile(const TileCore& p, const PrefillParams& e, int n, uint32_t tacc,
                              int row, const float* rope_tab) {
    const int D = e.head_dim, half = D / 2;
    const bool is_k = n < p.b_split;
    const int f0 = (is_k ? n : n - p.b_split) * p.bn;  // first feature within Hkv * D
    const dflash_kv_view& cv = e.cache;
    const bool live = row < p.rows;
    long long off = -1;  // element offset of the row in head 0 of its cache slot
    int pos = 0;
    float r = 1.f;
    if (live) {
      const int b = row / e.tokens_per_seq, t = row - b * e.tokens_per_seq;
      const int p0 = e.pos_snapshot[b];
      if (p0 >= 0) {
        pos = p0 + t;
        if (cv.page_table) {
          const int page = cv.page_table[static_cast<size_t>(b) * cv.max_pages + pos / cv.page_size];
          if (page >= 0)
            off = (static_cast<long long>(page) * e.n_kv_heads * cv.page_size + pos % cv.page_size) * D;
          else
            set_status(p.status, DFLASH_ST_PAGE_MISSING);
        } else {
          off = (static_cast<long long>(b) * e.n_kv_heads * cv.capacity + pos) * D;
        }
      }
      if (e.hidden_norm_w) {
        float tot = 0.f;
        for (int qq = 0; qq < e.fc_n_tiles; ++qq) tot += e.ss[static_cast<size_t>(qq) * p.rows + row];
        r = rsqrtf(tot / e.hidden + e.rms_eps);
      }
    }
    const long long head_stride =
        static_cast<long long>(cv.page_table ? cv.page_size : cv.capacity) * D;
    uint16_t* dst_base = static_cast<uint16_t*>(is_k ? cv.k : cv.v);
    const bool knorm = is_k && e.k_norm_w;
    for (int h0 = 0; h0 < p.bn; h0 += D) {
      const int head = (f0 + h0) / D;
      float rs = r;
      if (knorm) {
        float sq = 0.f;
        for (int c0 = 0; c0 < D; c0 += 16) {
          uint32_t v[16];
          tmem_ld_32x32b_x16(tacc + h0 + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float x = __uint_as_float(v[j]) * r;
            sq = fmaf(x, x, sq);
          }
        }
        rs = r * rsqrtf(sq / D + e.rms_eps);
      }
      for (int c0 = 0; c0 < half; c0 += 16) {
        uint32_t lo[16], hi[16];
        tmem_ld_32x32b_x16(tacc + h0 + c0, lo);
        tmem_ld_32x32b_x16(tacc + h0 + half + c0, hi);
        tmem_ld_wait();
        uint32_t plo[8], phi[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          float xl[2], xh[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int d = c0 + j + u;
            float a = __uint_as_float(lo[j + u]) * rs, c = __uint_as_float(hi[j + u]) * rs;
            if (is_k) {
              if (knorm) {
                a *= bf16_bits_to_float(__ldg(e.k_norm_w + d));
                c *= bf16_bits_to_float(__ldg(e.k_norm_w + d + half));
              }
              float sn, cs;
              rope_sincos(pos, rope_tab[d], rope_tab[64 + d], &sn, &cs);
              const float a2 = a * cs - c * sn;
              c = c * cs + a * sn;
              a = a2;
            }
            xl[u] = a;
            xh[u] = c;
          }
          plo[j / 2] = pack2_bf16(xl[0], xl[1]);
          phi[j / 2] = pack2_bf16(xh[0], xh[1]);
        }
        if (off >= 0) {
          uint16_t* dst = dst_base + off + head * head_stride + c0;
          uint4* d0 = reinterpret_cast<uint4*>(dst);
          uint4* d1 = reinterpret_cast<uint4*>(dst + half);
          d0[0] = make_uint4(plo[0], plo[1], plo[2], plo[3]);
          d0[1] = make_uint4(plo[4], plo[5], plo[6], plo[7]);
          d1[0] = make_uint4(phi[0], phi[1], phi[2], phi[3]);
          d1[1] = make_uint4(phi[4], phi[5], phi[6], phi[7]);
        }
      }
    }
  }
};

// Workspace of one prefill call: status word, write-position snapshot,
// partial sums of Y^2, bf16(g_h * Y).
struct PrefillPlan {
  int rows, fc_bn, fc_n_tiles, kv_bn;
  size_t off_status, off_pos, off_ss, off_yhat, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int make_prefill_plan(const dflash_dims& d, int tokens_per_seq, PrefillPlan* p) {
  int rc = check_dims(&d);
  if (rc) return rc;
  if (tokens_per_seq < 1) return DFLASH_E_ARG;
  const long long rows = static_cast<long long>(d.batch) * tokens_per_seq;
  if (rows > (1 << 24)) return DFLASH_E_UNSUPPORTED;
  const int kvd = d.n_kv_heads * d.head_dim;
  if (d.hidden % 128 || kvd % 128 || (d.head_dim != 64 && d.head_dim != 128))
    return DFLASH_E_UNSUPPORTED;
  PrefillPlan q = {};
  q.rows = static_cast<int>(rows);
  q.fc_bn = d.hidden % 256 == 0 ? 256 : 128;
  q.fc_n_tiles = d.hidden / q.fc_bn;
  q.kv_bn = kvd % 256 == 0 ? 256 : 128;
  size_t off = 0;
  q.off_status = off;  off = align256(off + 256);
  q.off_pos = off;     off = align256(off + sizeof(int32_t) * d.batch);
  q.off_ss = off;      off = align256(off + sizeof(float) * q.fc_n_tiles * rows);
  q.off_yhat = off;    off = align256(off + sizeof(uint16_t) * rows * d.hidden);
  q.total = off;
  *p = q;
  return DFLASH_OK;
}

template <class Epi>
int run_tile_gemm(TileCore& g, const TokenMaps& am, const WeightMaps& bm,
                  const PrefillParams& ep, cudaStream_t st) {
  g.stage_bytes = kATileBytes + g.bn * 128;
  const int tail = 2 * 8 + kTileTailFixed;  // per-stage barriers counted below
  g.n_stages = (kPrefillSmemBudget - 1024 - tail) / (g.stage_bytes + 16);
  if (g.n_stages > 8) g.n_stages = 8;
  const int smem = 1024 + g.n_stages * (g.stage_bytes + 16) + tail;
  // once per process and instantiation (thread-safe static initialisation):
  // the shared-memory limit (it covers any stage count) and how many clusters
  // of two fit on the device at once (at most one CTA per SM)
  static const int limit_rc = set_smem_limit(
      reinterpret_cast<const void*>(tile_gemm_kernel<Epi>), kPrefillSmemBudget);
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
  const int clusters = pairs < max_clusters ? pairs : max_clusters;
  cfg.gridDim = dim3(2 * clusters);
  cfg.numAttrs = 2;
  return cuda_err(cudaLaunchKernelEx(&cfg, tile_gemm_kernel<Epi>, am, bm, g, ep));
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" size_t dflash_prefill_workspace_bytes(const dflash_dims* dims, int32_t tokens_per_seq) {
  if (!dims) return 0;
  PrefillPlan p;
  if (make_prefill_plan(*dims, tokens_per_seq, &p)) return 0;
  return p.total;
}

extern "C" int dflash_ctx_prefill(const dflash_dims* dims, int32_t tokens_per_seq,
                                  const void* const* layer_hidden, const void* w_fc,
                                  const void* hidden_norm_w, const void* w_k, const void* w_v,
                                  const void* k_norm_w, const int32_t* write_pos,
                                  const dflash_kv_view* cache, void* ws, size_t ws_bytes,
                                  dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_ctx_prefill");
  if (!dims) return DFLASH_E_ARG;
  PrefillPlan plan;
  int rc = make_prefill_plan(*dims, tokens_per_seq, &plan);
  if (rc) return rc;
  if (!layer_hidden || !w_fc || !w_k || !w_v || !write_pos || !cache || !cache->k ||
      !cache->v || !cache->seq_len)
    return DFLASH_E_ARG;
  const int nL = dims->n_ctx_layers, H = dims->hidden;
  for (int l = 0; l < nL; ++l) {
    if (!layer_hidden[l]) return DFLASH_E_ARG;
    if (!aligned16(layer_hidden[l])) return DFLASH_E_ALIGN;
  }
  if (!aligned16(w_fc) || !aligned16(w_k) || !aligned16(w_v) || !aligned16(cache->k) ||
      !aligned16(cache->v) || (hidden_norm_w && !aligned16(hidden_norm_w)))
    return DFLASH_E_ALIGN;
  if (cache->page_table) {
    if (!cache->free_list || !cache->free_count || cache->page_size < 1 || cache->max_pages < 1)
      return DFLASH_E_ARG;
  } else if (cache->capacity < 1) {
    return DFLASH_E_ARG;
  }
  if (!ws) return DFLASH_E_WORKSPACE;
  if (ws_bytes < plan.total) return DFLASH_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int kvd = dims->n_kv_heads * dims->head_dim;
  const uint64_t rows = static_cast<uint64_t>(plan.rows);
  uint16_t* yhat = ws_at<uint16_t>(ws, plan.off_yhat);

  PrefillParams ep = {};
  ep.hidden = H;
  ep.fc_n_tiles = plan.fc_n_tiles;
  ep.tokens_per_seq = tokens_per_seq;
  ep.batch = dims->batch;
  ep.rms_eps = dims->rms_eps;
  ep.hidden_norm_w = static_cast<const uint16_t*>(hidden_norm_w);
  ep.yhat = yhat;
  ep.ss = ws_at<float>(ws, plan.off_ss);
  ep.write_pos = write_pos;
  ep.pos_snapshot = ws_at<int32_t>(ws, plan.off_pos);
  ep.cache = *cache;
  ep.n_kv_heads = dims->n_kv_heads;
  ep.head_dim = dims->head_dim;
  ep.k_norm_w = static_cast<const uint16_t*>(k_norm_w);
  fill_rope_table(ep.rope.hi, ep.rope.lo, dims->head_dim, dims->rope_theta);

  // ---- 1. fc GEMM: bf16(g_h * Y) and sums of Y^2 ----
  {
    TileCore g = {};
    g.status = ws_at<uint32_t>(ws, plan.off_status);
    g.rows = plan.rows;
    g.m_tiles = (plan.rows + kTileM - 1) / kTileM;
    g.bn = plan.fc_bn;
    g.n_tiles = plan.fc_n_tiles;
    g.k_tiles = nL * H / 64;
    g.layer_cols = H;
    g.b_split = g.n_tiles;
    TokenMaps am;
    for (int l = 0; l < nL; ++l)
      if ((rc = make_tmap_2d_bf16(&am.m[l], layer_hidden[l], H, rows,
                                  static_cast<uint64_t>(H) * 2, 64, kTileM)))
        return rc;
    for (int l = nL; l < kMaxCtxLayers; ++l) am.m[l] = am.m[0];
    WeightMaps bm;
    if ((rc = make_tmap_2d_bf16(&bm.m[0], w_fc, static_cast<uint64_t>(nL) * H, H,
                                static_cast<uint64_t>(nL) * H * 2, 64, g.bn / 2)))
      return rc;
    bm.m[1] = bm.m[0];
    if ((rc = run_tile_gemm<FcEpi>(g, am, bm, ep, st))) return rc;
  }
  // ---- 2. K/V GEMM: row factor, head norm + RoPE for K, cache stores ----
  {
    TileCore g = {};
    g.status = ws_at<uint32_t>(ws, plan.off_status);
    g.rows = plan.rows;
    g.m_tiles = (plan.rows + kTileM - 1) / kTileM;
    g.bn = plan.kv_bn;
    g.n_tiles = 2 * kvd / g.bn;
    g.k_tiles = H / 64;
    g.layer_cols = H;
    g.b_split = kvd / g.bn;
    TokenMaps am;
    if ((rc = make_tmap_2d_bf16(&am.m[0], yhat, H, rows, static_cast<uint64_t>(H) * 2, 64,
                                kTileM)))
      return rc;
    for (int l = 1; l < kMaxCtxLayers; ++l) am.m[l] = am.m[0];
    WeightMaps bm;
    if ((rc = make_tmap_2d_bf16(&bm.m[0], w_k, H, kvd, static_cast<uint64_t>(H) * 2, 64,
                                g.bn / 2)))
      return rc;
    if ((rc = make_tmap_2d_bf16(&bm.m[1], w_v, H, kvd, static_cast<uint64_t>(H) * 2, 64,
                                g.bn / 2)))
      return rc;
    if ((rc = run_tile_gemm<KvEpi>(g, am, bm, ep, st))) return rc;
  }
  return DFLASH_OK;
}
