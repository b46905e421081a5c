// a1 — context projection of the target's selected-layer hidden states into
// the drafter's context K/V cache.
//
// "DFlash双实现对比" (hotelren.com) §4: the hidden states of the layers in
// target_layer_ids are concatenated; §2: the drafter's context K/V are
// projected from them.  "dflash-mlx" (dpshk.com) 块扩散草稿 step 3: the
// drafter reads the target's multi-layer hidden states.
//
// Two kernels on one stream, both "swap-AB" stream-K GEMMs on the
// 5th-generation tensor cores (128 output features are the MMA's M, the token
// rows its N, fp32 accumulators in TMEM, the weight stream staged by a TMA
// pipeline).  At small batch the GEMMs are bound by the weight stream, so the
// work is cut into units of (output tile, k-stage) and every CTA of the grid
// (one per SM of the budget) streams one equal contiguous range of units:
// all SMs move weights, whatever the tile count.  A CTA's range crosses tile
// boundaries; each piece ("segment") accumulates in one of two TMEM slots
// (the epilogue drains one while the MMAs fill the other) and is added into
// an fp32 accumulator in the workspace with fire-and-forget atomic adds.  The
// CTA that completes a tile's count of contributions (atomic ticket, no
// waiting) reads the finished sums in one round trip, clears them for the
// next call and finishes the tile once its own pipeline has drained:
//  1. fc GEMM   Y = X W_fc^T.  X is never materialised: the k-loop reads
//     layer floor(k / H) through its own tensor map, which is the
//     concatenation.  Finisher: g_h * Y stored as a bf16 pair hi + lo
//     (exact to ~2^-17, so the next GEMM keeps Y's fp32 precision) and the
//     tile's partial sums of Y^2.  CTA 0 also snapshots the write positions,
//     maps the pages the block needs and sets seq_len = pos + 16.
//  2. K/V GEMM  [K;V] = [hi;lo] W_{k|v}^T.  Finisher: the RMSNorm scale of Y
//     (one factor per token row, so it commutes with the GEMM), per-head
//     RMSNorm and RoPE for K, bf16 store into the cache rows.
// The order of the fp32 additions across CTAs is not fixed, so results can
// differ between runs by fp32 rounding (well inside the bf16 outputs' ulp).
#include "common.cuh"
#include "host.h"

namespace dflash {
namespace {

constexpr int kGemmThreads = 192;
constexpr int kATile = 128 * 128;  // 128 rows x 64 bf16
constexpr int kMaxGemmStages = 12;
constexpr int kMaxSegments = 32;   // tiles one CTA may touch
#ifndef DFLASH_GEMM_CHUNKS_PER_STAGE
#define DFLASH_GEMM_CHUNKS_PER_STAGE 4
#endif
constexpr int kGemmChunksPerStage = DFLASH_GEMM_CHUNKS_PER_STAGE;

struct LayerMaps {
  CUtensorMap m[kMaxCtxLayers];
};

struct GemmParams {
  int mode;          // kModeFc or kModeKv (selects the finisher)
  int k_tiles;       // K / 64
  int k_stages;      // ceil(k_tiles / kb): work units per tile
  int n_units;       // out_tiles * n_chunks * k_stages
  int out_tiles;     // output features / 128
  int a_split;       // tiles >= a_split read the second weight map
  int layer_cols;    // columns per B map (fc: H); k-tile kt reads map (kt*64)/layer_cols
  int n_tok;
  int chunk_rows;    // token rows per chunk (B box rows)
  int n_chunks;
  int hilo;          // 1: B = [hi rows ; lo rows] of a 2*n_tok-row matrix, summed in the epilogue
  int ld_out;        // features per partial row
  int mma_n;         // MMA N = chunk_rows * (1 + hilo)
  int n_stages, stage_bytes, tmem_cols;
  int kb;            // 64-column K chunks per pipeline stage
  int b_chunk;       // bytes of the token tile of one chunk (1024-aligned)
  float* acc;        // [n_tok][ld_out] fp32 accumulator, zero between calls
  uint32_t* tickets; // [n_chunks * out_tiles] contributions so far, zero between calls
  uint32_t* status;
  // shared by both finishers
  int hidden, fc_out_tiles;
  float rms_eps;
  const uint16_t* hidden_norm_w;  // [H] or null
  uint16_t* yhat;                 // [2][n_tok][H]: hi, lo of g_h * Y
  float* ss;                      // [fc_out_tiles][n_tok]: partial sums of Y^2
  // fc kernel, CTA 0: write positions, page reservation, lengths
  int batch;
  const int32_t* write_pos;
  int32_t* pos_snapshot;
  dflash_kv_view cache;
  // kv finisher
  int n_kv_heads, head_dim;
  const uint16_t* k_norm_w;       // [D] or null
  RopeTable rope;
};

constexpr int kModeFc = 0;
constexpr int kModeKv = 1;

// Per sequence: snapshot the write position, map the pages that rows
// pos..pos+15 need (popping the free list), and set seq_len = pos + 16.
__device__ void reserve_block_rows(const GemmParams& p, int b) {
  const int pos = p.write_pos[b];
  p.pos_snapshot[b] = pos;
  const dflash_kv_view& v = p.cache;
  const int limit = v.page_table ? v.max_pages * v.page_size : v.capacity;
  if (pos < 0 || pos + kBlock > limit) {
    set_status(p.status, DFLASH_ST_CAPACITY);
    return;
  }
  if (v.page_table) {
    int32_t* tbl = v.page_table + static_cast<size_t>(b) * v.max_pages;
    for (int pg = pos / v.page_size; pg <= (pos + kBlock - 1) / v.page_size; ++pg) {
      if (tbl[pg] >= 0) continue;
      const int slot = atomicSub(v.free_count, 1) - 1;
      if (slot < 0) {
        atomicAdd(v.free_count, 1);
        set_status(p.status, DFLASH_ST_POOL_EMPTY);
        break;
      }
      tbl[pg] = v.free_list[slot];
    }
  }
  v.seq_len[b] = pos + kBlock;
}

constexpr int kTokGroup = 4;  // token rows a warp finishes together (loads in flight)

__device__ __forceinline__ uint2 pack4_bf16(float a, float b, float c, float d) {
  return make_uint2(static_cast<uint32_t>(float_to_bf16_bits(a)) |
                        (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16),
                    static_cast<uint32_t>(float_to_bf16_bits(c)) |
                        (static_cast<uint32_t>(float_to_bf16_bits(d)) << 16));
}

__device__ __forceinline__ float4 load4_bf16(const uint16_t* src) {
  const uint2 w = *reinterpret_cast<const uint2*>(src);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
}

// The finished sums of 4 consecutive features of token row `tok`, cleared
// again for the next call.
__device__ __forceinline__ float4 take4(const GemmParams& p, int tok, int f0) {
  float4* src = reinterpret_cast<float4*>(p.acc + static_cast<size_t>(tok) * p.ld_out + f0);
  const float4 v = __ldcg(src);
  __stcg(src, make_float4(0.f, 0.f, 0.f, 0.f));
  return v;
}

// fc finisher (CTA that completed an output tile): Y = the accumulated sum;
// hi/lo bf16 pair of g_h * Y for the next GEMM; the tile's partial sums of Y^2
// per token row (the RMSNorm scale itself is applied after the K/V GEMM,
// since it is one factor per token row).  Warp w takes token rows w, w + 4,
// ...; a lane owns 4 consecutive features.
__device__ void finish_fc(const GemmParams& p, int o, int c) {
  const int et = threadIdx.x - 64, warp = et >> 5, lane = et & 31;
  const int f0 = o * 128 + lane * 4;
  const float4 g = p.hidden_norm_w ? load4_bf16(p.hidden_norm_w + f0) : make_float4(1.f, 1.f, 1.f, 1.f);
  const int t0 = c * p.chunk_rows;
  const int nt = min(p.chunk_rows, p.n_tok - t0);
#pragma unroll 1
  for (int j0 = warp * kTokGroup; j0 < nt; j0 += 4 * kTokGroup) {
    float4 y[kTokGroup];
#pragma unroll
    for (int k = 0; k < kTokGroup; ++k)
      if (j0 + k < nt) y[k] = take4(p, t0 + j0 + k, f0);
#pragma unroll
    for (int k = 0; k < kTokGroup; ++k) {
      if (j0 + k >= nt) break;
      const int tok = t0 + j0 + k;
      const float a[4] = {y[k].x * g.x, y[k].y * g.y, y[k].z * g.z, y[k].w * g.w};
      float hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = bf16_bits_to_float(float_to_bf16_bits(a[e]));
        lo[e] = a[e] - hi[e];
      }
      *reinterpret_cast<uint2*>(p.yhat + static_cast<size_t>(tok) * p.hidden + f0) =
          pack4_bf16(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint2*>(p.yhat + (static_cast<size_t>(p.n_tok) + tok) * p.hidden + f0) =
          pack4_bf16(lo[0], lo[1], lo[2], lo[3]);
      float sq = y[k].x * y[k].x + y[k].y * y[k].y + y[k].z * y[k].z + y[k].w * y[k].w;
#pragma unroll
      for (int off = 16; off; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if (lane == 0) p.ss[static_cast<size_t>(o) * p.n_tok + tok] = sq;
    }
  }
}

// kv finisher (CTA that completed an output tile): K or V rows of 128
// features (one head at D = 128, two at D = 64) for every token row of the
// chunk: the accumulated sum, the RMSNorm scale of Y, per-head RMSNorm and
// RoPE for K, bf16 store into the cache row write_pos + t.  The per-token
// scale and cache offsets are set up first, one thread per token row; then
// warp w takes token rows w, w + 4, ..., a lane owning 4 consecutive features
// (a head spans D / 4 lanes, the RoPE partner of dims d < D/2 sits D / 8
// lanes further).
__device__ void finish_kv(const GemmParams& p, int o, int c, uint8_t* scratch) {
  const int et = threadIdx.x - 64, warp = et >> 5, lane = et & 31;
  const int D = p.head_dim;
  const bool is_k = o < p.a_split;
  const int feat0 = (is_k ? o : o - p.a_split) * 128 + lane * 4;  // within Hkv * D
  const int head = feat0 / D, d0 = feat0 - head * D;
  const int t0 = c * p.chunk_rows;
  const int nt = min(p.chunk_rows, p.n_tok - t0);
  float* rbuf = reinterpret_cast<float*>(scratch);                  // [chunk_rows]
  long long* dst_off = reinterpret_cast<long long*>(scratch + 1024); // [chunk_rows], -1 = skip
  int* posb = reinterpret_cast<int*>(scratch + 1024 + 8 * 256);     // [chunk_rows]
  float* rope_hi = reinterpret_cast<float*>(scratch + 4096);        // [D/2], read by index
  float* rope_lo = rope_hi + 64;
  if (et < D / 2) {
    rope_hi[et] = p.rope.hi[et];
    rope_lo[et] = p.rope.lo[et];
  }
  const dflash_kv_view& cv = p.cache;
  const int limit = cv.page_table ? cv.max_pages * cv.page_size : cv.capacity;
  // head-major caches: [B, Hkv, capacity, D] or [pages, Hkv, page_size, D]
  const long long head_stride =
      static_cast<long long>(cv.page_table ? cv.page_size : cv.capacity) * D;
  for (int j = et; j < nt; j += 128) {
    const int tok = t0 + j;
    const int b = tok / kBlock, t = tok - b * kBlock;
    const int pos0 = p.pos_snapshot[b];
    long long off = -1;
    if (pos0 >= 0 && pos0 + kBlock <= limit) {  // else flagged by the reservation
      const int pos = pos0 + t;
      if (cv.page_table) {
        const int page =
            cv.page_table[static_cast<size_t>(b) * cv.max_pages + pos / cv.page_size];
        if (page >= 0)
          off = (static_cast<long long>(page) * p.n_kv_heads * cv.page_size + pos % cv.page_size) * D;
        else
          set_status(p.status, DFLASH_ST_PAGE_MISSING);
      } else {
        off = (static_cast<long long>(b) * p.n_kv_heads * cv.capacity + pos) * D;
      }
    }
    dst_off[j] = off;
    posb[j] = pos0 + t;
    float r = 1.f;
    if (p.hidden_norm_w) {
      float tot = 0.f;
      for (int q = 0; q < p.fc_out_tiles; ++q) tot += p.ss[static_cast<size_t>(q) * p.n_tok + tok];
      r = rsqrtf(tot / p.hidden + p.rms_eps);
    }
    rbuf[j] = r;
  }
  named_bar_sync(1, 128);
  const float4 gk = (is_k && p.k_norm_w) ? load4_bf16(p.k_norm_w + d0) : make_float4(1.f, 1.f, 1.f, 1.f);
  const int half = D / 2;
  const bool lower = d0 < half;
  const int fi = lower ? d0 : d0 - half;                   // first of 4 frequencies
  uint16_t* dst_base = static_cast<uint16_t*>(is_k ? cv.k : cv.v);
#pragma unroll 1
  for (int j0 = warp * kTokGroup; j0 < nt; j0 += 4 * kTokGroup) {
    float4 v[kTokGroup];
#pragma unroll
    for (int k = 0; k < kTokGroup; ++k)
      if (j0 + k < nt) v[k] = take4(p, t0 + j0 + k, o * 128 + lane * 4);
#pragma unroll
    for (int k = 0; k < kTokGroup; ++k) {
      if (j0 + k >= nt) break;
      const int j = j0 + k;
      const float r = rbuf[j];
      float x[4] = {v[k].x * r, v[k].y * r, v[k].z * r, v[k].w * r};
      if (is_k) {
        if (p.k_norm_w) {
          float sq = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
          for (int off = D / 8; off; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
          const float rs = rsqrtf(sq / D + p.rms_eps);
          x[0] *= rs * gk.x;
          x[1] *= rs * gk.y;
          x[2] *= rs * gk.z;
          x[3] *= rs * gk.w;
        }
        const int pos = posb[j];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float partner = __shfl_xor_sync(0xffffffffu, x[e], D / 8);
          float sn, cs;
          rope_sincos(pos, rope_hi[fi + e], rope_lo[fi + e], &sn, &cs);
          x[e] = lower ? x[e] * cs - partner * sn : x[e] * cs + partner * sn;
        }
      }
      const long long off = dst_off[j];
      if (off >= 0)
        *reinterpret_cast<uint2*>(dst_base + off + head * head_stride + d0) =
            pack4_bf16(x[0], x[1], x[2], x[3]);
    }
  }
}

// Unit u = (tile T, k-stage ks) with u = T * k_stages + ks; tile T covers
// output features (T % out_tiles) * 128 .. +127 for token chunk T / out_tiles.
// CTA i of G streams units [U*i/G, U*(i+1)/G): every CTA moves the same
// number of weight bytes whatever the tile count.
__device__ __forceinline__ int unit_begin(const GemmParams& p, int i) {
  return static_cast<int>(static_cast<long long>(p.n_units) * i / gridDim.x);
}

// The CTA whose unit range holds unit u.
__device__ __forceinline__ int unit_owner(const GemmParams& p, int u) {
  return static_cast<int>((static_cast<long long>(gridDim.x) * (u + 1) - 1) / p.n_units);
}

// Number of CTAs that add partial sums into tile T.
__device__ __forceinline__ uint32_t tile_contributors(const GemmParams& p, int T) {
  const int first = T * p.k_stages;
  const int last = min(p.n_units, first + p.k_stages) - 1;
  return static_cast<uint32_t>(unit_owner(p, last) - unit_owner(p, first) + 1);
}

__global__ void __launch_bounds__(kGemmThreads)
streamk_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0,
                    const __grid_constant__ CUtensorMap tm_a1,
                    const __grid_constant__ LayerMaps tm_b, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.n_stages * p.stage_bytes);
  uint64_t* empty = full + p.n_stages;
  uint64_t* tfull = empty + p.n_stages;   // [2] accumulator slot ready
  uint64_t* tempty = tfull + 2;           // [2] accumulator slot drained
  uint64_t* mdrain = tempty + 2;          // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdrain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* seg_ok = reinterpret_cast<volatile int*>(tmem_slot + 2);
  volatile int* n_fin = reinterpret_cast<volatile int*>(tmem_slot + 3);
  int* fin_tiles = reinterpret_cast<int*>(tmem_slot + 4);  // [kMaxSegments]

  const int u0 = unit_begin(p, blockIdx.x);
  const int u1 = unit_begin(p, blockIdx.x + 1);
  const int KS = p.k_stages;

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
    *n_fin = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 2 * p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      const uint32_t bbytes = (1 + p.hilo) * p.chunk_rows * 128;
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      for (int u = u0; u < u1; ++u) {
        const int T = u / KS, kt = (u - T * KS) * p.kb;
        const int o = T % p.out_tiles, c = T / p.out_tiles;
        const CUtensorMap* ma = o < p.a_split ? &tm_a0 : &tm_a1;
        const int arow = (o < p.a_split ? o : o - p.a_split) * 128;
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) break;
        const int nck = min(p.kb, p.k_tiles - kt);
        uint8_t* a = smem + stage * p.stage_bytes;
        uint8_t* bt = a + p.kb * kATile;
        mbar_arrive_expect_tx(&full[stage], nck * (kATile + bbytes));
        // the chunks of a stage go out back to back: each weight row is
        // requested as nck * 128 contiguous bytes
        for (int j = 0; j < nck; ++j) {
          const int k = kt + j;
          tma_load_2d(a + j * kATile, ma, &full[stage], k * 64, arow, pol_w);
          const int l = (k * 64) / p.layer_cols;
          const int col = k * 64 - l * p.layer_cols;
          uint8_t* bj = bt + j * p.b_chunk;
          tma_load_2d(bj, &tm_b.m[l], &full[stage], col, c * p.chunk_rows, pol_x);
          if (p.hilo)
            tma_load_2d(bj + p.chunk_rows * 128, &tm_b.m[l], &full[stage], col,
                        p.n_tok + c * p.chunk_rows, pol_x);
        }
        ++issued;
        if (++stage == static_cast<uint32_t>(p.n_stages)) {
          stage = 0;
          phase ^= 1;
        }
      }
      // no copy may still be landing when the stages are reused by the finisher
      for (int st = 0; st < p.n_stages && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / p.n_stages) * p.n_stages;
        mbar_wait_drain(&full[st], static_cast<uint32_t>((last / p.n_stages) & 1), p.status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t base = smem_u32(smem);
      const uint32_t idesc = umma_idesc_bf16(128, p.mma_n);
      uint32_t stage = 0, phase = 0;
      int seg = 0;
      uint32_t acc = 0;
      bool first = true;
      for (int u = u0; u < u1; ++u) {
        const int ks = u % KS;
        if (u == u0 || ks == 0) {  // a segment (this CTA's part of one tile) starts
          const int slot = seg & 1;
          if (seg >= 2 &&
              !mbar_wait(&tempty[slot], static_cast<uint32_t>(((seg >> 1) - 1) & 1), abort_flag,
                         p.status))
            break;
          tc_fence_after();
          acc = tmem_base + slot * p.tmem_cols;
          first = true;
        }
        if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) break;
        tc_fence_after();
        const int nck = min(p.kb, p.k_tiles - ks * p.kb);
        const uint32_t a_addr = base + stage * p.stage_bytes;
        for (int j = 0; j < nck; ++j) {
          const uint64_t adesc = umma_sdesc_sw128(a_addr + j * kATile);
          const uint64_t bdesc = umma_sdesc_sw128(a_addr + p.kb * kATile + j * p.b_chunk);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            umma_bf16(acc, adesc + 2 * kk, bdesc + 2 * kk, idesc, first ? 0u : 1u);
            first = false;
          }
        }
        umma_commit(&empty[stage]);
        if (u == u1 - 1 || ks == KS - 1) {  // the segment ends: hand the slot over
          umma_commit(&tfull[seg & 1]);
          ++seg;
        }
        if (++stage == static_cast<uint32_t>(p.n_stages)) {
          stage = 0;
          phase ^= 1;
        }
      }
      umma_commit(mdrain);
      mbar_wait_drain(mdrain, 0, p.status);
    }
  } else {
    const int et = threadIdx.x - 64;
    if (p.mode == kModeFc && blockIdx.x == 0) {
      for (int b = et; b < p.batch; b += 128) reserve_block_rows(p, b);
    }
    // epilogue: TMEM lane = output feature, column = token (hi, then lo)
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    int seg = 0;
    for (int u = u0; u < u1; ++seg) {
      const int T = u / KS;
      const int o = T % p.out_tiles, c = T / p.out_tiles;
      const int slot = seg & 1;
      const bool ok = mbar_wait(&tfull[slot], static_cast<uint32_t>((seg >> 1) & 1), abort_flag,
                                p.status);
      named_bar_sync(1, 128);
      if (et == 0) *seg_ok = ok && !*abort_flag;
      named_bar_sync(1, 128);
      if (!*seg_ok) break;  // uniform over the four warps
      tc_fence_after();
      const uint32_t tacc = tmem_base + slot * p.tmem_cols + lane_base;
      // partial sums go to the fp32 accumulator by fire-and-forget atomic adds
      // at L2; the tile's finisher then needs one round trip
      float* dst = p.acc + o * 128 + q * 32 + lane;
      for (int c0 = 0; c0 < p.chunk_rows; c0 += 16) {
        uint32_t v[16], w[16];
        tmem_ld_32x32b_x16(tacc + c0, v);
        if (p.hilo) tmem_ld_32x32b_x16(tacc + p.chunk_rows + c0, w);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = c * p.chunk_rows + c0 + j;
          float val = __uint_as_float(v[j]);
          if (p.hilo) val += __uint_as_float(w[j]);
          if (tok < p.n_tok) atomicAdd(dst + static_cast<size_t>(tok) * p.ld_out, val);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[slot]);
      __threadfence();
      named_bar_sync(1, 128);
      if (et == 0 && atomicAdd(p.tickets + T, 1u) == tile_contributors(p, T) - 1u)
        fin_tiles[(*n_fin)++] = T;  // this CTA completed the tile's sum
      u = min(u1, (T + 1) * KS);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 2 * p.tmem_cols);
  }
  if (warp >= 2 && *n_fin > 0) {
    // finish the tiles this CTA completed; the pipeline is drained, so its
    // shared memory is free for the finisher
    __threadfence();
    const int nf = *n_fin;
    for (int i = 0; i < nf; ++i) {
      const int T = fin_tiles[i];
      const int o = T % p.out_tiles, c = T / p.out_tiles;
      if (p.mode == kModeFc) finish_fc(p, o, c); else finish_kv(p, o, c, smem);
      named_bar_sync(1, 128);  // scratch is reused by the next tile
      if (threadIdx.x == 64) p.tickets[T] = 0u;
    }
  }
  griddep_launch_dependents();
}

// Dynamic shared memory: 1 KB alignment slack, the stages with their full and
// empty barriers, then tfull[2], tempty[2], mdrain, four words and the
// finisher list.
constexpr int kGemmTail = 5 * 8 + 4 * 4 + kMaxSegments * 4;

int gemm_smem(int stage_bytes, int n_stages) {
  return 1024 + n_stages * (stage_bytes + 16) + kGemmTail;
}

int setup_gemm(GemmParams& g, int b_rows_per_stage) {
  g.b_chunk = ((b_rows_per_stage * 128 + 1023) / 1024) * 1024;
  // as many 64-column chunks per stage as still leave three stages
  g.kb = kGemmChunksPerStage;
  while (g.kb > 1 &&
         (kGemmSmemBudget - 1024 - kGemmTail) / (g.kb * (kATile + g.b_chunk) + 16) < 3)
    g.kb >>= 1;
  g.stage_bytes = g.kb * (kATile + g.b_chunk);
  g.n_stages = (kGemmSmemBudget - 1024 - kGemmTail) / (g.stage_bytes + 16);
  if (g.n_stages > kMaxGemmStages) g.n_stages = kMaxGemmStages;
  if (g.n_stages < 2) g.n_stages = 2;
  int cols = 32;
  while (cols < g.mma_n) cols *= 2;
  g.tmem_cols = cols;  // two slots of this width are allocated
  g.k_stages = (g.k_tiles + g.kb - 1) / g.kb;
  g.n_units = g.out_tiles * g.n_chunks * g.k_stages;
  return gemm_smem(g.stage_bytes, g.n_stages);
}

// CTAs of a stream-K launch: at most `ctas` (one per SM of the budget), at
// most one per unit, and enough that no CTA touches more than kMaxSegments
// tiles.
int streamk_grid(const GemmParams& g, int ctas) {
  int grid = ctas < g.n_units ? ctas : g.n_units;
  while (grid < g.n_units) {
    const int per = (g.n_units + grid - 1) / grid;
    if ((per + g.k_stages - 1) / g.k_stages + 1 <= kMaxSegments) break;
    ++grid;
  }
  return grid;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" int dflash_ctx_project(const dflash_dims* dims, const void* const* layer_hidden,
                                  const void* w_fc, const void* hidden_norm_w, const void* w_k,
                                  const void* w_v, const void* k_norm_w,
                                  const int32_t* write_pos, const dflash_kv_view* cache,
                                  void* ws, size_t ws_bytes, dflash_stream_t stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!layer_hidden || !w_fc || !w_k || !w_v || !write_pos || !cache || !cache->k ||
      !cache->v || !cache->seq_len)
    return DFLASH_E_ARG;
  const int nL = dims->n_ctx_layers;
  for (int l = 0; l < nL; ++l) {
    if (!layer_hidden[l]) return DFLASH_E_ARG;
    if (!aligned16(layer_hidden[l])) return DFLASH_E_ALIGN;
  }
  if (!aligned16(w_fc) || !aligned16(w_k) || !aligned16(w_v)) return DFLASH_E_ALIGN;
  if (cache->page_table) {
    if (!cache->free_list || !cache->free_count || cache->page_size < 1 || cache->max_pages < 1)
      return DFLASH_E_ARG;
  } else if (cache->capacity < kBlock) {
    return DFLASH_E_ARG;
  }
  if (!ws) return DFLASH_E_WORKSPACE;
  Plan plan;
  if ((rc = make_plan(*dims, &plan))) return rc;
  if (ws_bytes < plan.total) return DFLASH_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int H = dims->hidden, ntok = plan.ntok;
  const int kvd = dims->n_kv_heads * dims->head_dim;
  uint32_t* status = ws_at<uint32_t>(ws, plan.off_status);
  float* part_fc = ws_at<float>(ws, plan.off_fc);
  uint16_t* yhat = ws_at<uint16_t>(ws, plan.off_yhat);
  float* part_kv = ws_at<float>(ws, plan.off_kv);
  int32_t* pos_snap = ws_at<int32_t>(ws, plan.off_pos);

  GemmParams common = {};
  common.status = status;
  common.hidden = H;
  common.fc_out_tiles = plan.fc_out_tiles;
  common.rms_eps = dims->rms_eps;
  common.hidden_norm_w = static_cast<const uint16_t*>(hidden_norm_w);
  common.yhat = yhat;
  common.ss = ws_at<float>(ws, plan.off_ss);
  common.batch = dims->batch;
  common.write_pos = write_pos;
  common.pos_snapshot = pos_snap;
  common.cache = *cache;
  common.n_kv_heads = dims->n_kv_heads;
  common.head_dim = dims->head_dim;
  common.k_norm_w = static_cast<const uint16_t*>(k_norm_w);
  fill_rope_table(common.rope.hi, common.rope.lo, dims->head_dim, dims->rope_theta);
  uint32_t* tickets = ws_at<uint32_t>(ws, plan.off_ctx_tickets);

  // ---- 1. fc GEMM; its finisher writes hi/lo of g_h * Y and sums of Y^2 ----
  {
    GemmParams g = common;
    g.mode = kModeFc;
    g.k_tiles = plan.fc_k_tiles;
    g.out_tiles = plan.fc_out_tiles;
    g.a_split = plan.fc_out_tiles;
    g.layer_cols = H;
    g.n_tok = ntok;
    g.chunk_rows = ntok < 256 ? ntok : 256;
    g.n_chunks = plan.fc_tok_chunks;
    g.hilo = 0;
    g.ld_out = H;
    g.mma_n = g.chunk_rows;
    g.acc = part_fc;
    g.tickets = tickets;
    const int smem = setup_gemm(g, g.chunk_rows);
    CUtensorMap ta;
    if ((rc = make_tmap_2d_bf16(&ta, w_fc, static_cast<uint64_t>(nL) * H, H,
                                static_cast<uint64_t>(nL) * H * 2, 64, 128)))
      return rc;
    LayerMaps lm;
    for (int l = 0; l < nL; ++l)
      if ((rc = make_tmap_2d_bf16(&lm.m[l], layer_hidden[l], H, ntok,
                                  static_cast<uint64_t>(H) * 2, 64, g.chunk_rows)))
        return rc;
    for (int l = nL; l < kMaxCtxLayers; ++l) lm.m[l] = lm.m[0];
    if ((rc = set_smem_limit(reinterpret_cast<const void*>(streamk_gemm_kernel), smem))) return rc;
    const int grid = streamk_grid(g, plan.budget_sms);
    if ((rc = launch(streamk_gemm_kernel, dim3(grid), dim3(kGemmThreads), smem, st, ta, ta, lm, g)))
      return rc;
  }
  // ---- 2. K/V GEMM on [hi; lo]; its finisher scales, normalises, rotates, stores ----
  {
    GemmParams g = common;
    g.mode = kModeKv;
    g.k_tiles = plan.kv_k_tiles;
    g.out_tiles = plan.kv_out_tiles;
    g.a_split = plan.kv_out_tiles / 2;
    g.layer_cols = H;
    g.n_tok = ntok;
    g.chunk_rows = ntok < 128 ? ntok : 128;
    g.n_chunks = plan.kv_tok_chunks;
    g.hilo = 1;
    g.ld_out = 2 * kvd;
    g.mma_n = 2 * g.chunk_rows;
    g.acc = part_kv;
    g.tickets = tickets + plan.fc_out_tiles * plan.fc_tok_chunks;
    const int smem = setup_gemm(g, 2 * g.chunk_rows);
    CUtensorMap tk, tv;
    if ((rc = make_tmap_2d_bf16(&tk, w_k, H, kvd, static_cast<uint64_t>(H) * 2, 64, 128)))
      return rc;
    if ((rc = make_tmap_2d_bf16(&tv, w_v, H, kvd, static_cast<uint64_t>(H) * 2, 64, 128)))
      return rc;
    LayerMaps lm;
    if ((rc = make_tmap_2d_bf16(&lm.m[0], yhat, H, 2 * static_cast<uint64_t>(ntok),
                                static_cast<uint64_t>(H) * 2, 64, g.chunk_rows)))
      return rc;
    for (int l = 1; l < kMaxCtxLayers; ++l) lm.m[l] = lm.m[0];
    if ((rc = set_smem_limit(reinterpret_cast<const void*>(streamk_gemm_kernel), smem))) return rc;
    const int grid = streamk_grid(g, plan.budget_sms);
    if ((rc = launch(streamk_gemm_kernel, dim3(grid), dim3(kGemmThreads), smem, st, tk, tv, lm, g)))
      return rc;
  }
  return DFLASH_OK;
}
