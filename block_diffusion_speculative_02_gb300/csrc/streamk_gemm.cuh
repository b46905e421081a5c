// Stream-K skinny GEMM on the 5th-generation tensor cores, shared by the
// context projection and the drafter layer.
//
// Y[n_tok, N] = B[n_tok, K] W[N, K]^T computed "swap-AB": 128 output features
// are the MMA's M, the token rows its N, fp32 accumulators live in TMEM, the
// weight stream is staged by a TMA pipeline.  At small batch the GEMM is bound
// by the weight stream, so the work is cut into units of (output tile of 128
// features x token chunk, k-stage) and CTA i of the grid (one per SM of the
// budget) streams units [U*i/G, U*(i+1)/G): every CTA moves the same number
// of weight bytes whatever the tile count.  A CTA's range crosses tile
// boundaries; each piece accumulates in one of two TMEM slots (the epilogue
// drains one while the MMAs fill the other) and is stored as an fp32 partial
// tile in the workspace, in the slot of its piece index (the CTA's rank among
// the tile's contributors).  The CTA whose atomic ticket completes a tile's
// count of contributions (a closed form of the partition) runs the finisher
// policy `Fin` on it once its own pipeline has drained: the pieces are added
// in index order into shared memory and the finisher reads those sums, so
// the result does not depend on the order in which the CTAs arrive: the same
// inputs and grid give the same bits on every run.
//
// The weight matrix may be split over up to three tensor maps (tiles below
// a_split[0] read map 0, ...), and the token matrix over up to eight maps
// along K (k-tile kt reads map (kt * 64) / layer_cols): that is how the
// context projection reads the concatenation of the target's layers without
// materialising it.  With hilo set the token matrix is a pair [hi; lo] of
// bf16 rows whose products are added in the epilogue (an fp32 operand carried
// as two bf16 halves).
#pragma once

#include "common.cuh"
#include "host.h"

namespace dflash {
namespace sk {

constexpr int kGemmThreads = 192;
constexpr int kATile = 128 * 128;  // 128 rows x 64 bf16
constexpr int kMaxGemmStages = 12;
constexpr int kMaxSegments = 32;   // tiles one CTA may touch
constexpr int kMaxAMaps = 3;
#ifndef DFLASH_GEMM_CHUNKS_PER_STAGE
#define DFLASH_GEMM_CHUNKS_PER_STAGE 4
#endif
constexpr int kGemmChunksPerStage = DFLASH_GEMM_CHUNKS_PER_STAGE;

struct AMaps {
  CUtensorMap m[kMaxAMaps];
};

struct BMaps {
  CUtensorMap m[kMaxCtxLayers];
};

struct GemmCore {
  int k_tiles;       // K / 64
  int k_stages;      // ceil(k_tiles / kb): work units per tile
  int n_units;       // out_tiles * n_chunks * k_stages
  int out_tiles;     // output features / 128
  int a_split[kMaxAMaps - 1];  // first tile of weight maps 1 and 2
  int pair_stride;   // > 0: tiles o and o + pair_stride are finished together
  int layer_cols;    // columns per B map; k-tile kt reads map (kt*64)/layer_cols
  int n_tok;
  int chunk_rows;    // token rows per chunk (B box rows)
  int n_chunks;
  int hilo;          // 1: B = [hi rows ; lo rows] of a 2*n_tok-row matrix, summed in the epilogue
  int mma_n;         // MMA N = chunk_rows * (1 + hilo)
  int n_stages, stage_bytes, tmem_cols;
  int kb;            // 64-column K chunks per pipeline stage
  int b_chunk;       // bytes of the token tile of one chunk (1024-aligned)
  int max_pieces;    // partial-tile slots per tile (max_pieces() of the shape)
  float* part;       // [n_chunks * out_tiles][max_pieces][chunk_rows][128] fp32 partial tiles
  uint32_t* tickets; // [n_chunks * out_tiles] contributions so far, zero between calls
  uint32_t* status;
};

// Unit u = (tile T, k-stage ks) with u = T * k_stages + ks; tile T covers
// output features (T % out_tiles) * 128 .. +127 for token chunk T / out_tiles.
// CTA i of G streams units [U*i/G, U*(i+1)/G): every CTA moves the same
// number of weight bytes whatever the tile count.
__device__ __forceinline__ int unit_begin(const GemmCore& p, int i) {
  return static_cast<int>(static_cast<long long>(p.n_units) * i / gridDim.x);
}

// The CTA whose unit range holds unit u.
__device__ __forceinline__ int unit_owner(const GemmCore& p, int u) {
  return static_cast<int>((static_cast<long long>(gridDim.x) * (u + 1) - 1) / p.n_units);
}

// Number of CTAs that add partial sums into tile T.
__device__ __forceinline__ uint32_t tile_contributors(const GemmCore& p, int T) {
  const int first = T * p.k_stages;
  const int last = min(p.n_units, first + p.k_stages) - 1;
  return static_cast<uint32_t>(unit_owner(p, last) - unit_owner(p, first) + 1);
}

// Tiles are finished one by one, or -- pair_stride > 0 -- in pairs (o,
// o + pair_stride) of one token chunk, o < pair_stride: the pair's ticket is
// that of its first tile and counts the contributions to both.
__device__ __forceinline__ int ticket_tile(const GemmCore& p, int T) {
  if (p.pair_stride == 0) return T;
  const int o = T % p.out_tiles;
  return o < p.pair_stride ? T : T - p.pair_stride;
}

__device__ __forceinline__ uint32_t ticket_target(const GemmCore& p, int Tt) {
  return p.pair_stride == 0 ? tile_contributors(p, Tt)
                            : tile_contributors(p, Tt) + tile_contributors(p, Tt + p.pair_stride);
}

// Finishing a tile: its contributors' partial tiles are first added in piece
// order 0, 1, ... (a fixed order, so the sum is reproducible bit for bit) by
// all 128 epilogue threads, with up to kGatherLoads loads of each thread in
// flight, into shared memory at kFinSumsOffset (the pipeline stages are free
// by then): slot 0 holds the ticket tile, slot 1 its partner when tiles are
// finished in pairs, each [chunk_rows][128] fp32.  The finisher then reads
// the sums with take4.  The first kFinSumsOffset bytes stay the finisher's
// own scratch.
constexpr int kFinSumsOffset = 16 * 1024;
constexpr int kGatherPieces = 4;   // pieces of one position loaded together
constexpr int kGatherPos = 4;      // float4 positions of one thread loaded together

extern __shared__ uint8_t sk_dyn_smem[];

__device__ __forceinline__ float* fin_sums() {
  return reinterpret_cast<float*>(align_smem_1024(sk_dyn_smem) + kFinSumsOffset);
}

// Shared memory the finishing phase needs beyond the alignment slack.
inline int fin_smem_bytes(const GemmCore& g) {
  return kFinSumsOffset + (g.pair_stride > 0 ? 2 : 1) * g.chunk_rows * 128 * 4;
}

// Sum the pieces of tile T (token chunk c) into sums slot `slot` (epilogue
// threads et = 0..127).
__device__ __forceinline__ void gather_tile(const GemmCore& g, int T, int slot, int et) {
  const int c = T / g.out_tiles;
  const int nt = min(g.chunk_rows, g.n_tok - c * g.chunk_rows);
  const int n = static_cast<int>(tile_contributors(g, T));
  const float4* src = reinterpret_cast<const float4*>(
      g.part + static_cast<size_t>(T) * g.max_pieces * g.chunk_rows * 128);
  const size_t stride = static_cast<size_t>(g.chunk_rows) * 32;  // float4s between pieces
  float4* dst = reinterpret_cast<float4*>(fin_sums()) + slot * g.chunk_rows * 32;
  const int n_pos = nt * 32;                                     // float4s of the tile
  for (int q0 = et; q0 < n_pos; q0 += 128 * kGatherPos) {
    float4 s[kGatherPos];
    for (int i0 = 0; i0 < n; i0 += kGatherPieces) {
      float4 v[kGatherPos][kGatherPieces];
#pragma unroll
      for (int a = 0; a < kGatherPos; ++a)
#pragma unroll
        for (int i = 0; i < kGatherPieces; ++i)
          if (q0 + 128 * a < n_pos && i0 + i < n)
            v[a][i] = __ldcg(src + (i0 + i) * stride + q0 + 128 * a);
#pragma unroll
      for (int a = 0; a < kGatherPos; ++a)
#pragma unroll
        for (int i = 0; i < kGatherPieces; ++i) {
          if (i0 + i >= n) break;
          if (i0 + i == 0) {
            s[a] = v[a][0];
          } else {
            s[a].x += v[a][i].x;
            s[a].y += v[a][i].y;
            s[a].z += v[a][i].z;
            s[a].w += v[a][i].w;
          }
        }
    }
#pragma unroll
    for (int a = 0; a < kGatherPos; ++a)
      if (q0 + 128 * a < n_pos) dst[q0 + 128 * a] = s[a];
  }
}

// The finished sums of 4 consecutive features f0..f0+3 (global feature index)
// of token row `tok`, inside a finisher: slot 1 for the partner tile of a pair.
__device__ __forceinline__ float4 take4(const GemmCore& g, int tok, int f0) {
  const int r = tok % g.chunk_rows;
  const int slot = (g.pair_stride > 0 && ((f0 >> 7) % g.out_tiles) >= g.pair_stride) ? 1 : 0;
  return *reinterpret_cast<const float4*>(fin_sums() + (slot * g.chunk_rows + r) * 128 +
                                          (f0 & 127));
}

template <class Fin>
__global__ void __launch_bounds__(kGemmThreads, 1)
streamk_gemm_kernel(const __grid_constant__ AMaps tm_a, const __grid_constant__ BMaps tm_b,
                    const GemmCore p, const __grid_constant__ typename Fin::Params fp) {
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
        const bool a1 = o >= p.a_split[0], a2 = o >= p.a_split[1];
        const CUtensorMap* ma = a2 ? &tm_a.m[2] : (a1 ? &tm_a.m[1] : &tm_a.m[0]);
        const int arow = (o - (a2 ? p.a_split[1] : (a1 ? p.a_split[0] : 0))) * 128;
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
    if (blockIdx.x == 0) Fin::prologue(p, fp);
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
      // this CTA's piece of the tile goes to its own slot: rank among the
      // tile's contributors = this CTA's index - the first contributor's
      const int piece = static_cast<int>(blockIdx.x) - unit_owner(p, T * KS);
      float* dst = p.part +
                   (static_cast<size_t>(T) * p.max_pieces + piece) * p.chunk_rows * 128 +
                   q * 32 + lane;
      for (int c0 = 0; c0 < p.chunk_rows; c0 += 16) {
        uint32_t v[16], w[16];
        tmem_ld_32x32b_x16(tacc + c0, v);
        if (p.hilo) tmem_ld_32x32b_x16(tacc + p.chunk_rows + c0, w);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int r = c0 + j;
          float val = __uint_as_float(v[j]);
          if (p.hilo) val += __uint_as_float(w[j]);
          if (c * p.chunk_rows + r < p.n_tok) __stcg(dst + static_cast<size_t>(r) * 128, val);
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[slot]);
      __threadfence();
      named_bar_sync(1, 128);
      if (et == 0) {
        const int Tt = ticket_tile(p, T);
        if (atomicAdd(p.tickets + Tt, 1u) == ticket_target(p, Tt) - 1u)
          fin_tiles[(*n_fin)++] = Tt;  // this CTA completed the tile's (or pair's) sum
      }
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
      gather_tile(p, T, 0, threadIdx.x - 64);
      if (p.pair_stride > 0) gather_tile(p, T + p.pair_stride, 1, threadIdx.x - 64);
      named_bar_sync(1, 128);
      Fin::finish(p, fp, o, c, smem);
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

inline int gemm_smem(int stage_bytes, int n_stages) {
  return 1024 + n_stages * (stage_bytes + 16) + kGemmTail;
}

inline int setup_gemm(GemmCore& g, int b_rows_per_stage) {
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
inline int streamk_grid(const GemmCore& g, int ctas) {
  int grid = ctas < g.n_units ? ctas : g.n_units;
  while (grid < g.n_units) {
    const int per = (g.n_units + grid - 1) / grid;
    if ((per + g.k_stages - 1) / g.k_stages + 1 <= kMaxSegments) break;
    ++grid;
  }
  return grid;
}

// The shape fields of a GEMM of n_tok token rows, K = k_cols, out_tiles
// tiles of 128 features: token chunks of up to 256 rows (128 with hilo, whose
// MMA N is twice the chunk).  The launches and the workspace plans both start
// from it.
inline GemmCore gemm_dims(int n_tok, int k_cols, int out_tiles, int hilo) {
  GemmCore g = {};
  g.k_tiles = k_cols / 64;
  g.out_tiles = out_tiles;
  g.a_split[0] = g.a_split[1] = out_tiles;
  g.layer_cols = k_cols;
  g.n_tok = n_tok;
  const int cap = hilo ? 128 : 256;
  g.chunk_rows = n_tok < cap ? n_tok : cap;
  g.n_chunks = (n_tok + g.chunk_rows - 1) / g.chunk_rows;
  g.hilo = hilo;
  g.mma_n = (1 + hilo) * g.chunk_rows;
  return g;
}

// Partial-tile slots per tile: an upper bound on the CTAs that add a piece
// to one tile, over every grid streamk_grid may choose on a device of nsm SMs
// (any SM budget).  A CTA streams at least floor(U / G) units, so a tile of
// KS consecutive units meets at most (KS - 1) / floor(U / G) + 2 CTAs; the
// bound grows with G, whose largest value is max(min(nsm, U), streamk_grid(g, 1)).
// The result depends on the shape fields of gemm_dims and on nsm only.
inline int max_pieces(const GemmCore& shape, int nsm) {
  GemmCore g = shape;
  setup_gemm(g, (1 + g.hilo) * g.chunk_rows);
  int gmax = nsm < g.n_units ? nsm : g.n_units;
  const int gstar = streamk_grid(g, 1);
  if (gstar > gmax) gmax = gstar;
  const int per = g.n_units / gmax;
  int m = (g.k_stages - 1) / per + 2;
  if (m > g.k_stages) m = g.k_stages;
  if (m > gmax) m = gmax;
  return m;
}

// Bytes of the partial-tile buffer of a GEMM of this shape on nsm SMs.
inline size_t partial_bytes(const GemmCore& shape, int nsm) {
  return sizeof(float) * static_cast<size_t>(shape.out_tiles) * shape.n_chunks *
         max_pieces(shape, nsm) * shape.chunk_rows * 128;
}

// Launch one stream-K GEMM with finisher Fin on at most `ctas` CTAs (fills
// the pipeline fields of g; the token tile of a stage holds (1 + hilo) *
// chunk_rows rows).  g.part must hold partial_bytes(g, SM count) bytes
// (part_cap, else DFLASH_E_WORKSPACE).
template <class Fin>
inline int run_streamk(GemmCore& g, const AMaps& a, const BMaps& b,
                       const typename Fin::Params& fp, int ctas, cudaStream_t st,
                       size_t part_cap) {
  const int nsm = current_num_sms();
  if (nsm <= 0) return DFLASH_E_CUDA;
  if (partial_bytes(g, nsm) > part_cap) return DFLASH_E_WORKSPACE;
  g.max_pieces = max_pieces(g, nsm);
  const int smem = setup_gemm(g, (1 + g.hilo) * g.chunk_rows);
  // the finisher's sums reuse the stage area, below the barriers
  if (fin_smem_bytes(g) > g.n_stages * g.stage_bytes) return DFLASH_E_UNSUPPORTED;
  int rc = set_smem_limit(reinterpret_cast<const void*>(streamk_gemm_kernel<Fin>), smem);
  if (rc) return rc;
  const int grid = streamk_grid(g, ctas < nsm ? ctas : nsm);
  return launch(streamk_gemm_kernel<Fin>, dim3(grid), dim3(kGemmThreads), smem, st, a, b, g, fp);
}

}  // namespace sk
}  // namespace dflash
