// a2 — dual-source block attention of the drafter.
//
// "DFlash双实现对比" (hotelren.com) §2: Q comes only from the 16 block tokens;
// K/V is the concatenation of the context K/V (projected from the target's
// hidden states) with the block's own K/V; there is no causal mask inside the
// block.  "dflash-mlx" (dpshk.com) 块扩散草稿: the staged token and 15 masks
// are denoised in one parallel forward that reads the target's hidden states.
//
// Design (GB300): grid = (split, KV head, sequence).  Each CTA owns one KV
// head of one sequence and a page-aligned slice of its context, so the
// G = Hq/Hkv query heads sharing the KV head (R = 16 G query rows) read every
// KV byte once.  The two products run on the 5th-generation tensor cores with
// the query rows as the MMA's M (128 rows; R/4 real rows per 32-lane TMEM
// quadrant, so all four warps of the softmax work):
//   S = Q K^T   (M = 128, N = keys of the chunk, K = D)   -> TMEM, two buffers
//   O += P V    (M = 128, N = D, K = keys; V is read MN-major) -> TMEM
// One warp streams 64-key chunks of K and V with TMA (one 16-row box per
// page and 64-wide half of the head dim, or one 64-row box for a whole
// contiguous chunk; 128-byte swizzle), one thread issues the MMAs, and one
// thread pair per query row runs the online softmax straight from TMEM (for
// R <= 64 every query row is staged twice, at lanes i and i + 16 of its
// quadrant, and the pair splits the chunk's keys): row max, exp2, row sum,
// bf16 P into shared memory for the next MMA.  The running
// max only moves (and O in TMEM is rescaled) when a chunk raises it by more
// than 2^8, so P stays below 256 and rescales are rare.  The S MMA of chunk
// j + 1 overlaps the softmax of chunk j.  RoPE of the block queries and keys
// is applied while they are staged into shared memory, at positions L + i,
// from a sin/cos table of the 16 block positions built once per CTA.
// The split that owns the tail also folds in the 16 block keys (a 16-key
// chunk).  Partial (O, max, sum) go to the workspace and a second kernel
// merges the splits by log-sum-exp.
//
// The same kernel serves the target's attention: the verify forward (causal
// inside the block, the block's K/V appended to the cache) and the prefill
// of a prompt chunk of T rows.  A chunk is cut into 16-row sub-blocks; its
// rotated K and its V are first appended to the cache, then sub-block j (at
// positions L + 16 j ..) is a causal block whose context is the cache rows
// 0 .. L + 16 j - 1, which is causal attention over the whole chunk.  The
// grid's z index runs over (sequence, sub-block) with the longest contexts
// first, and with a single split the kernel writes the bf16 output itself.
#include <type_traits>

#include "common.cuh"
#include "host.h"

namespace dflash {
namespace {

constexpr int kChunk = 64;     // keys per pipeline stage
constexpr int kPage = 16;      // rows per TMA box
constexpr int kAttThreads = 320;  // TMA, MMA, two softmax warpgroups
// TMEM columns: S buffers at 0 and 64, the O accumulator at 128
template <int D>
__host__ __device__ constexpr int tmem_cols() { return 128 + D <= 256 ? 256 : 512; }
constexpr float kRescaleLog2 = 8.0f;

struct AttnParams {
  int batch, n_q_heads, n_kv_heads, group, splits, rows;  // rows R = group << sub_shift
  int paged, capacity, max_pages;
  // block rows: q/k/v row b * tokens + (j << sub_shift) + i for sub-block j
  // of sequence b (tokens = 16, sub_blocks = 1 for a single block); a
  // sequence is valid when 0 <= seq_len[b] and seq_len[b] + need_rows fits
  // the cache
  int tokens, sub_blocks, need_rows;
  // rows per sub-block = 1 << sub_shift (16, or 32 for the prompt attention
  // when G * 32 query rows fit the 128 MMA rows); self_cached: the sub-block's
  // own keys are already in the cache (the prompt attention appends first)
  // and are read with the context under a per-row causal limit, with no
  // block tile
  int sub_shift, self_cached;
  uint16_t* out_direct;  // splits == 1: bf16 output [B * tokens, Hq, D] written here
  const int32_t* seq_len;
  const int32_t* page_table;
  const uint16_t* q_blk;
  const uint16_t* k_blk;
  const uint16_t* v_blk;
  float scale_log2;
  float* part_o;
  float* part_ml;
  uint32_t* status;
  // the target's verify attention: causal inside the block, and the block's
  // rotated K and its V appended to the cache at rows L .. L + 15
  int causal;
  uint16_t* k_app;
  uint16_t* v_app;
  // shared-memory plan (byte offsets from the 1024-aligned base)
  int n_stages, off_q, off_st, off_blk, off_sc, off_xch, off_rope, off_bar;
  RopeTable rope;
};

struct CombineParams {
  int batch, n_q_heads, n_kv_heads, group, splits, rows, head_dim, limit;
  int tokens, sub_blocks, need_rows, sub_shift;
  const int32_t* seq_len;
  const float* part_o;
  const float* part_ml;
  uint16_t* out;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return static_cast<uint32_t>(float_to_bf16_bits(lo)) |
         (static_cast<uint32_t>(float_to_bf16_bits(hi)) << 16);
}

// 2^x on the special-function unit (one instruction; -inf gives +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct Cfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalf = kChunk * 128;              // one 64-col half of a chunk
  static constexpr int kTile = kHalves * kHalf;           // K or V of one 64-key chunk
  static constexpr int kStage = 2 * kTile;
  // the 16 block rows of K and V share one tile with the half stride of a
  // chunk: K in rows 0..15 of each half, V in rows 16..31
  static constexpr int kBlkTile = (kHalves - 1) * kHalf + 2 * kPage * 128;
  static constexpr int kBlkV = kPage * 128;
};

// Byte offset of (row, 16-byte chunk `c` of the 128-byte row) in a tile of
// rows x 128 B with the 128-byte swizzle (row stride 128 B).
__device__ __forceinline__ int swz_off(int row, int c) {
  return row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

// Rotate 8 consecutive dims (x1: d0..d0+7) against their partners (x2:
// d0+D/2..) with the (cos, sin) pairs sc[d0..d0+7] of one position; bf16 in,
// bf16 out.
__device__ __forceinline__ void rope8(const uint4& x1, const uint4& x2, const float2* sc, int d0,
                                      uint4& y1, uint4& y2) {
  const uint32_t w1[4] = {x1.x, x1.y, x1.z, x1.w}, w2[4] = {x2.x, x2.y, x2.z, x2.w};
  uint32_t r1[4], r2[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float o1[2], o2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float2 cs = sc[d0 + 2 * q + e];
      const float a = __uint_as_float(e ? (w1[q] & 0xFFFF0000u) : (w1[q] << 16));
      const float c = __uint_as_float(e ? (w2[q] & 0xFFFF0000u) : (w2[q] << 16));
      o1[e] = a * cs.x - c * cs.y;
      o2[e] = c * cs.x + a * cs.y;
    }
    r1[q] = pack_bf16(o1[0], o1[1]);
    r2[q] = pack_bf16(o2[0], o2[1]);
  }
  y1 = make_uint4(r1[0], r1[1], r1[2], r1[3]);
  y2 = make_uint4(r2[0], r2[1], r2[2], r2[3]);
}

template <int D, bool DUP>
__global__ void __launch_bounds__(kAttThreads, 1) block_attention_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ CUtensorMap tm_k64, const __grid_constant__ CUtensorMap tm_v64,
    const AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  const int R = p.rows;
  const int NS = p.n_stages;
  const int rq = R / 4;                        // real query rows per TMEM quadrant
  constexpr bool dup = DUP;                    // rows staged twice (lanes i, i + 16): R <= 64
  constexpr int kPBytes = 128 * 128;           // one P buffer: 128 rows x 64 keys bf16
  constexpr int kQHalf = 128 * 128;            // one 64-dim half of Q: 128 rows
  uint8_t* qs = smem + p.off_q;                // Q: [half][128 rows][128 B]
  uint8_t* stg = smem + p.off_st;
  uint8_t* blk = smem + p.off_blk;
  float2* sct = reinterpret_cast<float2*>(smem + p.off_sc);  // [16 positions][D/2] (cos, sin)
  float* rope_hi = reinterpret_cast<float*>(smem + p.off_rope);
  float* rope_lo = rope_hi + D / 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* empty = full + NS;
  uint64_t* s_full = empty + NS;   // [2] S(j) in TMEM buffer j & 1
  uint64_t* p_full = s_full + 2;   // [2] P(j) in shared buffer j & 1 (and O rescaled)
  uint64_t* pv_done = p_full + 2;  // [2] O += P(j) V(j) completed
  uint64_t* q_ready = pv_done + 2; // Q and the block tile staged (256 arrivals)
  uint64_t* o_done = q_ready + 1;
  uint64_t* mdrain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdrain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int s_idx = blockIdx.x, g = blockIdx.y;
  // (sequence, sub-block): the last sub-block, with the longest context, first
  const int b = blockIdx.z / p.sub_blocks;
  const int jsub = p.sub_blocks - 1 - (static_cast<int>(blockIdx.z) - b * p.sub_blocks);
  const int sub_rows = 1 << p.sub_shift;
  const int row0 = b * p.tokens + (jsub << p.sub_shift);  // first block row in q/k/v
  const int n_rows = min(sub_rows, p.tokens - (jsub << p.sub_shift));

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 256);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(q_ready, 256);
    mbar_init(o_done, 1);
    mbar_init(mdrain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < D / 2; i += blockDim.x) {
    rope_hi[i] = p.rope.hi[i];
    rope_lo[i] = p.rope.lo[i];
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_k64);
    tma_prefetch_desc(&tm_v64);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols<D>());
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();

  const int L0 = p.seq_len[b];
  const int limit = p.paged ? p.max_pages * kPage : p.capacity;
  const bool valid_len = L0 >= 0 && L0 + p.need_rows <= limit;
  if (!valid_len && threadIdx.x == 0 && s_idx == 0 && g == 0 && jsub == 0)
    set_status(p.status, DFLASH_ST_CAPACITY);
  const int L = L0 + (jsub << p.sub_shift);     // position of the sub-block's first row
  // keys read from the cache: the context, and the sub-block's own rows too
  // when they are already there
  const int Lc = valid_len ? (p.self_cached ? L + n_rows : L) : 0;
  const int Lq = valid_len ? L : 0;             // position of the block's row 0
  const int n_pg = (Lc + kPage - 1) / kPage;
  const int pps = (n_pg + p.splits - 1) / p.splits;
  const int pg_begin = s_idx * pps;
  const int pg_end = min(pg_begin + pps, n_pg);
  const int key_begin = pg_begin * kPage;
  const int key_end = min(pg_end * kPage, Lc);
  const int n_keys = key_end > key_begin ? key_end - key_begin : 0;
  const int n_chunks = (n_keys + kChunk - 1) / kChunk;
  const int has_block = (valid_len && !p.self_cached && s_idx == p.splits - 1) ? 1 : 0;
  const int n_total = n_chunks + has_block;    // chunk 0 is the block when has_block
  auto chunk_keys = [&](int j) {               // valid keys of chunk j
    if (has_block && j == 0) return kPage;
    return min(kChunk, key_end - (key_begin + (j - has_block) * kChunk));
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      for (int c = 0; c < n_chunks; ++c) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) break;
        uint8_t* kst = stg + stage * C::kStage;
        uint8_t* vst = kst + C::kTile;
        const int k0 = key_begin + c * kChunk;
        const int npg = min(kChunk / kPage, (key_end - k0 + kPage - 1) / kPage);
        // head-major caches: a page (16 rows) of one head is 16 * D contiguous
        // elements, a contiguous cache holds each head's rows back to back
        const int slab = b * p.n_kv_heads + g;
        if (!p.paged && npg == kChunk / kPage) {
          mbar_arrive_expect_tx(&full[stage], 2u * C::kHalves * kChunk * 128);
          for (int h = 0; h < C::kHalves; ++h) {
            tma_load_3d(kst + h * C::kHalf, &tm_k64, &full[stage], h * 64, k0, slab, pol);
            tma_load_3d(vst + h * C::kHalf, &tm_v64, &full[stage], h * 64, k0, slab, pol);
          }
        } else {
          int zc[kChunk / kPage];  // third coordinate of each page's box, -1 = unmapped
          uint32_t bytes = 0;
          for (int j = 0; j < npg; ++j) {
            const int lp = k0 / kPage + j;
            int z;
            if (p.paged) {
              const int id = p.page_table[static_cast<size_t>(b) * p.max_pages + lp];
              z = id >= 0 ? id * p.n_kv_heads + g : -1;
            } else {
              z = slab;
            }
            zc[j] = z;
            if (z >= 0) bytes += 2u * C::kHalves * kPage * 128;
          }
          // unmapped pages inside the length read as zeros
          bool zeroed = false;
          for (int j = 0; j < npg; ++j) {
            if (zc[j] >= 0) continue;
            set_status(p.status, DFLASH_ST_PAGE_MISSING);
            for (int h = 0; h < C::kHalves; ++h) {
              uint4* kz = reinterpret_cast<uint4*>(kst + h * C::kHalf + j * kPage * 128);
              uint4* vz = reinterpret_cast<uint4*>(vst + h * C::kHalf + j * kPage * 128);
              for (int i = 0; i < kPage * 128 / 16; ++i) kz[i] = vz[i] = make_uint4(0, 0, 0, 0);
            }
            zeroed = true;
          }
          if (zeroed) fence_proxy_async_smem();
          if (bytes) {
            mbar_arrive_expect_tx(&full[stage], bytes);
            for (int j = 0; j < npg; ++j) {
              if (zc[j] < 0) continue;
              const int row = p.paged ? 0 : k0 + j * kPage;
              for (int h = 0; h < C::kHalves; ++h) {
                tma_load_3d(kst + h * C::kHalf + j * kPage * 128, &tm_k, &full[stage], h * 64,
                            row, zc[j], pol);
                tma_load_3d(vst + h * C::kHalf + j * kPage * 128, &tm_v, &full[stage], h * 64,
                            row, zc[j], pol);
              }
            }
          } else {
            mbar_arrive(&full[stage]);
          }
        }
        ++issued;
        if (++stage == static_cast<uint32_t>(NS)) {
          stage = 0;
          phase ^= 1;
        }
      }
      // no copy may still be landing when the CTA exits
      for (int st = 0; st < NS && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / NS) * NS;
        mbar_wait_drain(&full[st], static_cast<uint32_t>((last / NS) & 1), p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && n_total > 0) {
      const uint32_t q_addr = smem_u32(qs);
      const uint32_t blk_addr = smem_u32(blk);
      const uint32_t st_addr = smem_u32(stg);
      const uint32_t p_addr = smem_u32(smem);    // P buffers at offsets 0 and kPBytes
      const uint32_t o_tmem = tmem_base + 128;
      const uint32_t idesc_pv = umma_idesc_bf16(128, D) | (1u << 16);  // B (= V) MN-major
      bool ok = mbar_wait(q_ready, 0, abort_flag, p.status);
      tc_fence_after();
      // S(j) = Q K_j^T into TMEM buffer j & 1
      auto issue_s = [&](int j) -> bool {
        const int nk = chunk_keys(j);
        const int ncol = (nk + 15) & ~15;
        uint32_t kb;
        if (has_block && j == 0) {
          kb = blk_addr;
        } else {
          const int c = j - has_block;
          if (!mbar_wait(&full[c % NS], static_cast<uint32_t>((c / NS) & 1), abort_flag, p.status))
            return false;
          tc_fence_after();
          kb = st_addr + (c % NS) * C::kStage;
        }
        const uint32_t idesc = umma_idesc_bf16(128, ncol);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = umma_sdesc_sw128(q_addr + (kk >> 2) * kQHalf + (kk & 3) * 32);
          const uint64_t bd = umma_sdesc_sw128(kb + (kk >> 2) * C::kHalf + (kk & 3) * 32);
          umma_bf16(tmem_base + (j & 1) * 64, a, bd, idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[j & 1]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && n_total > 1) ok = issue_s(1);
      for (int j = 0; ok && j < n_total; ++j) {
        if (!mbar_wait(&p_full[j & 1], static_cast<uint32_t>((j >> 1) & 1), abort_flag, p.status))
          break;
        tc_fence_after();
        const bool is_blk = has_block && j == 0;
        const int c = j - has_block;
        const uint32_t vb = is_blk ? blk_addr + C::kBlkV : st_addr + (c % NS) * C::kStage + C::kTile;
        const int ksteps = (chunk_keys(j) + 15) >> 4;
        for (int ks = 0; ks < ksteps; ++ks) {
          const uint64_t a = umma_sdesc_sw128(p_addr + (j & 1) * kPBytes + ks * 32);
          const uint64_t bd = umma_sdesc_sw128_mn(vb + ks * 2048, C::kHalf, 1024);
          umma_bf16(o_tmem, a, bd, idesc_pv, (j >= 1 || ks > 0) ? 1u : 0u);
        }
        umma_commit(&pv_done[j & 1]);
        if (!is_blk) umma_commit(&empty[c % NS]);
        if (j + 2 < n_total && !issue_s(j + 2)) break;
      }
      umma_commit(o_done);
      umma_commit(mdrain);
      mbar_wait_drain(mdrain, 0, p.status);
    }
  } else {
    // ---------------- staging, then softmax (warps 2..9) ----------------
    const int tid = threadIdx.x - 64;            // 0 .. 255
    // Q rows (rr = w * 16 + i for query head g * G + w) rotated at L + i, and
    // the block's K (rotated at L + j) and V, into the swizzled K-major tiles.
    // Q row rr goes to MMA row 32 (rr / rq) + rr % rq, and again 16 rows
    // further when rows are doubled.  Items of 8 dims with their rotary
    // partners; this thread's loads go out before the sin/cos table is built.
    {
      constexpr int kPer = D / 16;               // items per row
      constexpr int kMaxItems = 128 * kPer / 256;  // items per thread at R = 128
      const int q_items = R * kPer;
      uint4 x1[kMaxItems], x2[kMaxItems];
#pragma unroll
      for (int u = 0; u < kMaxItems; ++u) {
        const int it = u * 256 + tid;
        if (it < q_items) {
          const int rr = it / kPer, d0 = (it - rr * kPer) * 8;
          const int w = rr >> p.sub_shift, i = rr & (sub_rows - 1);
          if (i < n_rows) {
            const size_t src =
                (static_cast<size_t>(row0 + i) * p.n_q_heads + g * G + w) * D + d0;
            x1[u] = *reinterpret_cast<const uint4*>(p.q_blk + src);
            x2[u] = *reinterpret_cast<const uint4*>(p.q_blk + src + D / 2);
          } else {                               // past the chunk: a zero query row
            x1[u] = x2[u] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      // (cos, sin) of the sub-block's positions L + i, i < sub_rows, for every
      // frequency
      for (int k = tid; k < sub_rows * (D / 2); k += 256) {
        const int i = k / (D / 2), d = k - i * (D / 2);
        float sn, cs;
        rope_sincos(Lq + i, rope_hi[d], rope_lo[d], &sn, &cs);
        sct[k] = make_float2(cs, sn);
      }
      named_bar_sync(1, 256);
#pragma unroll
      for (int u = 0; u < kMaxItems; ++u) {
        const int it = u * 256 + tid;
        if (it < q_items) {
          const int rr = it / kPer, d0 = (it - rr * kPer) * 8;
          uint4 y1, y2;
          rope8(x1[u], x2[u], sct + (rr & (sub_rows - 1)) * (D / 2), d0, y1, y2);
          const int e2 = d0 + D / 2;
          const int m = 32 * (rr / rq) + rr % rq;
          *reinterpret_cast<uint4*>(qs + (d0 >> 6) * kQHalf + swz_off(m, (d0 & 63) >> 3)) = y1;
          *reinterpret_cast<uint4*>(qs + (e2 >> 6) * kQHalf + swz_off(m, (e2 & 63) >> 3)) = y2;
          if (dup) {
            *reinterpret_cast<uint4*>(qs + (d0 >> 6) * kQHalf + swz_off(m + 16, (d0 & 63) >> 3)) = y1;
            *reinterpret_cast<uint4*>(qs + (e2 >> 6) * kQHalf + swz_off(m + 16, (e2 & 63) >> 3)) = y2;
          }
        }
      }
      if (has_block) {
        for (int it = tid; it < kPage * kPer; it += 256) {
          const int j = it / kPer, d0 = (it - j * kPer) * 8;
          // rows past the chunk are zero keys that the causal mask hides from
          // every row of the chunk
          const bool in = j < n_rows;
          const size_t src = (static_cast<size_t>(row0 + (in ? j : 0)) * p.n_kv_heads + g) * D + d0;
          const uint4 zero = make_uint4(0, 0, 0, 0);
          const uint4 k1 = in ? *reinterpret_cast<const uint4*>(p.k_blk + src) : zero;
          const uint4 k2 = in ? *reinterpret_cast<const uint4*>(p.k_blk + src + D / 2) : zero;
          const uint4 v1 = in ? *reinterpret_cast<const uint4*>(p.v_blk + src) : zero;
          const uint4 v2 = in ? *reinterpret_cast<const uint4*>(p.v_blk + src + D / 2) : zero;
          uint4 y1, y2;
          rope8(k1, k2, sct + j * (D / 2), d0, y1, y2);
          const int e2 = d0 + D / 2;
          const int off1 = (d0 >> 6) * C::kHalf + swz_off(j, (d0 & 63) >> 3);
          const int off2 = (e2 >> 6) * C::kHalf + swz_off(j, (e2 & 63) >> 3);
          *reinterpret_cast<uint4*>(blk + off1) = y1;
          *reinterpret_cast<uint4*>(blk + off2) = y2;
          *reinterpret_cast<uint4*>(blk + C::kBlkV + off1) = v1;
          *reinterpret_cast<uint4*>(blk + C::kBlkV + off2) = v2;
          if (p.k_app && L + kBlock <= limit) {
            // head-major cache row L + j of KV head g
            long long row = -1;
            if (p.paged) {
              const int id = p.page_table[static_cast<size_t>(b) * p.max_pages + (L + j) / kPage];
              if (id >= 0)
                row = (static_cast<long long>(id) * p.n_kv_heads + g) * kPage + (L + j) % kPage;
              else
                set_status(p.status, DFLASH_ST_PAGE_MISSING);
            } else {
              row = (static_cast<long long>(b) * p.n_kv_heads + g) * p.capacity + L + j;
            }
            if (row >= 0) {
              *reinterpret_cast<uint4*>(p.k_app + row * D + d0) = y1;
              *reinterpret_cast<uint4*>(p.k_app + row * D + e2) = y2;
              *reinterpret_cast<uint4*>(p.v_app + row * D + d0) = v1;
              *reinterpret_cast<uint4*>(p.v_app + row * D + e2) = v2;
            }
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    }

    // ---- softmax: all eight warps work on every chunk ----
    // Warp w reads TMEM quadrant q4 = w & 3 (rows 32 q4 ..) and the key half
    // kh = (w - 2) >> 2 of the 64-key chunk (S columns 32 kh ..); with rows
    // doubled (R <= 64) lanes l and l + 16 hold the same row and split the
    // half again.  A row's keys are spread over 4 threads (16 each), else 2
    // (32 each); the row max is combined within the warp (shuffle) and with
    // the quadrant's other warp through shared memory (one named barrier per
    // chunk and quadrant, which also carries the two warps' ok flags so that
    // they stop together).  S(j + 1) runs on the tensor cores while this
    // softmax works on chunk j.
    const int q4 = warp & 3;                    // TMEM lane quadrant of this warp
    const int kh = (warp - 2) >> 2;             // key half of the chunk
    const int i_row = dup ? (lane & 15) : lane;
    const int khalf = dup ? (lane >> 4) : 0;
    const bool real = i_row < rq;
    const int rr = q4 * rq + i_row;             // row in the partial outputs
    const int m = q4 * 32 + i_row;              // MMA row that carries P of this query row
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16);
    const uint32_t o_col = 128;                 // the O accumulator
    constexpr int kMine = dup ? 16 : 32;        // keys of a chunk per thread
    const int kbase = 32 * kh + kMine * khalf;  // this thread's first key of a chunk
    // exchange slots: [chunk parity][key half][128 lanes] maxima, ok flags
    float* xmax = reinterpret_cast<float*>(smem + p.off_xch);
    int* xok = reinterpret_cast<int*>(smem + p.off_xch + 2 * 2 * 128 * 4);  // [parity][kh][4 q]
    const uint32_t bar_q = 3 + q4;              // the quadrant's two warps
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true, okp_prev = true;
    for (int j = 0; j < n_total; ++j) {
      const int nk = chunk_keys(j);
      // a wait of the previous chunk that gave up stops the pair here, together
      bool okw = okp_prev && mbar_wait(&s_full[j & 1], static_cast<uint32_t>((j >> 1) & 1),
                                       abort_flag, p.status);
      okw = __all_sync(0xffffffffu, okw);
      float x[kMine];
      float mx = -INFINITY;
      // keys of this row: all valid ones, or -- causal block chunk -- block
      // rows 0 .. i of the row's own block position i
      // (the prompt attention: keys up to the row's own position L + i)
      const int n_see =
          p.self_cached ? max(0, min(nk, L + (rr & (sub_rows - 1)) + 1 - (key_begin + j * kChunk)))
          : (p.causal && has_block && j == 0) ? min(nk, (rr & 15) + 1)
                                              : nk;
      if (okw) {
        tc_fence_after();
        uint32_t sv[2][16];
#pragma unroll
        for (int c16 = 0; c16 < 2; ++c16)
          if (32 * kh + c16 * 16 < nk)
            tmem_ld_32x32b_x16(lane_addr + (j & 1) * 64 + 32 * kh + c16 * 16, sv[c16]);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < kMine; ++e) {
          // column within the warp's 32: e, or 16 khalf + e with rows doubled
          const uint32_t v = dup ? (khalf ? sv[1][e & 15] : sv[0][e & 15]) : sv[e >> 4][e & 15];
          x[e] = kbase + e < n_see ? __uint_as_float(v) : -INFINITY;
          mx = fmaxf(mx, x[e]);
        }
        if (dup) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      }
      xmax[((j & 1) * 2 + kh) * 128 + q4 * 32 + lane] = mx;
      if (lane == 0) xok[((j & 1) * 2 + kh) * 4 + q4] = okw ? 1 : 0;
      named_bar_sync(bar_q, 64);
      const bool ok_pair = okw && xok[((j & 1) * 2 + (kh ^ 1)) * 4 + q4] != 0;
      if (!ok_pair) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, xmax[((j & 1) * 2 + (kh ^ 1)) * 128 + q4 * 32 + lane]);
      const float mx_s = mx * p.scale_log2;
      float alpha = 1.f;
      if (m_run == -INFINITY) {
        m_run = mx_s;                         // first chunk: O and l empty
      } else if (mx_s > m_run + kRescaleLog2) {
        alpha = fast_exp2(m_run - mx_s);
        m_run = mx_s;
      }
      // P of this thread's keys, packed bf16 pairs (0 where masked; a row
      // that has seen no key yet -- the prompt attention's later splits --
      // keeps m = -inf and gets P = 0)
      const float m_sub = m_run == -INFINITY ? 0.f : m_run;
      uint32_t pk[kMine / 2];
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < kMine; e += 2) {
        const float p0 = fast_exp2(fmaf(x[e], p.scale_log2, -m_sub));
        const float p1 = fast_exp2(fmaf(x[e + 1], p.scale_log2, -m_sub));
        sum4[(e >> 1) & 3] += p0 + p1;
        pk[e >> 1] = pack_bf16(p0, p1);
      }
      l_run = l_run * alpha + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
      // P buffer j & 1 is free once P(j - 2) V(j - 2) has completed
      bool okp = true;
      if (j >= 2)
        okp = mbar_wait(&pv_done[j & 1], static_cast<uint32_t>(((j - 2) >> 1) & 1), abort_flag,
                        p.status);
      // a rescale of O needs P(j - 1) V(j - 1) completed (warps of key half 0
      // rescale their lanes; P(j) V(j) waits for every thread's arrival)
      if (kh == 0 && __any_sync(0xffffffffu, real && alpha != 1.f)) {
        if (j >= 1)
          okp = okp && mbar_wait(&pv_done[(j - 1) & 1], static_cast<uint32_t>(((j - 1) >> 1) & 1),
                                 abort_flag, p.status);
        if (__all_sync(0xffffffffu, okp)) {
          tc_fence_after();
#pragma unroll 1
          for (int c16 = 0; c16 < D / 16; ++c16) {
            uint32_t ov[16];
            tmem_ld_32x32b_x16(lane_addr + o_col + c16 * 16, ov);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st_32x32b_x16(lane_addr + o_col + c16 * 16, ov);
          }
          tmem_st_wait();
        }
      }
      if (q4 == 0 && kh == 0 && (nk & 15) && !(has_block && j == 0)) {
        // rows past the length inside the last 16-key group came with their
        // page: zero their V so that 0-probability keys cannot inject
        // NaN/Inf from stale memory into O
        uint8_t* vst = stg + ((j - has_block) % NS) * C::kStage + C::kTile;
        const int n_fill = (nk + 15) & ~15;
        for (int i = lane; i < (n_fill - nk) * C::kHalves * 8; i += 32) {
          const int r = nk + i / (C::kHalves * 8);
          const int ch = i % (C::kHalves * 8);
          *reinterpret_cast<uint4*>(vst + (ch >> 3) * C::kHalf + swz_off(r, ch & 7)) =
              make_uint4(0, 0, 0, 0);
        }
      }
      // P(j) into shared buffer j & 1: row m, this thread's keys
      uint8_t* prow = smem + (j & 1) * kPBytes;
      const int ncol = (nk + 15) & ~15;         // keys the P V MMA reads (p = 0 past nk)
#pragma unroll
      for (int c8 = 0; c8 < kMine / 8; ++c8) {  // 8 keys = one 16-byte chunk of the P row
        const int key0 = kbase + 8 * c8;
        if (real && key0 < ncol)
          *reinterpret_cast<uint4*>(prow + swz_off(m, key0 >> 3)) =
              make_uint4(pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[j & 1]);
      // an abandoned wait ends the loop at the next chunk's exchange, where
      // the quadrant's other warp learns of it too (the MMA thread stops at
      // its own bounded wait)
      okp_prev = __all_sync(0xffffffffu, okp);
      if (!okp_prev && j == n_total - 1) ok = false;
    }
    // the row's sum over its 4 (2) threads: shuffle, then the other warp
    if (dup) l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
    float* lx = xmax;                           // the exchange slots are free now
    named_bar_sync(2, 256);
    if (kh == 1) lx[q4 * 32 + lane] = ok ? l_run : 0.f;
    if (kh == 1 && lane == 0) xok[q4] = ok ? 1 : 0;
    named_bar_sync(2, 256);
    if (kh == 0) {
      const bool writer = real && khalf == 0;
      // partials of grid unit (z, KV head, split): z = (sequence, sub-block)
      const size_t unit = (static_cast<size_t>(blockIdx.z) * p.n_kv_heads + g) * p.splits + s_idx;
      float* po = p.part_o + (unit * R + rr) * D;
      float* pml = p.part_ml + (unit * R + rr) * 2;
      bool have_o = ok && xok[q4] != 0 && n_total > 0;
      have_o = __all_sync(0xffffffffu, have_o);
      if (have_o) {
        const bool done = mbar_wait(o_done, 0, abort_flag, p.status);
        have_o = __all_sync(0xffffffffu, done);
      }
      float M = m_run, l_tot = l_run + lx[q4 * 32 + lane];
      // single split: the normalised bf16 row goes straight to the output
      // (row i of query head g * G + w), rows past the chunk are dropped
      const int wq = rr >> p.sub_shift, iq = rr & (sub_rows - 1);
      uint16_t* od = p.out_direct
                         ? p.out_direct +
                               (static_cast<size_t>(row0 + iq) * p.n_q_heads + g * G + wq) * D
                         : nullptr;
      const bool direct_row = od != nullptr && iq < n_rows && valid_len;
      const float inv_l = 1.f / l_tot;
      if (have_o) {
        tc_fence_after();
#pragma unroll 1
        for (int c16 = 0; c16 < D / 16; c16 += 2) {
          uint32_t oa[16], ob[16];
          tmem_ld_32x32b_x16(lane_addr + o_col + c16 * 16, oa);
          tmem_ld_32x32b_x16(lane_addr + o_col + c16 * 16 + 16, ob);
          tmem_ld_wait();
          if (writer) {
            if (od) {
              if (direct_row) {
                uint32_t pa[8], pb[8];
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                  pa[e >> 1] = pack_bf16(__uint_as_float(oa[e]) * inv_l,
                                         __uint_as_float(oa[e + 1]) * inv_l);
                  pb[e >> 1] = pack_bf16(__uint_as_float(ob[e]) * inv_l,
                                         __uint_as_float(ob[e + 1]) * inv_l);
                }
                uint4* d4 = reinterpret_cast<uint4*>(od + c16 * 16);
                d4[0] = make_uint4(pa[0], pa[1], pa[2], pa[3]);
                d4[1] = make_uint4(pa[4], pa[5], pa[6], pa[7]);
                d4[2] = make_uint4(pb[0], pb[1], pb[2], pb[3]);
                d4[3] = make_uint4(pb[4], pb[5], pb[6], pb[7]);
              }
            } else {
              float4* d4 = reinterpret_cast<float4*>(po + c16 * 16);
#pragma unroll
              for (int e = 0; e < 16; e += 4) {
                d4[e >> 2] = make_float4(__uint_as_float(oa[e]), __uint_as_float(oa[e + 1]),
                                         __uint_as_float(oa[e + 2]), __uint_as_float(oa[e + 3]));
                d4[4 + (e >> 2)] =
                    make_float4(__uint_as_float(ob[e]), __uint_as_float(ob[e + 1]),
                                __uint_as_float(ob[e + 2]), __uint_as_float(ob[e + 3]));
              }
            }
          }
        }
      } else if (writer && !od) {
        for (int e = 0; e < D; e += 4) *reinterpret_cast<float4*>(po + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        M = -INFINITY;
        l_tot = 0.f;
      }
      if (writer && !od) *reinterpret_cast<float2*>(pml) = make_float2(M, l_tot);
    }
  }
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols<D>());
  }
}

// Merge the split partials by log-sum-exp.  One warp per output row (b, i, h),
// four rows per CTA.  A lane holds the (max, sum) pairs of splits lane and
// lane + 32 and D/32 output elements; the partial rows are read in batches of
// kBatch splits whose loads are all in flight together, and the first batch
// is requested before the maxima are known, so a row costs about one global
// round trip per batch.
constexpr int kCombineRows = 4;

template <int D>
__global__ void __launch_bounds__(32 * kCombineRows) attn_combine_kernel(const CombineParams p) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int per = D / 32;  // 2 or 4 elements per lane
  constexpr int kBatch = 32;
  using Vec = typename std::conditional<per == 4, float4, float2>::type;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kCombineRows + warp;
  const int rows_out = p.batch * p.tokens * p.n_q_heads;
  if (row >= rows_out) return;
  // output row (b, t, h): block row i = t % 16 of sub-block j = t / 16, whose
  // grid index z runs the sub-blocks of a sequence last to first
  const int b = row / (p.tokens * p.n_q_heads);
  const int rem = row - b * p.tokens * p.n_q_heads;
  const int t = rem / p.n_q_heads;
  const int h = rem - t * p.n_q_heads;
  const int i = t & ((1 << p.sub_shift) - 1);
  const int z = b * p.sub_blocks + (p.sub_blocks - 1 - (t >> p.sub_shift));
  const int g = h / p.group, w = h - g * p.group;
  const int rr = (w << p.sub_shift) + i;
  const size_t unit0 = (static_cast<size_t>(z) * p.n_kv_heads + g) * p.splits;
  const int L0 = p.seq_len[b];
  float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
  if (lane < p.splits) {
    const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + ((unit0 + lane) * p.rows + rr) * 2);
    m0 = ml.x;
    l0 = ml.y;
  }
  if (lane + 32 < p.splits) {
    const float2 ml =
        *reinterpret_cast<const float2*>(p.part_ml + ((unit0 + lane + 32) * p.rows + rr) * 2);
    m1 = ml.x;
    l1 = ml.y;
  }
  const float* base = p.part_o + (unit0 * p.rows + rr) * D + lane * per;
  const size_t stride = static_cast<size_t>(p.rows) * D;
  Vec v[kBatch];
#pragma unroll
  for (int k = 0; k < kBatch; ++k)
    if (k < p.splits) v[k] = *reinterpret_cast<const Vec*>(base + k * stride);
  if (L0 < 0 || L0 + p.need_rows > p.limit) return;
  float M = fmaxf(m0, m1);
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  const float w0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M);
  const float w1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M);
  float lsum = w0 * l0 + w1 * l1;
#pragma unroll
  for (int off = 16; off; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
  float acc[per];
#pragma unroll
  for (int e = 0; e < per; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < p.splits; s0 += kBatch) {
    if (s0 > 0) {
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        if (s0 + k < p.splits) v[k] = *reinterpret_cast<const Vec*>(base + (s0 + k) * stride);
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int sp = s0 + k;
      const float wk = __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31);
      if (sp < p.splits) {
        const float* f = reinterpret_cast<const float*>(&v[k]);
#pragma unroll
        for (int e = 0; e < per; ++e) acc[e] = fmaf(wk, f[e], acc[e]);
      }
    }
  }
  const float inv = 1.f / lsum;
  uint16_t* dst = p.out + static_cast<size_t>(row) * D + lane * per;
  if constexpr (per == 4) {
    uint2 o;
    o.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    o.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = o;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16(acc[0] * inv, acc[1] * inv);
  }
}

// Shared-memory plan of the attention kernel: two P buffers (128 rows x 64
// keys each), Q ([half][128 rows][128 B]), the K/V stages, the block tile,
// the sin/cos table, the odd group's (max, sum), the rotary table and the
// barriers.  One CTA per SM, with as many stages (up to 6) as fit.
constexpr int kSmemPerCta = 232448;  // opt-in maximum of one CTA

template <int D>
int attention_smem_for(AttnParams& p, int n_stages) {
  using C = Cfg<D>;
  p.n_stages = n_stages;
  p.off_q = 2 * 128 * 128;                              // after the two P buffers
  p.off_st = p.off_q + C::kHalves * 128 * 128;
  p.off_blk = p.off_st + n_stages * C::kStage;
  p.off_sc = p.off_blk + C::kBlkTile;                   // [16][D/2] float2
  p.off_xch = p.off_sc + (1 << p.sub_shift) * (D / 2) * 8;  // [2][2][128] float + [2][2][4] int
  p.off_rope = p.off_xch + 2 * 2 * 128 * 4 + 2 * 2 * 4 * 4;
  p.off_bar = p.off_rope + D * 4;
  return 1024 + p.off_bar + (2 * n_stages + 9) * 8 + 8;
}

template <int D>
int plan_attention_smem(AttnParams& p) {
  for (int ns = 6; ns >= 2; --ns) {
    const int smem = attention_smem_for<D>(p, ns);
    if (smem <= kSmemPerCta) return smem;
  }
  return attention_smem_for<D>(p, 2);
}

// The target's attention appends n rows at L .. L + n - 1 (16 for the verify
// forward, a prompt chunk for the prefill): map the pages those rows need
// before anything writes them, and move the length past them once every
// kernel that reads L has finished.
__global__ void append_reserve_kernel(const dflash_kv_view v, int batch, int n,
                                      uint32_t* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int L = v.seq_len[b];
  const int limit = v.max_pages * v.page_size;
  if (L >= 0 && L + n <= limit) map_rows(v, b, L, n, status);
}

__global__ void append_length_kernel(int32_t* seq_len, int batch, int n, int limit,
                                     uint32_t* status) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int L = seq_len[b];
  if (L >= 0 && L + n <= limit)
    seq_len[b] = L + n;
  else
    set_status(status, DFLASH_ST_CAPACITY);
}

// Prefill: the chunk's K rotated at L + t and its V, for every row t < T and
// KV head, written into the cache rows L + t before the attention reads them
// (the rotation is the one the attention applies to a block's keys).  One
// thread per (row, KV head, 8-dim item of the first half of the head).
template <int D>
__global__ void __launch_bounds__(256) prefill_append_kernel(const dflash_kv_view v,
                                                             const uint16_t* __restrict__ k,
                                                             const uint16_t* __restrict__ vv,
                                                             int batch, int tokens, int n_kv_heads,
                                                             const RopeTable rope,
                                                             uint32_t* status) {
  griddep_wait();
  constexpr int kItems = D / 16;                     // items of 8 dims per half head
  const long long it = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(batch) * tokens * n_kv_heads * kItems;
  if (it < total) {
    const int item = static_cast<int>(it % kItems);
    const long long rg = it / kItems;                // (b * T + t) * Hkv + g
    const int g = static_cast<int>(rg % n_kv_heads);
    const long long bt = rg / n_kv_heads;
    const int b = static_cast<int>(bt / tokens), t = static_cast<int>(bt % tokens);
    const int L = v.seq_len[b];
    const int limit = v.page_table ? v.max_pages * v.page_size : v.capacity;
    if (L >= 0 && L + tokens <= limit) {
      const int pos = L + t;
      long long row = -1;
      if (v.page_table) {
        const int id = v.page_table[static_cast<size_t>(b) * v.max_pages + pos / kPage];
        if (id >= 0)
          row = (static_cast<long long>(id) * n_kv_heads + g) * kPage + pos % kPage;
        else
          set_status(status, DFLASH_ST_PAGE_MISSING);
      } else {
        row = (static_cast<long long>(b) * n_kv_heads + g) * v.capacity + pos;
      }
      if (row >= 0) {
        const int d0 = item * 8, e2 = d0 + D / 2;
        const size_t src = static_cast<size_t>(rg) * D;
        float2 sc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float sn, cs;
          rope_sincos(pos, rope.hi[d0 + e], rope.lo[d0 + e], &sn, &cs);
          sc[e] = make_float2(cs, sn);
        }
        uint4 y1, y2;
        rope8(*reinterpret_cast<const uint4*>(k + src + d0),
              *reinterpret_cast<const uint4*>(k + src + e2), sc, 0, y1, y2);
        uint16_t* kd = static_cast<uint16_t*>(v.k) + row * D;
        uint16_t* vd = static_cast<uint16_t*>(v.v) + row * D;
        *reinterpret_cast<uint4*>(kd + d0) = y1;
        *reinterpret_cast<uint4*>(kd + e2) = y2;
        *reinterpret_cast<uint4*>(vd + d0) = *reinterpret_cast<const uint4*>(vv + src + d0);
        *reinterpret_cast<uint4*>(vd + e2) = *reinterpret_cast<const uint4*>(vv + src + e2);
      }
    }
  }
  griddep_launch_dependents();
}

template <int D>
int launch_attention(const dflash_dims& dims, int splits, const dflash_kv_view& cache,
                     AttnParams& p, CombineParams& cp, cudaStream_t stream) {
  using C = Cfg<D>;
  // head-major caches: contiguous [B, Hkv, cap, D] is a stack of (sequence,
  // head) slabs of cap rows; paged [pages, Hkv, 16, D] a stack of 16-row slabs
  CUtensorMap tm_k, tm_v, tm_k64, tm_v64;
  const uint64_t pitch_row = static_cast<uint64_t>(D) * 2;
  int rc;
  if (p.paged) {
    const uint64_t slabs = static_cast<uint64_t>(cache.n_pages) * dims.n_kv_heads;
    if ((rc = make_tmap_3d_bf16(&tm_k, cache.k, D, kPage, slabs, pitch_row, pitch_row * kPage, 64,
                                kPage, 1)))
      return rc;
    if ((rc = make_tmap_3d_bf16(&tm_v, cache.v, D, kPage, slabs, pitch_row, pitch_row * kPage, 64,
                                kPage, 1)))
      return rc;
    tm_k64 = tm_k;
    tm_v64 = tm_v;
  } else {
    const uint64_t slabs = static_cast<uint64_t>(dims.batch) * dims.n_kv_heads;
    const uint64_t cap = static_cast<uint64_t>(cache.capacity);
    if ((rc = make_tmap_3d_bf16(&tm_k, cache.k, D, cap, slabs, pitch_row, pitch_row * cap, 64,
                                kPage, 1)))
      return rc;
    if ((rc = make_tmap_3d_bf16(&tm_v, cache.v, D, cap, slabs, pitch_row, pitch_row * cap, 64,
                                kPage, 1)))
      return rc;
    if ((rc = make_tmap_3d_bf16(&tm_k64, cache.k, D, cap, slabs, pitch_row, pitch_row * cap, 64,
                                kChunk, 1)))
      return rc;
    if ((rc = make_tmap_3d_bf16(&tm_v64, cache.v, D, cap, slabs, pitch_row, pitch_row * cap, 64,
                                kChunk, 1)))
      return rc;
  }
  const int smem = plan_attention_smem<D>(p);
  // query rows are doubled across the TMEM lanes when they fill at most half
  auto kernel = p.rows <= 64 ? block_attention_kernel<D, true> : block_attention_kernel<D, false>;
  if ((rc = set_smem_limit(reinterpret_cast<const void*>(kernel), smem))) return rc;
  rc = launch(kernel, dim3(splits, dims.n_kv_heads, dims.batch * p.sub_blocks),
              dim3(kAttThreads), smem, stream, tm_k, tm_v, tm_k64, tm_v64, p);
  if (rc) return rc;
  if (!p.out_direct) {
    const long long rows_out = static_cast<long long>(dims.batch) * p.tokens * dims.n_q_heads;
    rc = launch(attn_combine_kernel<D>,
                dim3(static_cast<unsigned>((rows_out + kCombineRows - 1) / kCombineRows)),
                dim3(32 * kCombineRows), 0, stream, cp);
    if (rc) return rc;
  }
  if (!p.k_app && p.need_rows == 0) return DFLASH_OK;
  // the verify forward's block, or the prefill chunk, is now part of the cache
  return launch(append_length_kernel, dim3((dims.batch + 127) / 128), dim3(128), 0, stream,
                cache.seq_len, dims.batch, p.k_app ? kBlock : p.tokens, cp.limit, p.status);
}

}  // namespace
}  // namespace dflash

using namespace dflash;

namespace {

int run_attention(const dflash_dims* dims, const void* q_blk, const void* k_blk,
                  const void* v_blk, const dflash_kv_view* cache, float scale, void* out,
                  void* ws, size_t ws_bytes, dflash_stream_t stream, bool verify) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!q_blk || !k_blk || !v_blk || !cache || !out || !cache->k || !cache->v || !cache->seq_len)
    return DFLASH_E_ARG;
  if (!aligned16(q_blk) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(out) ||
      !aligned16(cache->k) || !aligned16(cache->v))
    return DFLASH_E_ALIGN;
  if (!(scale > 0.0f)) return DFLASH_E_ARG;
  const bool paged = cache->page_table != nullptr;
  if (paged) {
    if (cache->page_size != 16) return DFLASH_E_UNSUPPORTED;
    if (cache->max_pages < 1 || cache->n_pages < 1) return DFLASH_E_ARG;
  } else if (cache->capacity < 1) {
    return DFLASH_E_ARG;
  }
  if (!ws) return DFLASH_E_WORKSPACE;
  Plan plan;
  if ((rc = make_plan(*dims, &plan))) return rc;
  if (ws_bytes < plan.total) return DFLASH_E_WORKSPACE;

  AttnParams p = {};
  p.tokens = kBlock;
  p.sub_blocks = 1;
  p.sub_shift = 4;
  p.need_rows = 0;
  p.batch = dims->batch;
  p.n_q_heads = dims->n_q_heads;
  p.n_kv_heads = dims->n_kv_heads;
  p.group = dims->n_q_heads / dims->n_kv_heads;
  p.splits = plan.att_splits;
  p.rows = plan.att_rows;
  p.paged = paged ? 1 : 0;
  p.capacity = cache->capacity;
  p.max_pages = cache->max_pages;
  p.seq_len = cache->seq_len;
  p.page_table = cache->page_table;
  p.q_blk = static_cast<const uint16_t*>(q_blk);
  p.k_blk = static_cast<const uint16_t*>(k_blk);
  p.v_blk = static_cast<const uint16_t*>(v_blk);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.part_o = ws_at<float>(ws, plan.off_att_o);
  p.part_ml = ws_at<float>(ws, plan.off_att_ml);
  p.status = ws_at<uint32_t>(ws, plan.off_status);
  fill_rope_table(p.rope.hi, p.rope.lo, dims->head_dim, dims->rope_theta);

  CombineParams cp = {};
  cp.tokens = kBlock;
  cp.sub_blocks = 1;
  cp.sub_shift = 4;
  cp.need_rows = 0;
  cp.batch = dims->batch;
  cp.n_q_heads = dims->n_q_heads;
  cp.n_kv_heads = dims->n_kv_heads;
  cp.group = p.group;
  cp.splits = p.splits;
  cp.rows = p.rows;
  cp.head_dim = dims->head_dim;
  cp.limit = paged ? cache->max_pages * 16 : cache->capacity;
  cp.seq_len = cache->seq_len;
  cp.part_o = p.part_o;
  cp.part_ml = p.part_ml;
  cp.out = static_cast<uint16_t*>(out);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (verify) {
    p.causal = 1;
    p.k_app = static_cast<uint16_t*>(cache->k);
    p.v_app = static_cast<uint16_t*>(cache->v);
    if (paged && (!cache->free_list || !cache->free_count)) return DFLASH_E_ARG;
    if (paged && (rc = launch(append_reserve_kernel, dim3((dims->batch + 127) / 128), dim3(128),
                              0, s, *cache, dims->batch, kBlock, p.status)))
      return rc;
  }
  return dims->head_dim == 128 ? launch_attention<128>(*dims, plan.att_splits, *cache, p, cp, s)
                               : launch_attention<64>(*dims, plan.att_splits, *cache, p, cp, s);
}

}  // namespace

namespace dflash {

// Workspace of dflash_prefill_attention: the status word, then the split
// partials when a chunk's (sequence, sub-block, KV head) units are too few to
// fill the device with one split each.
struct PrefillAttnPlan {
  int sub_shift, sub_blocks, splits, rows;
  size_t off_status, off_o, off_ml, total;
};

int make_prefill_attn_plan(const dflash_dims& d, int tokens, PrefillAttnPlan* out) {
  int rc = check_dims(&d);
  if (rc) return rc;
  if (tokens < 1) return DFLASH_E_ARG;
  PrefillAttnPlan q = {};
  // 32 prompt rows per CTA when the G query heads of a KV head then fill the
  // 128 MMA rows (G <= 4), else 16: every CTA streams its KV head's prefix
  // once, so more rows per CTA means fewer passes over the prefix
  const int G = d.n_q_heads / d.n_kv_heads;
  q.sub_shift = G * 32 <= 128 ? 5 : 4;
  q.sub_blocks = (tokens + (1 << q.sub_shift) - 1) >> q.sub_shift;
  if (static_cast<long long>(d.batch) * q.sub_blocks > 65535) return DFLASH_E_UNSUPPORTED;
  // splits: enough (sequence, sub-block, KV head, split) CTAs for one per
  // SM of the GB300 (152); fixed rather than read from the device, so that
  // the workspace size is a function of the shapes alone
  constexpr int kFillCtas = 152;
  const long long units = static_cast<long long>(d.batch) * q.sub_blocks * d.n_kv_heads;
  int s = units >= kFillCtas ? 1 : static_cast<int>((kFillCtas + units - 1) / units);
  const int pages = (d.max_ctx + kPage - 1) / kPage;
  if (s > pages) s = pages;
  if (s > kMaxAttSplits) s = kMaxAttSplits;
  if (s < 1) s = 1;
  q.splits = s;
  q.rows = G << q.sub_shift;
  size_t off = 256;  // status word at 0
  q.off_status = 0;
  if (s > 1) {
    const size_t n = static_cast<size_t>(units) * s * q.rows;
    q.off_o = off;
    off += sizeof(float) * n * d.head_dim;
    q.off_ml = off;
    off += sizeof(float) * 2 * n;
  }
  q.total = (off + 255) & ~static_cast<size_t>(255);
  *out = q;
  return DFLASH_OK;
}

size_t prefill_attention_workspace(const dflash_dims& d, int tokens_per_seq) {
  PrefillAttnPlan p;
  return make_prefill_attn_plan(d, tokens_per_seq, &p) ? 0 : p.total;
}

}  // namespace dflash

extern "C" int dflash_prefill_attention(const dflash_dims* dims, int32_t tokens_per_seq,
                                        const void* q, const void* k, const void* v,
                                        const dflash_kv_view* cache, float scale, void* out,
                                        void* ws, size_t ws_bytes, dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_prefill_attention");
  int rc = check_dims(dims);
  if (rc) return rc;
  PrefillAttnPlan plan;
  if ((rc = make_prefill_attn_plan(*dims, tokens_per_seq, &plan))) return rc;
  if (!q || !k || !v || !cache || !out || !cache->k || !cache->v || !cache->seq_len)
    return DFLASH_E_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(cache->k) || !aligned16(cache->v))
    return DFLASH_E_ALIGN;
  if (!(scale > 0.0f)) return DFLASH_E_ARG;
  const bool paged = cache->page_table != nullptr;
  if (paged) {
    if (cache->page_size != 16) return DFLASH_E_UNSUPPORTED;
    if (cache->max_pages < 1 || cache->n_pages < 1 || !cache->free_list || !cache->free_count)
      return DFLASH_E_ARG;
  } else if (cache->capacity < 1) {
    return DFLASH_E_ARG;
  }
  if (!ws) return DFLASH_E_WORKSPACE;
  if (ws_bytes < plan.total) return DFLASH_E_WORKSPACE;
  const int T = tokens_per_seq;

  AttnParams p = {};
  p.batch = dims->batch;
  p.n_q_heads = dims->n_q_heads;
  p.n_kv_heads = dims->n_kv_heads;
  p.group = dims->n_q_heads / dims->n_kv_heads;
  p.splits = plan.splits;
  p.rows = plan.rows;
  p.paged = paged ? 1 : 0;
  p.capacity = cache->capacity;
  p.max_pages = cache->max_pages;
  p.seq_len = cache->seq_len;
  p.page_table = cache->page_table;
  p.q_blk = static_cast<const uint16_t*>(q);
  p.k_blk = static_cast<const uint16_t*>(k);
  p.v_blk = static_cast<const uint16_t*>(v);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = ws_at<uint32_t>(ws, plan.off_status);
  p.causal = 1;
  p.tokens = T;
  p.sub_blocks = plan.sub_blocks;
  p.sub_shift = plan.sub_shift;
  p.self_cached = 1;
  p.need_rows = T;
  if (plan.splits > 1) {
    p.part_o = ws_at<float>(ws, plan.off_o);
    p.part_ml = ws_at<float>(ws, plan.off_ml);
  } else {
    p.out_direct = static_cast<uint16_t*>(out);
  }
  fill_rope_table(p.rope.hi, p.rope.lo, dims->head_dim, dims->rope_theta);

  CombineParams cp = {};
  cp.batch = dims->batch;
  cp.n_q_heads = dims->n_q_heads;
  cp.n_kv_heads = dims->n_kv_heads;
  cp.group = p.group;
  cp.splits = p.splits;
  cp.rows = p.rows;
  cp.head_dim = dims->head_dim;
  cp.limit = paged ? cache->max_pages * 16 : cache->capacity;
  cp.tokens = T;
  cp.sub_blocks = plan.sub_blocks;
  cp.sub_shift = plan.sub_shift;
  cp.need_rows = T;
  cp.seq_len = cache->seq_len;
  cp.part_o = p.part_o;
  cp.part_ml = p.part_ml;
  cp.out = static_cast<uint16_t*>(out);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // 1. pages for the chunk's rows; 2. the chunk's rotated K and V into the
  // cache; 3. causal attention of its sub-blocks; 4. the length
  if (paged && (rc = launch(append_reserve_kernel, dim3((dims->batch + 127) / 128), dim3(128), 0,
                            s, *cache, dims->batch, T, p.status)))
    return rc;
  const long long items =
      static_cast<long long>(dims->batch) * T * dims->n_kv_heads * (dims->head_dim / 16);
  const dim3 agrid(static_cast<unsigned>((items + 255) / 256));
  rc = dims->head_dim == 128
           ? launch(prefill_append_kernel<128>, agrid, dim3(256), 0, s, *cache, p.k_blk, p.v_blk,
                    dims->batch, T, dims->n_kv_heads, p.rope, p.status)
           : launch(prefill_append_kernel<64>, agrid, dim3(256), 0, s, *cache, p.k_blk, p.v_blk,
                    dims->batch, T, dims->n_kv_heads, p.rope, p.status);
  if (rc) return rc;
  return dims->head_dim == 128 ? launch_attention<128>(*dims, plan.splits, *cache, p, cp, s)
                               : launch_attention<64>(*dims, plan.splits, *cache, p, cp, s);
}

extern "C" int dflash_block_attention(const dflash_dims* dims, const void* q_blk,
                                      const void* k_blk, const void* v_blk,
                                      const dflash_kv_view* cache, float scale, void* out,
                                      void* ws, size_t ws_bytes, dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_block_attention");
  return run_attention(dims, q_blk, k_blk, v_blk, cache, scale, out, ws, ws_bytes, stream,
                       false);
}

extern "C" int dflash_verify_attention(const dflash_dims* dims, const void* q_blk,
                                       const void* k_blk, const void* v_blk,
                                       const dflash_kv_view* cache, float scale, void* out,
                                       void* ws, size_t ws_bytes, dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_verify_attention");
  return run_attention(dims, q_blk, k_blk, v_blk, cache, scale, out, ws, ws_bytes, stream,
                       true);
}
