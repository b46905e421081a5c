// a2 — dual-source block attention of the drafter.
//
// "DFlash双实现对比" (hotelren.com) §2: Q comes only from the 16 block tokens;
// K/V is the concatenation of the context K/V (projected from the target's
// hidden states) with the block's own K/V; there is no causal mask inside the
// block.  "dflash-mlx" (dpshk.com) 块扩散草稿: the staged token and 15 masks
// are denoised in one parallel forward that reads the target's hidden states.
//
// Design (GB300): decode-style attention is bound by the context KV read
// (64 flop per byte with GQA packing).  Grid = (split, KV head, sequence): each
// CTA owns one KV head of one sequence and a page-aligned slice of its
// context, so the G = Hq/Hkv query heads that share the KV head (G*16 query
// rows) read every KV byte once.  One producer warp streams 64-key chunks of
// K and V through a 3-stage TMA pipeline (one 16-row box per page and 64-wide
// half of the head dim, 128-byte swizzle; contiguous and paged caches differ
// only in the row coordinate of each box).  G consumer warps (one per query
// head, 16 rows each) run QK^T and PV on mma.sync bf16 tensor cores with an
// fp32 online softmax (quad shuffles for row max/sum).  RoPE of the block
// queries/keys is applied in registers at positions L + i.  The split that
// owns the tail also folds in the 16 block keys.  Partial (O, max, sum) go to
// the workspace and a second kernel merges the splits by log-sum-exp.
#include <type_traits>

#include "common.cuh"
#include "host.h"

namespace dflash {
namespace {

constexpr int kChunk = 64;   // keys per pipeline stage
constexpr int kPage = 16;    // rows per TMA box
#ifndef DFLASH_ATT_STAGES
#define DFLASH_ATT_STAGES 3
#endif
constexpr int kStages = DFLASH_ATT_STAGES;

struct AttnParams {
  int batch, n_q_heads, n_kv_heads, group, splits, rows;  // rows = group * 16
  int paged, capacity, max_pages;
  const int32_t* seq_len;
  const int32_t* page_table;
  const uint16_t* q_blk;
  const uint16_t* k_blk;
  const uint16_t* v_blk;
  float scale_log2;
  float* part_o;
  float* part_ml;
  uint32_t* status;
  RopeTable rope;
};

struct CombineParams {
  int batch, n_q_heads, n_kv_heads, group, splits, rows, head_dim, limit;
  const int32_t* seq_len;
  const float* part_o;
  const float* part_ml;
  uint16_t* out;
};

__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return static_cast<uint32_t>(float_to_bf16_bits(lo)) |
         (static_cast<uint32_t>(float_to_bf16_bits(hi)) << 16);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte address of (row, 16-byte chunk) in a tile stored as 64-column halves of
// kChunk rows x 128 B with the 128-byte swizzle.  The row stride of a half is
// a compile-time constant, so the addresses of a fully unrolled chunk fold to
// a per-lane base plus immediates.
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
  return base + static_cast<uint32_t>((chunk >> 3) * kChunk * 128 + row * 128 +
                                      (((chunk & 7) ^ (row & 7)) << 4));
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
  static constexpr int kTile = kHalves * kChunk * 128;   // K or V of one 64-key chunk
  static constexpr int kStage = 2 * kTile;
  // the 16 block rows of K and V share one tile with the same half stride as a
  // chunk: K in rows 0..15 of each half, V in rows 16..31
  static constexpr int kBlkTile = (kHalves - 1) * kChunk * 128 + 2 * kPage * 128;
  static constexpr int kBlkV = kPage * 128;              // V offset inside that tile
};

// One chunk of keys for one warp: S = Q K^T, online softmax, O += P V.  The
// running max m is kept in the scaled log2 domain, so each probability is one
// FFMA and one ex2.
template <int D>
__device__ __forceinline__ void attend_chunk(const uint32_t (&qf)[D / 16][4], uint32_t kbase,
                                             uint32_t vbase, int n_valid, float scale_log2,
                                             float (&o)[D / 8][4], float& m_a, float& m_b,
                                             float& l_a, float& l_b) {
  const int lane = threadIdx.x & 31;
  const int t = lane & 3;
  const int n16 = (n_valid + 15) >> 4;
  float s[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int np = 0; np < 4; ++np) {
      if (np < n16) {
        const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int chunk = 2 * kk + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(swz(kbase, key, chunk), b0, b1, b2, b3);
        mma_16816(s[2 * np], qf[kk], b0, b1);
        mma_16816(s[2 * np + 1], qf[kk], b2, b3);
      }
    }
  }
  if (n_valid < kChunk) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (nt * 8 + 2 * t + (e & 1) >= n_valid) s[nt][e] = -INFINITY;
    }
  }
  float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    mx_a = fmaxf(mx_a, fmaxf(s[nt][0], s[nt][1]));
    mx_b = fmaxf(mx_b, fmaxf(s[nt][2], s[nt][3]));
  }
  mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
  mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
  mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
  mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
  const float mn_a = fmaxf(m_a, mx_a * scale_log2), mn_b = fmaxf(m_b, mx_b * scale_log2);
  const float al_a = fast_exp2(m_a - mn_a), al_b = fast_exp2(m_b - mn_b);
  m_a = mn_a;
  m_b = mn_b;
  float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    s[nt][0] = fast_exp2(fmaf(s[nt][0], scale_log2, -mn_a));
    s[nt][1] = fast_exp2(fmaf(s[nt][1], scale_log2, -mn_a));
    s[nt][2] = fast_exp2(fmaf(s[nt][2], scale_log2, -mn_b));
    s[nt][3] = fast_exp2(fmaf(s[nt][3], scale_log2, -mn_b));
    sum_a += s[nt][0] + s[nt][1];
    sum_b += s[nt][2] + s[nt][3];
  }
  l_a = l_a * al_a + sum_a;
  l_b = l_b * al_b + sum_b;
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    o[dt][0] *= al_a;
    o[dt][1] *= al_a;
    o[dt][2] *= al_b;
    o[dt][3] *= al_b;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (j < n16) {
      uint32_t a[4];
      a[0] = pack_bf16(s[2 * j][0], s[2 * j][1]);
      a[1] = pack_bf16(s[2 * j][2], s[2 * j][3]);
      a[2] = pack_bf16(s[2 * j + 1][0], s[2 * j + 1][1]);
      a[3] = pack_bf16(s[2 * j + 1][2], s[2 * j + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int key = 16 * j + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int chunk = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(swz(vbase, key, chunk), b0, b1, b2, b3);
        mma_16816(o[2 * dp], a, b0, b1);
        mma_16816(o[2 * dp + 1], a, b2, b3);
      }
    }
  }
}

template <int D>
__global__ void __launch_bounds__(288) block_attention_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __grid_constant__ CUtensorMap tm_k64, const __grid_constant__ CUtensorMap tm_v64,
    const AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint8_t* blk = smem + kStages * C::kStage;  // block K (rows 0..15) and V (rows 16..31)
  float* rope_hi = reinterpret_cast<float*>(blk + C::kBlkTile);  // inv_freq as hi + lo
  float* rope_lo = rope_hi + D / 2;
  uint64_t* full = reinterpret_cast<uint64_t*>(rope_lo + D / 2);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int s_idx = blockIdx.x, g = blockIdx.y, b = blockIdx.z;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], G);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // the rotary table goes to shared memory once: lanes then read it by index
  // without serialising on the parameter bank
  for (int i = threadIdx.x; i < D / 2; i += blockDim.x) {
    rope_hi[i] = p.rope.hi[i];
    rope_lo[i] = p.rope.lo[i];
  }
  if (warp == G && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_k64);
    tma_prefetch_desc(&tm_v64);
  }
  __syncthreads();
  griddep_wait();

  const int L = p.seq_len[b];
  const int limit = p.paged ? p.max_pages * kPage : p.capacity;
  const bool valid_len = L >= 0 && L <= limit;
  if (!valid_len && threadIdx.x == 0 && s_idx == 0 && g == 0)
    set_status(p.status, DFLASH_ST_CAPACITY);
  const int Lc = valid_len ? L : 0;
  const int n_pg = (Lc + kPage - 1) / kPage;
  const int pps = (n_pg + p.splits - 1) / p.splits;
  const int pg_begin = s_idx * pps;
  const int pg_end = min(pg_begin + pps, n_pg);
  const int key_begin = pg_begin * kPage;
  const int key_end = min(pg_end * kPage, Lc);
  const int n_keys = key_end > key_begin ? key_end - key_begin : 0;
  const int n_chunks = (n_keys + kChunk - 1) / kChunk;
  const bool has_block = valid_len && (s_idx == p.splits - 1);

  if (warp == G) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      uint32_t stage = 0, phase = 0;
      for (int c = 0; c < n_chunks; ++c) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) break;
        uint8_t* kst = smem + stage * C::kStage;
        uint8_t* vst = kst + C::kTile;
        const int k0 = key_begin + c * kChunk;
        const int npg = min(kChunk / kPage, (key_end - k0 + kPage - 1) / kPage);
        // head-major caches: a page (16 rows) of one head is 16 * D contiguous
        // elements, a contiguous cache holds each head's rows back to back
        const int slab = b * p.n_kv_heads + g;  // contiguous: (sequence, head) slab
        if (!p.paged && npg == kChunk / kPage) {
          // whole chunk of a contiguous cache: one 64-row box per half
          mbar_arrive_expect_tx(&full[stage], 2u * C::kHalves * kChunk * 128);
          for (int h = 0; h < C::kHalves; ++h) {
            tma_load_3d(kst + h * kChunk * 128, &tm_k64, &full[stage], h * 64, k0, slab, pol);
            tma_load_3d(vst + h * kChunk * 128, &tm_v64, &full[stage], h * 64, k0, slab, pol);
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
              uint4* kz = reinterpret_cast<uint4*>(kst + h * kChunk * 128 + j * kPage * 128);
              uint4* vz = reinterpret_cast<uint4*>(vst + h * kChunk * 128 + j * kPage * 128);
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
                tma_load_3d(kst + h * kChunk * 128 + j * kPage * 128, &tm_k, &full[stage], h * 64,
                            row, zc[j], pol);
                tma_load_3d(vst + h * kChunk * 128 + j * kPage * 128, &tm_v, &full[stage], h * 64,
                            row, zc[j], pol);
              }
            }
          } else {
            mbar_arrive(&full[stage]);
          }
        }
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      // drain copies still in flight (only matters after an abort)
      const int issued = n_chunks;
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int last = st + ((issued - 1 - st) / kStages) * kStages;
        mbar_wait_drain(&full[st], static_cast<uint32_t>((last / kStages) & 1), p.status);
      }
    }
    return;
  }

  // ---------------- consumers: warp w = query head g*G + w ----------------
  const int h = g * G + warp;
  const int t = lane & 3;
  const int ra = lane >> 2, rb = ra + 8;  // block rows owned by this thread

  // block keys/values (RoPE'd) into shared memory, by the split that owns them.
  // One item = 8 consecutive dims d0..d0+7 of block row j and their rotary
  // partners d0+D/2..: four 16-byte loads, all issued before any arithmetic.
  if (has_block) {
    constexpr int kItems = kPage * (D / 16);
    for (int it = threadIdx.x; it < kItems; it += 32 * G) {
      const int j = it / (D / 16);
      const int d0 = (it - j * (D / 16)) * 8;
      const size_t src = (static_cast<size_t>(b * kBlock + j) * p.n_kv_heads + g) * D + d0;
      const uint4 k1 = *reinterpret_cast<const uint4*>(p.k_blk + src);
      const uint4 k2 = *reinterpret_cast<const uint4*>(p.k_blk + src + D / 2);
      const uint4 v1 = *reinterpret_cast<const uint4*>(p.v_blk + src);
      const uint4 v2 = *reinterpret_cast<const uint4*>(p.v_blk + src + D / 2);
      const uint32_t kw1[4] = {k1.x, k1.y, k1.z, k1.w}, kw2[4] = {k2.x, k2.y, k2.z, k2.w};
      uint32_t r1[4], r2[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float o1[2], o2[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int d = d0 + 2 * q + e;
          const float x1 = __uint_as_float(e ? (kw1[q] & 0xFFFF0000u) : (kw1[q] << 16));
          const float x2 = __uint_as_float(e ? (kw2[q] & 0xFFFF0000u) : (kw2[q] << 16));
          float sn, cs;
          rope_sincos(L + j, rope_hi[d], rope_lo[d], &sn, &cs);
          o1[e] = x1 * cs - x2 * sn;
          o2[e] = x2 * cs + x1 * sn;
        }
        r1[q] = pack_bf16(o1[0], o1[1]);
        r2[q] = pack_bf16(o2[0], o2[1]);
      }
      // swizzled 16-byte chunks: dims d0.. sit in half d0 >> 6, chunk (d0 & 63) >> 3
      const int e2 = d0 + D / 2;
      const int off1 = (d0 >> 6) * kChunk * 128 + j * 128 + ((((d0 & 63) >> 3) ^ (j & 7)) << 4);
      const int off2 = (e2 >> 6) * kChunk * 128 + j * 128 + ((((e2 & 63) >> 3) ^ (j & 7)) << 4);
      *reinterpret_cast<uint4*>(blk + off1) = make_uint4(r1[0], r1[1], r1[2], r1[3]);
      *reinterpret_cast<uint4*>(blk + off2) = make_uint4(r2[0], r2[1], r2[2], r2[3]);
      *reinterpret_cast<uint4*>(blk + C::kBlkV + off1) = v1;
      *reinterpret_cast<uint4*>(blk + C::kBlkV + off2) = v2;
    }
    named_bar_sync(1, 32 * G);
  }

  // query fragments (A operand of m16n8k16), rotated in registers: element d
  // and its RoPE partner d + D/2 sit in the same thread, D/32 k-steps apart.
  uint32_t qf[D / 16][4];
  {
    float qv[D / 16][2][4];  // [k-step][row a/b][k offsets 2t, 2t+1, 2t+8, 2t+9]
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int row = r ? rb : ra;
        const uint16_t* src =
            p.q_blk + (static_cast<size_t>(b * kBlock + row) * p.n_q_heads + h) * D + kk * 16 + 2 * t;
        const uint32_t lo = *reinterpret_cast<const uint32_t*>(src);
        const uint32_t hi = *reinterpret_cast<const uint32_t*>(src + 8);
        qv[kk][r][0] = __uint_as_float(lo << 16);
        qv[kk][r][1] = __uint_as_float(lo & 0xFFFF0000u);
        qv[kk][r][2] = __uint_as_float(hi << 16);
        qv[kk][r][3] = __uint_as_float(hi & 0xFFFF0000u);
      }
    }
#pragma unroll
    for (int kk = 0; kk < D / 32; ++kk) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = kk * 16 + 2 * t + (e & 1) + ((e >> 1) << 3);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int pos = Lc + (r ? rb : ra);
          float sn, cs;
          rope_sincos(pos, rope_hi[d], rope_lo[d], &sn, &cs);
          const float x1 = qv[kk][r][e], x2 = qv[kk + D / 32][r][e];
          qv[kk][r][e] = x1 * cs - x2 * sn;
          qv[kk + D / 32][r][e] = x2 * cs + x1 * sn;
        }
      }
    }
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qf[kk][0] = pack_bf16(qv[kk][0][0], qv[kk][0][1]);
      qf[kk][1] = pack_bf16(qv[kk][1][0], qv[kk][1][1]);
      qf[kk][2] = pack_bf16(qv[kk][0][2], qv[kk][0][3]);
      qf[kk][3] = pack_bf16(qv[kk][1][2], qv[kk][1][3]);
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

  // iteration -1 is the 16 block keys (only in the split that owns them), then
  // the context chunks; one copy of the chunk code keeps the loop in the
  // instruction cache
  uint32_t stage = 0, phase = 0;
  for (int c = has_block ? -1 : 0; c < n_chunks; ++c) {
    uint32_t kb, vb;
    int n_valid;
    uint8_t* vst = nullptr;
    if (c < 0) {
      kb = smem_u32(blk);
      vb = kb + C::kBlkV;
      n_valid = kPage;
    } else {
      const bool ok = mbar_wait(&full[stage], phase, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;
      uint8_t* kst = smem + stage * C::kStage;
      vst = kst + C::kTile;
      kb = smem_u32(kst);
      vb = smem_u32(vst);
      n_valid = min(kChunk, key_end - (key_begin + c * kChunk));
      const int n_fill = ((n_valid + 15) >> 4) << 4;
      if (n_valid < n_fill) {
        // rows past the length inside the last 16-key group: zero V so that
        // 0-probability keys cannot inject NaN/Inf from stale memory
        for (int i = lane; i < (n_fill - n_valid) * C::kHalves * 8; i += 32) {
          const int row = n_valid + i / (C::kHalves * 8);
          const int ch = i % (C::kHalves * 8);
          *reinterpret_cast<uint4*>(vst + (ch >> 3) * kChunk * 128 + row * 128 +
                                    (((ch & 7) ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
    }
    attend_chunk<D>(qf, kb, vb, n_valid, p.scale_log2, o, m_a, m_b, l_a, l_b);
    if (c >= 0) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == kStages) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
  griddep_launch_dependents();

  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

  const size_t unit = (static_cast<size_t>(b) * p.n_kv_heads + g) * p.splits + s_idx;
  float* po = p.part_o + unit * p.rows * D;
  float* pml = p.part_ml + unit * p.rows * 2;
  const int rra = warp * kBlock + ra, rrb = warp * kBlock + rb;
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int d = dt * 8 + 2 * t;
    *reinterpret_cast<float2*>(po + static_cast<size_t>(rra) * D + d) = make_float2(o[dt][0], o[dt][1]);
    *reinterpret_cast<float2*>(po + static_cast<size_t>(rrb) * D + d) = make_float2(o[dt][2], o[dt][3]);
  }
  if (t == 0) {
    *reinterpret_cast<float2*>(pml + rra * 2) = make_float2(m_a, l_a);
    *reinterpret_cast<float2*>(pml + rrb * 2) = make_float2(m_b, l_b);
  }
}

// Merge the split partials by log-sum-exp.  One warp per output row (b, i, h),
// four rows per CTA.  A lane holds the (max, sum) pairs of splits lane and
// lane + 32 and D/32 output elements; the partial rows are read in batches of
// kBatch splits whose loads are all in flight together, and the first batch
// is requested before the maxima are known, so a row costs about one global
// round trip per batch.
constexpr int kMaxSplits = 64;
constexpr int kCombineRows = 4;

template <int D>
__global__ void __launch_bounds__(32 * kCombineRows) attn_combine_kernel(const CombineParams p) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int per = D / 32;  // 2 or 4 elements per lane
  constexpr int kBatch = 16;
  using Vec = typename std::conditional<per == 4, float4, float2>::type;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kCombineRows + warp;
  const int rows_out = p.batch * kBlock * p.n_q_heads;
  if (row >= rows_out) return;
  const int b = row / (kBlock * p.n_q_heads);
  const int rem = row - b * kBlock * p.n_q_heads;
  const int i = rem / p.n_q_heads;
  const int h = rem - i * p.n_q_heads;
  const int g = h / p.group, w = h - g * p.group;
  const int rr = w * kBlock + i;
  const size_t unit0 = (static_cast<size_t>(b) * p.n_kv_heads + g) * p.splits;
  const int L = p.seq_len[b];
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
  if (L < 0 || L > p.limit) return;
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

template <int D>
int launch_attention(const dflash_dims& dims, const Plan& plan, const dflash_kv_view& cache,
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
  const int smem = 1024 + kStages * C::kStage + C::kBlkTile + D * 4 + 2 * kStages * 8 + 16;
  if ((rc = set_smem_limit(reinterpret_cast<const void*>(block_attention_kernel<D>), smem)))
    return rc;
  rc = launch(block_attention_kernel<D>, dim3(plan.att_splits, dims.n_kv_heads, dims.batch),
              dim3(32 * (p.group + 1)), smem, stream, tm_k, tm_v, tm_k64, tm_v64, p);
  if (rc) return rc;
  const int rows_out = dims.batch * kBlock * dims.n_q_heads;
  return launch(attn_combine_kernel<D>, dim3((rows_out + kCombineRows - 1) / kCombineRows),
                dim3(32 * kCombineRows), 0, stream, cp);
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" int dflash_block_attention(const dflash_dims* dims, const void* q_blk,
                                      const void* k_blk, const void* v_blk,
                                      const dflash_kv_view* cache, float scale, void* out,
                                      void* ws, size_t ws_bytes, dflash_stream_t stream) {
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
  return dims->head_dim == 128 ? launch_attention<128>(*dims, plan, *cache, p, cp, s)
                               : launch_attention<64>(*dims, plan, *cache, p, cp, s);
}
