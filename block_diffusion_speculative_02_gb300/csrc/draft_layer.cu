// Next: the rest of one drafter layer (its block Q/K/V, the output
// projection and the MLP) around the dual-source block attention.
//
// "DFlash双实现对比" (hotelren.com) §1: the drafter reuses Qwen3 components
// (RMSNorm, rotary embedding, MLP), i.e. pre-norm decoder layers with a
// per-head RMSNorm of q and k and a SwiGLU MLP; "dflash-mlx" (dpshk.com)
// 块扩散草稿 steps 1-2: the whole block (staged token + 15 masks) goes through
// one forward.  Per layer, on the 16 B rows of the block:
//   h  = RMSNorm(x) * ln1
//   q  = RMSNorm_head(h W_q^T) * q_norm,  k = RMSNorm_head(h W_k^T) * k_norm,
//   v  = h W_v^T                              (dflash_draft_qkv)
//   O  = block attention (dflash_block_attention, which rotates q and k)
//   x1 = x + O W_o^T,  h2 = RMSNorm(x1) * ln2
//   x2 = x1 + (silu(h2 W_gate^T) * (h2 W_up^T)) W_down^T   (dflash_draft_mlp)
//
// Every product is the stream-K GEMM of streamk_gemm.cuh (the weights are
// streamed once by every SM of the budget; the CTA completing a tile's sum
// finishes it).  The RMSNorm's per-row factor commutes with the GEMM, so the
// GEMMs read x * g (carried as a bf16 pair hi + lo, exact to ~2^-17) and the
// finishers apply 1/rms(x): no normalised copy of x is ever rounded to bf16.
// The gate and up tiles of the same features are finished together (paired
// tickets), so silu(g) * u never leaves the SM in fp32.
#include "streamk_gemm.cuh"
#include "tile_gemm.cuh"

namespace dflash {
namespace {

using sk::GemmCore;
using sk::take4;

constexpr int kTokGroup = 4;  // token rows a warp finishes together (loads in flight)

__device__ __forceinline__ uint2 pack4(float a, float b, float c, float d) {
  return make_uint2(static_cast<uint32_t>(float_to_bf16_bits(a)) |
                        (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16),
                    static_cast<uint32_t>(float_to_bf16_bits(c)) |
                        (static_cast<uint32_t>(float_to_bf16_bits(d)) << 16));
}

__device__ __forceinline__ float4 ld4_bf16(const uint16_t* src) {
  const uint2 w = *reinterpret_cast<const uint2*>(src);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
}

// Store a (x) as the bf16 pair hi + lo at rows tok and n_tok + tok.
__device__ __forceinline__ void store_hilo4(uint16_t* hl, int n_tok, int width, int tok, int f0,
                                            const float (&a)[4]) {
  float hi[4], lo[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    hi[e] = bf16_bits_to_float(float_to_bf16_bits(a[e]));
    lo[e] = a[e] - hi[e];
  }
  *reinterpret_cast<uint2*>(hl + static_cast<size_t>(tok) * width + f0) =
      pack4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint2*>(hl + (static_cast<size_t>(n_tok) + tok) * width + f0) =
      pack4(lo[0], lo[1], lo[2], lo[3]);
}

__device__ __forceinline__ float silu(float x) { return x / (1.f + __expf(-x)); }

// Per token row (one CTA of 128 threads per row): sum(x^2), and x * g either
// as a hi/lo bf16 pair (hl != null) or rounded once to bf16 (out != null).
// A thread's loads of up to kRowBatch groups of 4 features go out together
// before any of them is used (the row is a handful of round trips otherwise).
constexpr int kRowBatch = 8;

__global__ void __launch_bounds__(128) row_gain_kernel(const uint16_t* __restrict__ x,
                                                       const uint16_t* __restrict__ gain, int H,
                                                       int n_tok, uint16_t* __restrict__ hl,
                                                       float* __restrict__ ss,
                                                       uint16_t* __restrict__ out) {
  griddep_wait();
  __shared__ float red[4];
  const int row = blockIdx.x;
  const uint16_t* xr = x + static_cast<size_t>(row) * H;
  float sq = 0.f;
  for (int base = threadIdx.x * 4; base < H; base += kRowBatch * 128 * 4) {
    float4 v[kRowBatch], gv[kRowBatch];
#pragma unroll
    for (int u = 0; u < kRowBatch; ++u) {
      const int f0 = base + u * 128 * 4;
      v[u] = f0 < H ? ld4_bf16(xr + f0) : make_float4(0.f, 0.f, 0.f, 0.f);
      gv[u] = (gain && f0 < H) ? ld4_bf16(gain + f0) : make_float4(1.f, 1.f, 1.f, 1.f);
    }
#pragma unroll
    for (int u = 0; u < kRowBatch; ++u) {
      const int f0 = base + u * 128 * 4;
      if (f0 >= H) break;
      sq += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
      const float a[4] = {v[u].x * gv[u].x, v[u].y * gv[u].y, v[u].z * gv[u].z, v[u].w * gv[u].w};
      if (hl) store_hilo4(hl, n_tok, H, row, f0, a);
      if (out)
        *reinterpret_cast<uint2*>(out + static_cast<size_t>(row) * H + f0) =
            pack4(a[0], a[1], a[2], a[3]);
    }
  }
  griddep_launch_dependents();
  if (!ss) return;
#pragma unroll
  for (int off = 16; off; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sq;
  __syncthreads();
  if (threadIdx.x == 0) ss[row] = red[0] + red[1] + red[2] + red[3];
}

struct DraftParams {
  int hidden, ffn, n_q_heads, n_kv_heads, head_dim;
  float rms_eps;
  // q/k/v
  const float* ss_rows;      // [n_tok] sum(x^2) of the layer input
  const uint16_t* q_norm_w;  // [D] or null
  const uint16_t* k_norm_w;
  uint16_t* q_out;           // [n_tok, Hq*D]
  uint16_t* k_out;           // [n_tok, Hkv*D]
  uint16_t* v_out;
  // output projection / MLP
  const uint16_t* x;         // [n_tok, H] layer input (residual)
  const uint16_t* ln2_w;     // [H]
  float* x1;                 // [n_tok, H] x + O W_o^T
  uint16_t* xhl;             // [2, n_tok, H] hi/lo of x1 * ln2
  float* ss_x1;              // [H/128, n_tok] partial sums of x1^2
  uint16_t* mhl;             // [2, n_tok, F] hi/lo of silu(g) * u
  uint16_t* x_out;           // [n_tok, H]
};

// q/k/v: scale by 1/rms(x), per-head RMSNorm of q and k, bf16 store.  A lane
// owns 4 consecutive features; a head spans D / 4 lanes.
struct QkvFin {
  using Params = DraftParams;
  static __device__ void prologue(const GemmCore&, const Params&) {}
  static __device__ void finish(const GemmCore& g, const Params& p, int o, int c, uint8_t*) {
    const int et = threadIdx.x - 64, warp = et >> 5, lane = et & 31;
    const int D = p.head_dim;
    const int region = (o >= g.a_split[0]) + (o >= g.a_split[1]);  // 0 q, 1 k, 2 v
    const int tile0 = region == 0 ? 0 : (region == 1 ? g.a_split[0] : g.a_split[1]);
    const int feat0 = (o - tile0) * 128 + lane * 4;
    const int width = (region == 0 ? p.n_q_heads : p.n_kv_heads) * D;
    uint16_t* out = region == 0 ? p.q_out : (region == 1 ? p.k_out : p.v_out);
    const uint16_t* nw = region == 0 ? p.q_norm_w : (region == 1 ? p.k_norm_w : nullptr);
    const float4 gn = nw ? ld4_bf16(nw + feat0 % D) : make_float4(1.f, 1.f, 1.f, 1.f);
    const int t0 = c * g.chunk_rows;
    const int nt = min(g.chunk_rows, g.n_tok - t0);
#pragma unroll 1
    for (int j0 = warp * kTokGroup; j0 < nt; j0 += 4 * kTokGroup) {
      float4 v[kTokGroup];
      float r[kTokGroup];
#pragma unroll
      for (int k = 0; k < kTokGroup; ++k) {
        if (j0 + k < nt) {
          v[k] = take4(g, t0 + j0 + k, o * 128 + lane * 4);
          r[k] = rsqrtf(__ldcg(p.ss_rows + t0 + j0 + k) / p.hidden + p.rms_eps);
        }
      }
#pragma unroll
      for (int k = 0; k < kTokGroup; ++k) {
        if (j0 + k >= nt) break;
        float x4[4] = {v[k].x * r[k], v[k].y * r[k], v[k].z * r[k], v[k].w * r[k]};
        if (nw) {
          float sq = x4[0] * x4[0] + x4[1] * x4[1] + x4[2] * x4[2] + x4[3] * x4[3];
          for (int off = D / 8; off; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
          const float rs = rsqrtf(sq / D + p.rms_eps);
          x4[0] *= rs * gn.x;
          x4[1] *= rs * gn.y;
          x4[2] *= rs * gn.z;
          x4[3] *= rs * gn.w;
        }
        *reinterpret_cast<uint2*>(out + static_cast<size_t>(t0 + j0 + k) * width + feat0) =
            pack4(x4[0], x4[1], x4[2], x4[3]);
      }
    }
  }
};

// Output projection: x1 = x + O W_o^T (fp32), hi/lo of x1 * ln2 for the MLP
// and the tile's partial sums of x1^2 (the RMSNorm factor is applied later).
struct OprojFin {
  using Params = DraftParams;
  static __device__ void prologue(const GemmCore&, const Params&) {}
  static __device__ void finish(const GemmCore& g, const Params& p, int o, int c, uint8_t*) {
    const int et = threadIdx.x - 64, warp = et >> 5, lane = et & 31;
    const int H = p.hidden;
    const int f0 = o * 128 + lane * 4;
    const float4 gn = ld4_bf16(p.ln2_w + f0);
    const int t0 = c * g.chunk_rows;
    const int nt = min(g.chunk_rows, g.n_tok - t0);
#pragma unroll 1
    for (int j0 = warp * kTokGroup; j0 < nt; j0 += 4 * kTokGroup) {
      float4 a[kTokGroup], xin[kTokGroup];
#pragma unroll
      for (int k = 0; k < kTokGroup; ++k) {
        if (j0 + k < nt) {
          a[k] = take4(g, t0 + j0 + k, f0);
          xin[k] = ld4_bf16(p.x + static_cast<size_t>(t0 + j0 + k) * H + f0);
        }
      }
#pragma unroll
      for (int k = 0; k < kTokGroup; ++k) {
        if (j0 + k >= nt) break;
        const int tok = t0 + j0 + k;
        const float4 y = make_float4(xin[k].x + a[k].x, xin[k].y + a[k].y, xin[k].z + a[k].z,
                                     xin[k].w + a[k].w);
        *reinterpret_cast<float4*>(p.x1 + static_cast<size_t>(tok) * H + f0) = y;
        const float z[4] = {y.x * gn.x, y.y * gn.y, y.z * gn.z, y.w * gn.w};
        store_hilo4(p.xhl, g.n_tok, H, tok, f0, z);
        float sq = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
#pragma unroll
        for (int off = 16; off; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
        if (lane == 0) p.ss_x1[static_cast<size_t>(o) * g.n_tok + tok] = sq;
      }
    }
  }
};

// Gate and up tiles of the same 128 features, finished together: the RMSNorm
// factor of x1, silu(gate) * up, stored as hi/lo for the down projection.
struct GateUpFin {
  using Params = DraftParams;
  static __device__ void prologue(const GemmCore&, const Params&) {}
  static __device__ void finish(const GemmCore& g, const Params& p, int o, int c, uint8_t*) {
    const int et = threadIdx.x - 64, warp = et >> 5, lane = et & 31;
    const int F = p.ffn, n_ss = p.hidden / 128;
    const int f0 = o * 128 + lane * 4;  // o < F / 128: the gate tile of the pair
    const int t0 = c * g.chunk_rows;
    const int nt = min(g.chunk_rows, g.n_tok - t0);
#pragma unroll 1
    for (int j0 = warp * kTokGroup; j0 < nt; j0 += 4 * kTokGroup) {
      float4 gv[kTokGroup], uv[kTokGroup];
      float ssum[kTokGroup];
#pragma unroll
      for (int k = 0; k < kTokGroup; ++k) {
        ssum[k] = 0.f;
        if (j0 + k < nt) {
          const int tok = t0 + j0 + k;
          gv[k] = take4(g, tok, f0);
          uv[k] = take4(g, tok, F + f0);
          for (int q = lane; q < n_ss; q += 32)
            ssum[k] += __ldcg(p.ss_x1 + static_cast<size_t>(q) * g.n_tok + tok);
        }
      }
#pragma unroll
      for (int k = 0; k < kTokGroup; ++k) {
        if (j0 + k >= nt) break;
        float tot = ssum[k];
#pragma unroll
        for (int off = 16; off; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
        const float r = rsqrtf(tot / p.hidden + p.rms_eps);
        const float m[4] = {silu(gv[k].x * r) * (uv[k].x * r), silu(gv[k].y * r) * (uv[k].y * r),
                            silu(gv[k].z * r) * (uv[k].z * r), silu(gv[k].w * r) * (uv[k].w * r)};
        store_hilo4(p.mhl, g.n_tok, F, t0 + j0 + k, f0, m);
      }
    }
  }
};

// Down projection: x2 = x1 + M W_down^T, bf16.
struct DownFin {
  using Params = DraftParams;
  static __device__ void prologue(const GemmCore&, const Params&) {}
  static __device__ void finish(const GemmCore& g, const Params& p, int o, int c, uint8_t*) {
    const int et = threadIdx.x - 64, warp = et >> 5, lane = et & 31;
    const int H = p.hidden;
    const int f0 = o * 128 + lane * 4;
    const int t0 = c * g.chunk_rows;
    const int nt = min(g.chunk_rows, g.n_tok - t0);
#pragma unroll 1
    for (int j0 = warp * kTokGroup; j0 < nt; j0 += 4 * kTokGroup) {
      float4 a[kTokGroup], xr[kTokGroup];
#pragma unroll
      for (int k = 0; k < kTokGroup; ++k) {
        if (j0 + k < nt) {
          a[k] = take4(g, t0 + j0 + k, f0);
          xr[k] = __ldcg(reinterpret_cast<const float4*>(p.x1 + static_cast<size_t>(t0 + j0 + k) * H + f0));
        }
      }
#pragma unroll
      for (int k = 0; k < kTokGroup; ++k) {
        if (j0 + k >= nt) break;
        *reinterpret_cast<uint2*>(p.x_out + static_cast<size_t>(t0 + j0 + k) * H + f0) =
            pack4(xr[k].x + a[k].x, xr[k].y + a[k].y, xr[k].z + a[k].z, xr[k].w + a[k].w);
      }
    }
  }
};

// Past 256 token rows (batch 17 and up) the MLP's two GEMMs are bound by the
// tensor cores: they run on the clustered tile GEMM of tile_gemm.cuh with the
// same operands (hi/lo pairs summed along a doubled K) and these epilogues,
// thread = token row.
constexpr int kTiledDraftRows = 257;

// q/k/v: one tile of BN features of q, k or v (weight maps 0, 1, 2): the
// row's 1/rms(x), per-head RMSNorm of q and k (a first pass over the head's
// columns for the sum of squares), bf16 store.
struct QkvTileEpi {
  using Params = DraftParams;
  static __device__ void setup(const Params&, float*, int) {}
  static __device__ void prologue(const TileCore&, const Params&) {}
  static __device__ void tile(const TileCore& p, const Params& e, int n, uint32_t tacc, int row,
                              const float*) {
    const int D = e.head_dim;
    const int region = n < p.b_split ? 0 : (n < p.b_split2 ? 1 : 2);  // q, k, v
    const int f0 = (n - (region == 0 ? 0 : (region == 1 ? p.b_split : p.b_split2))) * p.bn;
    const int width = (region == 0 ? e.n_q_heads : e.n_kv_heads) * D;
    uint16_t* out = region == 0 ? e.q_out : (region == 1 ? e.k_out : e.v_out);
    const uint16_t* nw = region == 0 ? e.q_norm_w : (region == 1 ? e.k_norm_w : nullptr);
    const bool live = row < p.rows;
    const float r = live ? rsqrtf(__ldcg(e.ss_rows + row) / e.hidden + e.rms_eps) : 0.f;
    for (int h0 = 0; h0 < p.bn; h0 += D) {
      float rs = 1.f;
      if (nw) {
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
        rs = rsqrtf(sq / D + e.rms_eps);
      }
      for (int c0 = 0; c0 < D; c0 += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tacc + h0 + c0, v);
        tmem_ld_wait();
        if (!live) continue;
        const float s = r * rs;
        uint16_t* dst = out + static_cast<size_t>(row) * width + f0 + h0 + c0;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 gn = nw ? ld4_bf16(nw + c0 + 4 * q4) : make_float4(1.f, 1.f, 1.f, 1.f);
          *reinterpret_cast<uint2*>(dst + 4 * q4) =
              pack4(__uint_as_float(v[4 * q4]) * s * gn.x, __uint_as_float(v[4 * q4 + 1]) * s * gn.y,
                    __uint_as_float(v[4 * q4 + 2]) * s * gn.z,
                    __uint_as_float(v[4 * q4 + 3]) * s * gn.w);
        }
      }
    }
  }
};

// Output projection: x1 = x + O W_o^T (fp32), hi/lo of x1 * ln2 and, per 128
// features, the partial sums of x1^2 (the layout of the streamed path).
struct OprojTileEpi {
  using Params = DraftParams;
  static __device__ void setup(const Params&, float*, int) {}
  static __device__ void prologue(const TileCore&, const Params&) {}
  static __device__ void tile(const TileCore& p, const Params& e, int n, uint32_t tacc, int row,
                              const float*) {
    const int H = e.hidden, f0 = n * p.bn;
    const bool live = row < p.rows;
    for (int half = 0; half < p.bn; half += 128) {
      float sq = 0.f;
      for (int c0 = half; c0 < half + 128; c0 += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tacc + c0, v);
        tmem_ld_wait();
        if (!live) continue;
        const size_t off = static_cast<size_t>(row) * H + f0 + c0;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float4 xin = ld4_bf16(e.x + off + 4 * q4);
          const float4 gn = ld4_bf16(e.ln2_w + f0 + c0 + 4 * q4);
          const float4 y = make_float4(xin.x + __uint_as_float(v[4 * q4]),
                                       xin.y + __uint_as_float(v[4 * q4 + 1]),
                                       xin.z + __uint_as_float(v[4 * q4 + 2]),
                                       xin.w + __uint_as_float(v[4 * q4 + 3]));
          *reinterpret_cast<float4*>(e.x1 + off + 4 * q4) = y;
          sq += y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
          const float z[4] = {y.x * gn.x, y.y * gn.y, y.z * gn.z, y.w * gn.w};
          store_hilo4(e.xhl, p.rows, H, row, f0 + c0 + 4 * q4, z);
        }
      }
      if (live) e.ss_x1[static_cast<size_t>((f0 + half) / 128) * p.rows + row] = sq;
    }
  }
};

// Gate and up: CTA c of a pair loads the rows of the same 128 features from
// W_gate (c = 0) or W_up (c = 1), so accumulator columns [0, 128) are the
// gate and [128, 256) the up products of features 128 n ...: the RMSNorm
// factor of x1, silu(gate) * up, hi/lo for the down projection.
struct GateUpTileEpi {
  using Params = DraftParams;
  static __device__ void setup(const Params&, float*, int) {}
  static __device__ void prologue(const TileCore&, const Params&) {}
  static __device__ void tile(const TileCore& p, const Params& e, int n, uint32_t tacc, int row,
                              const float*) {
    const int n_ss = e.hidden / 128, f0 = n * 128;
    const bool live = row < p.rows;
    float tot = 0.f;
    if (live) {
#pragma unroll 8
      for (int q = 0; q < n_ss; ++q) tot += __ldcg(e.ss_x1 + static_cast<size_t>(q) * p.rows + row);
    }
    const float r = rsqrtf(tot / e.hidden + e.rms_eps);
    for (int c0 = 0; c0 < 128; c0 += 16) {
      uint32_t gv[16], uv[16];
      tmem_ld_32x32b_x16(tacc + c0, gv);
      tmem_ld_32x32b_x16(tacc + 128 + c0, uv);
      tmem_ld_wait();
      if (!live) continue;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float m[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          m[j] = silu(__uint_as_float(gv[4 * q4 + j]) * r) * (__uint_as_float(uv[4 * q4 + j]) * r);
        store_hilo4(e.mhl, p.rows, e.ffn, row, f0 + c0 + 4 * q4, m);
      }
    }
  }
};

// Down: x2 = x1 + M W_down^T, bf16.
struct DownTileEpi {
  using Params = DraftParams;
  static __device__ void setup(const Params&, float*, int) {}
  static __device__ void prologue(const TileCore&, const Params&) {}
  static __device__ void tile(const TileCore& p, const Params& e, int n, uint32_t tacc, int row,
                              const float*) {
    const int H = e.hidden, f0 = n * p.bn;
    const bool live = row < p.rows;
    for (int c0 = 0; c0 < p.bn; c0 += 16) {
      uint32_t v[16];
      tmem_ld_32x32b_x16(tacc + c0, v);
      tmem_ld_wait();
      if (!live) continue;
      const size_t off = static_cast<size_t>(row) * H + f0 + c0;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(e.x1 + off) + q4);
        *reinterpret_cast<uint2*>(e.x_out + off + 4 * q4) =
            pack4(x.x + __uint_as_float(v[4 * q4]), x.y + __uint_as_float(v[4 * q4 + 1]),
                  x.z + __uint_as_float(v[4 * q4 + 2]), x.w + __uint_as_float(v[4 * q4 + 3]));
      }
    }
  }
};

// The token operand of a tiled GEMM: the hi rows (map 0) and lo rows (map 1)
// of a [2, rows, cols] pair.
int hilo_token_maps(TokenMaps& am, const uint16_t* hl, int rows, int cols) {
  const uint64_t pitch = static_cast<uint64_t>(cols) * 2;
  int rc = make_tmap_2d_bf16(&am.m[0], hl, cols, rows, pitch, 64, kTileM);
  if (!rc) rc = make_tmap_2d_bf16(&am.m[1], hl + static_cast<size_t>(rows) * cols, cols, rows,
                                  pitch, 64, kTileM);
  for (int l = 2; l < kMaxCtxLayers; ++l) am.m[l] = am.m[0];
  return rc;
}

// The GEMM fields for n_tok token rows of a K-column operand.
GemmCore gemm_shape(const DraftPlan& plan, int k_cols, int out_tiles, int hilo,
                    uint32_t* tickets, float* part, void* ws) {
  GemmCore g = sk::gemm_dims(plan.ntok, k_cols, out_tiles, hilo);
  g.status = ws_at<uint32_t>(ws, plan.off_status);
  g.part = part;
  g.tickets = tickets;
  return g;
}

int token_map(sk::BMaps& bm, const void* base, int cols, int rows, int box_rows) {
  int rc = make_tmap_2d_bf16(&bm.m[0], base, cols, rows, static_cast<uint64_t>(cols) * 2, 64,
                             box_rows);
  for (int l = 1; l < kMaxCtxLayers; ++l) bm.m[l] = bm.m[0];
  return rc;
}

int weight_map(CUtensorMap* m, const void* w, int rows, int cols) {
  return make_tmap_2d_bf16(m, w, cols, rows, static_cast<uint64_t>(cols) * 2, 64, 128);
}

}  // namespace

int make_draft_plan(const dflash_dims& d, int ffn, DraftPlan* out) {
  int rc = check_dims(&d);
  if (rc) return rc;
  if (ffn < 128 || ffn % 128) return DFLASH_E_UNSUPPORTED;
  if ((d.n_q_heads * d.head_dim) % 128) return DFLASH_E_UNSUPPORTED;
  DraftPlan p = {};
  p.num_sms = current_num_sms();
  if (p.num_sms <= 0) return DFLASH_E_CUDA;
  p.budget_sms = d.sm_budget > 0 && d.sm_budget < p.num_sms ? d.sm_budget : p.num_sms;
  p.ntok = d.batch * kBlock;
  const int H = d.hidden, qd = d.n_q_heads * d.head_dim, kvd = d.n_kv_heads * d.head_dim;
  const int chunks_hilo = (p.ntok + 127) / 128, chunks_plain = (p.ntok + 255) / 256;
  p.qkv_tiles = (qd + 2 * kvd) / 128;
  p.o_tiles = H / 128;
  p.gu_tiles = 2 * ffn / 128;
  p.down_tiles = H / 128;
  auto al = [](size_t x, size_t a) { return (x + a - 1) / a * a; };
  // partial tiles of the stream-K GEMMs: Q/K/V and the output projection
  // share region a, gate|up and down region b (each sized for the larger)
  const int nt = p.ntok;
  size_t acc_a = sk::partial_bytes(sk::gemm_dims(nt, H, p.qkv_tiles, 1), p.num_sms);
  const size_t o_bytes = sk::partial_bytes(sk::gemm_dims(nt, qd, p.o_tiles, 0), p.num_sms);
  if (o_bytes > acc_a) acc_a = o_bytes;
  size_t acc_b = sk::partial_bytes(sk::gemm_dims(nt, H, p.gu_tiles, 1), p.num_sms);
  const size_t d_bytes = sk::partial_bytes(sk::gemm_dims(nt, ffn, p.down_tiles, 1), p.num_sms);
  if (d_bytes > acc_b) acc_b = d_bytes;
  // buffers that do not depend on ffn first, so that the Q/K/V and token
  // steps find them at the same offsets whatever ffn the workspace was sized for
  size_t off = 0;
  p.off_status = off;  off += 64;
  p.off_lm_ticket = off; off += 64;
  p.off_tickets_qkv = off; off = al(off + 4 * (size_t)p.qkv_tiles * chunks_hilo, 64);
  p.off_tickets_o = off;   off = al(off + 4 * (size_t)p.o_tiles * chunks_plain, 256);
  p.off_keys = off;    off = al(off + 8 * (size_t)p.ntok, 256);
  p.off_ss_rows = off; off = al(off + 4 * (size_t)p.ntok, 256);
  p.off_ss_x1 = off;   off = al(off + 4 * (size_t)p.ntok * (H / 128), 256);
  p.off_xhl = off;     off = al(off + 2 * 2 * (size_t)p.ntok * H, 1024);
  p.off_x1 = off;      off = al(off + 4 * (size_t)p.ntok * H, 256);
  p.off_xg = off;      off = al(off + 2 * (size_t)p.ntok * H, 1024);
  p.off_acc_a = off;   off = al(off + acc_a, 256);
  p.ffn_begin = off;
  p.off_tickets_gu = off;  off = al(off + 4 * (size_t)p.gu_tiles * chunks_hilo, 64);
  p.off_tickets_down = off; off = al(off + 4 * (size_t)p.down_tiles * chunks_hilo, 1024);
  p.off_mhl = off;     off = al(off + 2 * 2 * (size_t)p.ntok * ffn, 1024);
  p.off_acc_b = off;   off = al(off + acc_b, 256);
  p.total = off;
  *out = p;
  return DFLASH_OK;
}

int launch_row_gain(const void* x, const void* gain, int H, int n_tok, void* hl, float* ss,
                    void* out, cudaStream_t st) {
  return launch(row_gain_kernel, dim3(n_tok), dim3(128), 0, st, static_cast<const uint16_t*>(x),
                static_cast<const uint16_t*>(gain), H, n_tok, static_cast<uint16_t*>(hl), ss,
                static_cast<uint16_t*>(out));
}

}  // namespace dflash

using namespace dflash;

extern "C" size_t dflash_draft_workspace_bytes(const dflash_dims* dims, int32_t ffn) {
  if (check_dims(dims)) return 0;
  DraftPlan p;
  if (make_draft_plan(*dims, ffn, &p)) return 0;
  return p.total;
}

extern "C" int dflash_draft_qkv(const dflash_dims* dims, const void* x, const void* ln1_w,
                                const void* w_q, const void* w_k, const void* w_v,
                                const void* q_norm_w, const void* k_norm_w, void* q_out,
                                void* k_out, void* v_out, void* ws, size_t ws_bytes,
                                dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_draft_qkv");
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!x || !ln1_w || !w_q || !w_k || !w_v || !q_out || !k_out || !v_out) return DFLASH_E_ARG;
  if (!aligned16(x) || !aligned16(w_q) || !aligned16(w_k) || !aligned16(w_v) ||
      !aligned16(q_out) || !aligned16(k_out) || !aligned16(v_out))
    return DFLASH_E_ALIGN;
  if (!ws) return DFLASH_E_WORKSPACE;
  DraftPlan plan;
  // the Q/K/V step does not touch the MLP buffers: size the plan for the
  // smallest MLP so that a workspace for any ffn is accepted
  if ((rc = make_draft_plan(*dims, 128, &plan))) return rc;
  if (ws_bytes < plan.ffn_begin) return DFLASH_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int H = dims->hidden, D = dims->head_dim;
  const int qd = dims->n_q_heads * D, kvd = dims->n_kv_heads * D;
  uint16_t* xhl = ws_at<uint16_t>(ws, plan.off_xhl);
  float* ss_rows = ws_at<float>(ws, plan.off_ss_rows);
  if ((rc = launch_row_gain(x, ln1_w, H, plan.ntok, xhl, ss_rows, nullptr, st))) return rc;

  DraftParams fp = {};
  fp.hidden = H;
  fp.n_q_heads = dims->n_q_heads;
  fp.n_kv_heads = dims->n_kv_heads;
  fp.head_dim = D;
  fp.rms_eps = dims->rms_eps;
  fp.ss_rows = ss_rows;
  fp.q_norm_w = static_cast<const uint16_t*>(q_norm_w);
  fp.k_norm_w = static_cast<const uint16_t*>(k_norm_w);
  fp.q_out = static_cast<uint16_t*>(q_out);
  fp.k_out = static_cast<uint16_t*>(k_out);
  fp.v_out = static_cast<uint16_t*>(v_out);

  const int tbn = (qd % 256 == 0 && kvd % 256 == 0) ? 256 : 128;
  if (plan.ntok >= kTiledDraftRows && qd % tbn == 0 && kvd % tbn == 0) {
    TileCore t = {};
    t.status = ws_at<uint32_t>(ws, plan.off_status);
    t.rows = plan.ntok;
    t.m_tiles = (plan.ntok + kTileM - 1) / kTileM;
    t.bn = tbn;
    t.n_tiles = (qd + 2 * kvd) / tbn;
    t.k_tiles = 2 * H / 64;
    t.layer_cols = H;
    t.b_split = qd / tbn;
    t.b_split2 = (qd + kvd) / tbn;
    t.b_cols = H;
    TokenMaps am;
    WeightMaps bm;
    if ((rc = hilo_token_maps(am, xhl, plan.ntok, H))) return rc;
    const uint64_t pitch = static_cast<uint64_t>(H) * 2;
    if ((rc = make_tmap_2d_bf16(&bm.m[0], w_q, H, qd, pitch, 64, tbn / 2)) ||
        (rc = make_tmap_2d_bf16(&bm.m[1], w_k, H, kvd, pitch, 64, tbn / 2)) ||
        (rc = make_tmap_2d_bf16(&bm.m[2], w_v, H, kvd, pitch, 64, tbn / 2)))
      return rc;
    return run_tile_gemm<QkvTileEpi>(t, am, bm, fp, st, plan.budget_sms);
  }

  GemmCore g = gemm_shape(plan, H, plan.qkv_tiles, 1, ws_at<uint32_t>(ws, plan.off_tickets_qkv),
                          ws_at<float>(ws, plan.off_acc_a), ws);
  g.a_split[0] = qd / 128;
  g.a_split[1] = (qd + kvd) / 128;
  sk::AMaps am;
  sk::BMaps bm;
  if ((rc = weight_map(&am.m[0], w_q, qd, H)) || (rc = weight_map(&am.m[1], w_k, kvd, H)) ||
      (rc = weight_map(&am.m[2], w_v, kvd, H)))
    return rc;
  if ((rc = token_map(bm, xhl, H, 2 * plan.ntok, g.chunk_rows))) return rc;
  return sk::run_streamk<QkvFin>(g, am, bm, fp, plan.budget_sms, st,
                                 plan.ffn_begin - plan.off_acc_a);
}

extern "C" int dflash_draft_mlp(const dflash_dims* dims, int32_t ffn, const void* x,
                                const void* attn_out, const void* w_o, const void* ln2_w,
                                const void* w_gate, const void* w_up, const void* w_down,
                                void* x_out, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_draft_mlp");
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!x || !attn_out || !w_o || !ln2_w || !w_gate || !w_up || !w_down || !x_out)
    return DFLASH_E_ARG;
  if (!aligned16(x) || !aligned16(attn_out) || !aligned16(w_o) || !aligned16(w_gate) ||
      !aligned16(w_up) || !aligned16(w_down) || !aligned16(x_out))
    return DFLASH_E_ALIGN;
  if (!ws) return DFLASH_E_WORKSPACE;
  DraftPlan plan;
  if ((rc = make_draft_plan(*dims, ffn, &plan))) return rc;
  if (ws_bytes < plan.total) return DFLASH_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int H = dims->hidden, qd = dims->n_q_heads * dims->head_dim;

  DraftParams fp = {};
  fp.hidden = H;
  fp.ffn = ffn;
  fp.rms_eps = dims->rms_eps;
  fp.x = static_cast<const uint16_t*>(x);
  fp.ln2_w = static_cast<const uint16_t*>(ln2_w);
  fp.x1 = ws_at<float>(ws, plan.off_x1);
  fp.xhl = ws_at<uint16_t>(ws, plan.off_xhl);
  fp.ss_x1 = ws_at<float>(ws, plan.off_ss_x1);
  fp.mhl = ws_at<uint16_t>(ws, plan.off_mhl);
  fp.x_out = static_cast<uint16_t*>(x_out);

  // 1. x1 = x + O W_o^T; hi/lo of x1 * ln2; sums of x1^2
  if (plan.ntok >= kTiledDraftRows) {
    TileCore t = {};
    t.status = ws_at<uint32_t>(ws, plan.off_status);
    t.rows = plan.ntok;
    t.m_tiles = (plan.ntok + kTileM - 1) / kTileM;
    t.bn = H % 256 == 0 ? 256 : 128;
    t.n_tiles = H / t.bn;
    t.k_tiles = qd / 64;
    t.layer_cols = qd;
    t.b_split = t.n_tiles;
    TokenMaps am;
    WeightMaps bm;
    if ((rc = make_tmap_2d_bf16(&am.m[0], attn_out, qd, plan.ntok,
                                static_cast<uint64_t>(qd) * 2, 64, kTileM)))
      return rc;
    for (int l = 1; l < kMaxCtxLayers; ++l) am.m[l] = am.m[0];
    if ((rc = make_tmap_2d_bf16(&bm.m[0], w_o, qd, H, static_cast<uint64_t>(qd) * 2, 64,
                                t.bn / 2)))
      return rc;
    bm.m[1] = bm.m[2] = bm.m[0];
    if ((rc = run_tile_gemm<OprojTileEpi>(t, am, bm, fp, st, plan.budget_sms))) return rc;
  } else {
    GemmCore g = gemm_shape(plan, qd, plan.o_tiles, 0, ws_at<uint32_t>(ws, plan.off_tickets_o),
                            ws_at<float>(ws, plan.off_acc_a), ws);
    sk::AMaps am;
    sk::BMaps bm;
    if ((rc = weight_map(&am.m[0], w_o, H, qd))) return rc;
    am.m[1] = am.m[2] = am.m[0];
    if ((rc = token_map(bm, attn_out, qd, plan.ntok, g.chunk_rows))) return rc;
    if ((rc = sk::run_streamk<OprojFin>(g, am, bm, fp, plan.budget_sms, st,
                                        plan.ffn_begin - plan.off_acc_a)))
      return rc;
  }
  if (plan.ntok >= kTiledDraftRows) {
    // 2. gate | up of the same features in one tile; silu(g) * u as hi/lo
    TileCore g = {};
    g.status = ws_at<uint32_t>(ws, plan.off_status);
    g.rows = plan.ntok;
    g.m_tiles = (plan.ntok + kTileM - 1) / kTileM;
    g.bn = 256;
    g.n_tiles = ffn / 128;
    g.k_tiles = 2 * H / 64;
    g.layer_cols = H;
    g.b_split = g.n_tiles;
    g.b_cols = H;
    g.b_paired = 1;
    TokenMaps am;
    WeightMaps bm;
    if ((rc = hilo_token_maps(am, fp.xhl, plan.ntok, H))) return rc;
    if ((rc = make_tmap_2d_bf16(&bm.m[0], w_gate, H, ffn, static_cast<uint64_t>(H) * 2, 64,
                                128)) ||
        (rc = make_tmap_2d_bf16(&bm.m[1], w_up, H, ffn, static_cast<uint64_t>(H) * 2, 64, 128)))
      return rc;
    bm.m[2] = bm.m[1];
    if ((rc = run_tile_gemm<GateUpTileEpi>(g, am, bm, fp, st, plan.budget_sms))) return rc;
    // 3. x2 = x1 + M W_down^T
    TileCore d = {};
    d.status = g.status;
    d.rows = plan.ntok;
    d.m_tiles = g.m_tiles;
    d.bn = H % 256 == 0 ? 256 : 128;
    d.n_tiles = H / d.bn;
    d.k_tiles = 2 * ffn / 64;
    d.layer_cols = ffn;
    d.b_split = d.n_tiles;
    d.b_cols = ffn;
    TokenMaps dm;
    WeightMaps wm;
    if ((rc = hilo_token_maps(dm, fp.mhl, plan.ntok, ffn))) return rc;
    if ((rc = make_tmap_2d_bf16(&wm.m[0], w_down, ffn, H, static_cast<uint64_t>(ffn) * 2, 64,
                                d.bn / 2)))
      return rc;
    wm.m[1] = wm.m[2] = wm.m[0];
    return run_tile_gemm<DownTileEpi>(d, dm, wm, fp, st, plan.budget_sms);
  }
  // 2. [gate; up] on hi/lo of x1 * ln2; paired finishing: silu(g) * u as hi/lo
  {
    GemmCore g = gemm_shape(plan, H, plan.gu_tiles, 1, ws_at<uint32_t>(ws, plan.off_tickets_gu),
                            ws_at<float>(ws, plan.off_acc_b), ws);
    g.a_split[0] = ffn / 128;
    g.a_split[1] = plan.gu_tiles;
    g.pair_stride = ffn / 128;
    sk::AMaps am;
    sk::BMaps bm;
    if ((rc = weight_map(&am.m[0], w_gate, ffn, H)) || (rc = weight_map(&am.m[1], w_up, ffn, H)))
      return rc;
    am.m[2] = am.m[1];
    if ((rc = token_map(bm, fp.xhl, H, 2 * plan.ntok, g.chunk_rows))) return rc;
    if ((rc = sk::run_streamk<GateUpFin>(g, am, bm, fp, plan.budget_sms, st,
                                         plan.total - plan.off_acc_b)))
      return rc;
  }
  // 3. x2 = x1 + M W_down^T
  {
    GemmCore g = gemm_shape(plan, ffn, plan.down_tiles, 1,
                            ws_at<uint32_t>(ws, plan.off_tickets_down),
                            ws_at<float>(ws, plan.off_acc_b), ws);
    sk::AMaps am;
    sk::BMaps bm;
    if ((rc = weight_map(&am.m[0], w_down, H, ffn))) return rc;
    am.m[1] = am.m[2] = am.m[0];
    if ((rc = token_map(bm, fp.mhl, ffn, 2 * plan.ntok, g.chunk_rows))) return rc;
    return sk::run_streamk<DownFin>(g, am, bm, fp, plan.budget_sms, st,
                                    plan.total - plan.off_acc_b);
  }
}
