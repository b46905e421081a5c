// a1 — context projection of the target's selected-layer hidden states into
// the drafter's context K/V cache.
//
// "DFlash双实现对比" (hotelren.com) §4: the hidden states of the layers in
// target_layer_ids are concatenated; §2: the drafter's context K/V are
// projected from them.  "dflash-mlx" (dpshk.com) 块扩散草稿 step 3: the
// drafter reads the target's multi-layer hidden states.
//
// Two launches on one stream of the stream-K GEMM of streamk_gemm.cuh (weights
// streamed once by every SM of the budget, fp32 sums in the workspace, the
// CTA that completes a tile's sum finishes it), with two finishers:
//  1. fc GEMM   Y = X W_fc^T.  X is never materialised: the k-loop reads
//     layer floor(k / H) through its own tensor map, which is the
//     concatenation.  Finisher: g_h * Y stored as a bf16 pair hi + lo
//     (exact to ~2^-17, so the next GEMM keeps Y's fp32 precision) and the
//     tile's partial sums of Y^2.  CTA 0 also snapshots the write positions,
//     maps the pages the block needs and sets seq_len = pos + 16.
//  2. K/V GEMM  [K;V] = [hi;lo] W_{k|v}^T.  Finisher: the RMSNorm scale of Y
//     (one factor per token row, so it commutes with the GEMM), per-head
//     RMSNorm and RoPE for K, bf16 store into the cache rows.
// The CTAs' partial sums of a tile are added in a fixed order, so the same
// inputs give the same cache bytes on every run (with the same SM budget).
#include "streamk_gemm.cuh"

namespace dflash {
namespace {

using sk::GemmCore;
using sk::take4;

// Parameters of both finishers.
struct ProjParams {
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

// Per sequence: snapshot the write position, map the pages that rows
// pos..pos+15 need (popping the free list), and set seq_len = pos + 16.
__device__ void reserve_block_rows(const ProjParams& p, uint32_t* status, int b) {
  const int pos = p.write_pos[b];
  p.pos_snapshot[b] = pos;
  const dflash_kv_view& v = p.cache;
  const int limit = v.page_table ? v.max_pages * v.page_size : v.capacity;
  if (pos < 0 || pos + kBlock > limit) {
    set_status(status, DFLASH_ST_CAPACITY);
    return;
  }
  if (v.page_table) map_rows(v, b, pos, kBlock, status);
  v.seq_len[b] = pos + kBlock;
}

constexpr int kTokGroup = 4;  // token rows a warp finishes together (loads in flight)
constexpr int kTiledProjectionRows = 257;  // from here on the tiled GEMMs project

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

// fc finisher (CTA that completed an output tile): Y = the accumulated sum;
// hi/lo bf16 pair of g_h * Y for the next GEMM; the tile's partial sums of Y^2
// per token row (the RMSNorm scale itself is applied after the K/V GEMM,
// since it is one factor per token row).  Warp w takes token rows w, w + 4,
// ...; a lane owns 4 consecutive features.
__device__ void finish_fc(const GemmCore& g, const ProjParams& p, int o, int c) {
  const int et = threadIdx.x - 64, warp = et >> 5, lane = et & 31;
  const int f0 = o * 128 + lane * 4;
  const float4 gn = p.hidden_norm_w ? load4_bf16(p.hidden_norm_w + f0) : make_float4(1.f, 1.f, 1.f, 1.f);
  const int t0 = c * g.chunk_rows;
  const int nt = min(g.chunk_rows, g.n_tok - t0);
#pragma unroll 1
  for (int j0 = warp * kTokGroup; j0 < nt; j0 += 4 * kTokGroup) {
    float4 y[kTokGroup];
#pragma unroll
    for (int k = 0; k < kTokGroup; ++k)
      if (j0 + k < nt) y[k] = take4(g, t0 + j0 + k, f0);
#pragma unroll
    for (int k = 0; k < kTokGroup; ++k) {
      if (j0 + k >= nt) break;
      const int tok = t0 + j0 + k;
      const float a[4] = {y[k].x * gn.x, y[k].y * gn.y, y[k].z * gn.z, y[k].w * gn.w};
      float hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        hi[e] = bf16_bits_to_float(float_to_bf16_bits(a[e]));
        lo[e] = a[e] - hi[e];
      }
      *reinterpret_cast<uint2*>(p.yhat + static_cast<size_t>(tok) * p.hidden + f0) =
          pack4_bf16(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint2*>(p.yhat + (static_cast<size_t>(g.n_tok) + tok) * p.hidden + f0) =
          pack4_bf16(lo[0], lo[1], lo[2], lo[3]);
      float sq = y[k].x * y[k].x + y[k].y * y[k].y + y[k].z * y[k].z + y[k].w * y[k].w;
#pragma unroll
      for (int off = 16; off; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if (lane == 0) p.ss[static_cast<size_t>(o) * g.n_tok + tok] = sq;
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
__device__ void finish_kv(const GemmCore& g, const ProjParams& p, int o, int c,
                          uint8_t* scratch) {
  const int et = threadIdx.x - 64, warp = et >> 5, lane = et & 31;
  const int D = p.head_dim;
  const bool is_k = o < g.a_split[0];
  const int feat0 = (is_k ? o : o - g.a_split[0]) * 128 + lane * 4;  // within Hkv * D
  const int head = feat0 / D, d0 = feat0 - head * D;
  const int t0 = c * g.chunk_rows;
  const int nt = min(g.chunk_rows, g.n_tok - t0);
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
          set_status(g.status, DFLASH_ST_PAGE_MISSING);
      } else {
        off = (static_cast<long long>(b) * p.n_kv_heads * cv.capacity + pos) * D;
      }
    }
    dst_off[j] = off;
    posb[j] = pos0 + t;
    float r = 1.f;
    if (p.hidden_norm_w) {
      float tot = 0.f;
      for (int q = 0; q < p.fc_out_tiles; ++q) tot += p.ss[static_cast<size_t>(q) * g.n_tok + tok];
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
      if (j0 + k < nt) v[k] = take4(g, t0 + j0 + k, o * 128 + lane * 4);
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

struct FcFin {
  using Params = ProjParams;
  // CTA 0 snapshots the write positions, maps the block's pages, sets lengths
  static __device__ void prologue(const GemmCore& g, const Params& p) {
    for (int b = threadIdx.x - 64; b < p.batch; b += 128) reserve_block_rows(p, g.status, b);
  }
  static __device__ void finish(const GemmCore& g, const Params& p, int o, int c, uint8_t*) {
    finish_fc(g, p, o, c);
  }
};

struct KvFin {
  using Params = ProjParams;
  static __device__ void prologue(const GemmCore&, const Params&) {}
  static __device__ void finish(const GemmCore& g, const Params& p, int o, int c,
                                uint8_t* scratch) {
    finish_kv(g, p, o, c, scratch);
  }
};

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" int dflash_ctx_project(const dflash_dims* dims, const void* const* layer_hidden,
                                  const void* w_fc, const void* hidden_norm_w, const void* w_k,
                                  const void* w_v, const void* k_norm_w,
                                  const int32_t* write_pos, const dflash_kv_view* cache,
                                  void* ws, size_t ws_bytes, dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_ctx_project");
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

  ProjParams fp = {};
  fp.hidden = H;
  fp.fc_out_tiles = plan.fc_out_tiles;
  fp.rms_eps = dims->rms_eps;
  fp.hidden_norm_w = static_cast<const uint16_t*>(hidden_norm_w);
  fp.yhat = yhat;
  fp.ss = ws_at<float>(ws, plan.off_ss);
  fp.batch = dims->batch;
  fp.write_pos = write_pos;
  fp.pos_snapshot = pos_snap;
  fp.cache = *cache;
  fp.n_kv_heads = dims->n_kv_heads;
  fp.head_dim = dims->head_dim;
  fp.k_norm_w = static_cast<const uint16_t*>(k_norm_w);
  fill_rope_table(fp.rope.hi, fp.rope.lo, dims->head_dim, dims->rope_theta);
  uint32_t* tickets = ws_at<uint32_t>(ws, plan.off_ctx_tickets);

  // Past 256 token rows (batch 17 and up) the projection is bound by the
  // tensor cores, not by the weight stream.  Confined to part of the device
  // (beside the verification) it runs on the tiled GEMMs of the prefill, 16
  // rows per sequence, with g_h Y kept as the same hi/lo bf16 pair (the two
  // halves in the hi and lo rows of this workspace region): at 512 rows and
  // 23 SMs they take the verify || projection phase from 765 to 525 us.  With
  // the whole device the streamed GEMMs stay faster (168 vs 209 us at 512
  // rows: the fc GEMM's 32 tile pairs leave most clusters idle).  Shapes the
  // tiles do not cover stay here too.
  if (ntok >= kTiledProjectionRows && plan.budget_sms < plan.num_sms &&
      aligned16(cache->k) && aligned16(cache->v) &&
      (!hidden_norm_w || aligned16(hidden_norm_w))) {
    rc = tiled_projection(*dims, kBlock, layer_hidden, w_fc, hidden_norm_w, w_k, w_v, k_norm_w,
                          write_pos, *cache, status, pos_snap, fp.ss, yhat,
                          yhat + static_cast<size_t>(ntok) * H, plan.budget_sms, st);
    if (rc != DFLASH_E_UNSUPPORTED) return rc;
  }

  // ---- 1. fc GEMM; its finisher writes hi/lo of g_h * Y and sums of Y^2 ----
  {
    GemmCore g = sk::gemm_dims(ntok, nL * H, plan.fc_out_tiles, 0);
    g.status = status;
    g.layer_cols = H;  // the k-loop moves to the next layer's map every H columns
    g.part = part_fc;
    g.tickets = tickets;
    sk::AMaps am;
    if ((rc = make_tmap_2d_bf16(&am.m[0], w_fc, static_cast<uint64_t>(nL) * H, H,
                                static_cast<uint64_t>(nL) * H * 2, 64, 128)))
      return rc;
    am.m[1] = am.m[2] = am.m[0];
    sk::BMaps bm;
    for (int l = 0; l < nL; ++l)
      if ((rc = make_tmap_2d_bf16(&bm.m[l], layer_hidden[l], H, ntok,
                                  static_cast<uint64_t>(H) * 2, 64, g.chunk_rows)))
        return rc;
    for (int l = nL; l < kMaxCtxLayers; ++l) bm.m[l] = bm.m[0];
    if ((rc = sk::run_streamk<FcFin>(g, am, bm, fp, plan.budget_sms, st,
                                     plan.off_yhat - plan.off_fc)))
      return rc;
  }
  // ---- 2. K/V GEMM on [hi; lo]; its finisher scales, normalises, rotates, stores ----
  {
    GemmCore g = sk::gemm_dims(ntok, H, plan.kv_out_tiles, 1);
    g.status = status;
    g.a_split[0] = plan.kv_out_tiles / 2;
    g.part = part_kv;
    g.tickets = tickets + plan.fc_out_tiles * plan.fc_tok_chunks;
    sk::AMaps am;
    if ((rc = make_tmap_2d_bf16(&am.m[0], w_k, H, kvd, static_cast<uint64_t>(H) * 2, 64, 128)))
      return rc;
    if ((rc = make_tmap_2d_bf16(&am.m[1], w_v, H, kvd, static_cast<uint64_t>(H) * 2, 64, 128)))
      return rc;
    am.m[2] = am.m[1];
    sk::BMaps bm;
    if ((rc = make_tmap_2d_bf16(&bm.m[0], yhat, H, 2 * static_cast<uint64_t>(ntok),
                                static_cast<uint64_t>(H) * 2, 64, g.chunk_rows)))
      return rc;
    for (int l = 1; l < kMaxCtxLayers; ++l) bm.m[l] = bm.m[0];
    if ((rc = sk::run_streamk<KvFin>(g, am, bm, fp, plan.budget_sms, st,
                                     plan.off_att_o - plan.off_kv)))
      return rc;
  }
  return DFLASH_OK;
}
