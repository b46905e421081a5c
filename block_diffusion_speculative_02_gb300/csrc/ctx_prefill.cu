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
// weight stream, so they run on the tiled GEMM of tile_gemm.cuh (persistent
// clusters of two CTAs over 128 x BN output tiles, the pair reading each
// weight box once from DRAM and once from L2, TMEM lane = token row) rather
// than on the stream-K one; the row-wise work of the epilogues (sums of
// squares, head norms, the RoPE partner at d + D/2) stays inside one thread.
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
#include "tile_gemm.cuh"

namespace dflash {
namespace {

struct PrefillParams {
  int hidden, fc_n_tiles, tokens_per_seq, batch;
  float rms_eps;
  const uint16_t* hidden_norm_w;  // [H] or null
  uint16_t* yhat;                 // [rows][H]: bf16(g_h * Y)
  uint16_t* yhat_lo;              // [rows][H]: bf16(g_h * Y - yhat), or null (not kept)
  float* ss;                      // [fc_n_tiles][rows]: partial sums of Y^2
  const int32_t* write_pos;
  int32_t* pos_snapshot;          // [B]; -1: the sequence's rows are skipped
  dflash_kv_view cache;
  int n_kv_heads, head_dim;
  const uint16_t* k_norm_w;       // [D] or null
  RopeTable rope;
};

__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  return static_cast<uint32_t>(float_to_bf16_bits(a)) |
         (static_cast<uint32_t>(float_to_bf16_bits(b)) << 16);
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
  using Params = PrefillParams;
  static __device__ void setup(const PrefillParams&, float*, int) {}
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
      uint32_t out[8], lo[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float y0 = __uint_as_float(v[2 * j]), y1 = __uint_as_float(v[2 * j + 1]);
        ss = fmaf(y0, y0, fmaf(y1, y1, ss));
        const float a0 = y0 * g[2 * j], a1 = y1 * g[2 * j + 1];
        out[j] = pack2_bf16(a0, a1);
        lo[j] = pack2_bf16(a0 - __uint_as_float(out[j] << 16),
                           a1 - __uint_as_float(out[j] & 0xFFFF0000u));
      }
      if (live) {
        uint4* d = reinterpret_cast<uint4*>(dst + c0);
        d[0] = make_uint4(out[0], out[1], out[2], out[3]);
        d[1] = make_uint4(out[4], out[5], out[6], out[7]);
        if (e.yhat_lo) {
          uint4* dl = reinterpret_cast<uint4*>(e.yhat_lo + (dst - e.yhat) + c0);
          dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        }
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
  using Params = PrefillParams;
  // the RoPE table (hi[64], lo[64]) into shared memory
  static __device__ void setup(const PrefillParams& e, float* tab, int i) {
    if (i < 64) {
      tab[i] = e.rope.hi[i];
      tab[64 + i] = e.rope.lo[i];
    }
  }
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


}  // namespace
}  // namespace dflash

namespace dflash {

// The two tiled GEMMs of the projection for tokens_per_seq rows per sequence
// (arguments checked by the caller; the scratch pointers are regions of the
// caller's workspace).  Also used by dflash_ctx_project when its batch makes
// the projection tensor-bound, with the lo half of g_h Y kept.
int tiled_projection(const dflash_dims& d, int tokens_per_seq, const void* const* layer_hidden,
                     const void* w_fc, const void* hidden_norm_w, const void* w_k,
                     const void* w_v, const void* k_norm_w, const int32_t* write_pos,
                     const dflash_kv_view& cache_view, uint32_t* status, int32_t* pos_snapshot,
                     float* ss, uint16_t* yhat, uint16_t* yhat_lo, int max_ctas,
                     cudaStream_t st) {
  PrefillPlan plan;
  int rc = make_prefill_plan(d, tokens_per_seq, &plan);
  if (rc) return rc;
  const dflash_dims* dims = &d;
  const dflash_kv_view* cache = &cache_view;
  const int nL = d.n_ctx_layers, H = d.hidden;
  const int kvd = d.n_kv_heads * d.head_dim;
  const uint64_t rows = static_cast<uint64_t>(plan.rows);
  PrefillParams ep = {};
  ep.hidden = H;
  ep.fc_n_tiles = plan.fc_n_tiles;
  ep.tokens_per_seq = tokens_per_seq;
  ep.batch = dims->batch;
  ep.rms_eps = dims->rms_eps;
  ep.hidden_norm_w = static_cast<const uint16_t*>(hidden_norm_w);
  ep.yhat = yhat;
  ep.yhat_lo = yhat_lo;
  ep.ss = ss;
  ep.write_pos = write_pos;
  ep.pos_snapshot = pos_snapshot;
  ep.cache = *cache;
  ep.n_kv_heads = dims->n_kv_heads;
  ep.head_dim = dims->head_dim;
  ep.k_norm_w = static_cast<const uint16_t*>(k_norm_w);
  fill_rope_table(ep.rope.hi, ep.rope.lo, dims->head_dim, dims->rope_theta);

  // ---- 1. fc GEMM: bf16(g_h * Y) and sums of Y^2 ----
  {
    TileCore g = {};
    g.status = status;
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
    bm.m[1] = bm.m[2] = bm.m[0];
    if ((rc = run_tile_gemm<FcEpi>(g, am, bm, ep, st, max_ctas))) return rc;
  }
  // ---- 2. K/V GEMM: row factor, head norm + RoPE for K, cache stores ----
  {
    TileCore g = {};
    g.status = status;
    g.rows = plan.rows;
    g.m_tiles = (plan.rows + kTileM - 1) / kTileM;
    g.bn = plan.kv_bn;
    g.n_tiles = 2 * kvd / g.bn;
    // with the lo half kept, K runs twice over the weights: bf16(g_h Y) and
    // then its rounding remainder, summed in the accumulator
    g.k_tiles = (yhat_lo ? 2 : 1) * H / 64;
    g.layer_cols = H;
    g.b_split = kvd / g.bn;
    g.b_cols = H;
    TokenMaps am;
    if ((rc = make_tmap_2d_bf16(&am.m[0], yhat, H, rows, static_cast<uint64_t>(H) * 2, 64,
                                kTileM)))
      return rc;
    for (int l = 1; l < kMaxCtxLayers; ++l) am.m[l] = am.m[0];
    if (yhat_lo && (rc = make_tmap_2d_bf16(&am.m[1], yhat_lo, H, rows,
                                           static_cast<uint64_t>(H) * 2, 64, kTileM)))
      return rc;
    WeightMaps bm;
    if ((rc = make_tmap_2d_bf16(&bm.m[0], w_k, H, kvd, static_cast<uint64_t>(H) * 2, 64,
                                g.bn / 2)))
      return rc;
    if ((rc = make_tmap_2d_bf16(&bm.m[1], w_v, H, kvd, static_cast<uint64_t>(H) * 2, 64,
                                g.bn / 2)))
      return rc;
    bm.m[2] = bm.m[1];
    if ((rc = run_tile_gemm<KvEpi>(g, am, bm, ep, st, max_ctas))) return rc;
  }
  return DFLASH_OK;
}

}  // namespace dflash

using namespace dflash;

extern "C" size_t dflash_prefill_workspace_bytes(const dflash_dims* dims, int32_t tokens_per_seq) {
  if (!dims) return 0;
  PrefillPlan p;
  if (make_prefill_plan(*dims, tokens_per_seq, &p)) return 0;
  // one workspace serves both prefill calls (status word at offset 0 in both)
  const size_t att = prefill_attention_workspace(*dims, tokens_per_seq);
  if (att == 0) return 0;
  return att > p.total ? att : p.total;
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
  const int nL = dims->n_ctx_layers;
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
  return tiled_projection(*dims, tokens_per_seq, layer_hidden, w_fc, hidden_norm_w, w_k, w_v,
                          k_norm_w, write_pos, *cache, ws_at<uint32_t>(ws, plan.off_status),
                          ws_at<int32_t>(ws, plan.off_pos), ws_at<float>(ws, plan.off_ss),
                          ws_at<uint16_t>(ws, plan.off_yhat), nullptr, 0,
                          reinterpret_cast<cudaStream_t>(stream));
}
