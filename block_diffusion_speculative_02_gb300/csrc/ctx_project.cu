// a1 — context projection of the target's selected-layer hidden states into
// the drafter's context K/V cache.
//
// "DFlash双实现对比" (hotelren.com) §4: the hidden states of the layers in
// target_layer_ids are concatenated; §2: the drafter's context K/V are
// projected from them.  "dflash-mlx" (dpshk.com) 块扩散草稿 step 3: the
// drafter reads the target's multi-layer hidden states.
//
// Pipeline of four kernels on one stream:
//  1. fc GEMM   Y_part[s] = X[:, k-split s] W_fc[:, k-split s]^T   (split-K)
//     X is never materialised: the k-loop reads layer floor(k / H) through its
//     own tensor map, which is the concatenation.
//  2. reduce    Y = sum_s Y_part[s] (fp32), Y^ = RMSNorm(Y) * g_h, stored as a
//     bf16 pair hi + lo (Y^ ~= hi + lo to ~2^-17) so that the next GEMM does not
//     lose the fp32 precision of Y^; also snapshots the write positions,
//     reserves pages of a paged cache and sets seq_len = pos + 16.
//  3. kv GEMM   [K;V]_part[s] = [hi;lo] W_{k|v}^T                (split-K)
//  4. finish    sum splits and hi+lo, per-head RMSNorm of K, RoPE at the row
//     positions, bf16 store into the cache rows.
// Both GEMMs are "swap-AB" on the 5th-generation tensor cores: 128 output
// features are the MMA's M, the token rows its N, accumulators in TMEM, the
// weight stream staged by a TMA pipeline; they are memory-bound at small
// batch, so the grid is split along K until every SM streams weights.
#include "common.cuh"
#include "host.h"

namespace dflash {
namespace {

constexpr int kGemmThreads = 192;
constexpr int kATile = 128 * 128;  // 128 rows x 64 bf16
constexpr int kGemmSmemBudget = 110 * 1024;  // two CTAs per SM
constexpr int kMaxGemmStages = 8;

struct LayerMaps {
  CUtensorMap m[kMaxCtxLayers];
};

struct GemmParams {
  int k_tiles;       // K / 64
  int splits;
  int out_tiles;     // output features / 128
  int a_split;       // tiles >= a_split read the second weight map
  int layer_cols;    // columns per B map (fc: H); k-tile kt reads map (kt*64)/layer_cols
  int n_tok;
  int chunk_rows;    // token rows per chunk (B box rows)
  int n_chunks;
  int hilo;          // 1: B = [hi rows ; lo rows] of a 2*n_tok-row matrix, summed in the epilogue
  int ld_out;        // features per output row
  int mma_n;         // MMA N = chunk_rows * (1 + hilo)
  int n_stages, stage_bytes, tmem_cols;
  float* part;       // [splits][n_tok][ld_out]
  uint32_t* status;
};

__global__ void __launch_bounds__(kGemmThreads)
splitk_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0,
                   const __grid_constant__ CUtensorMap tm_a1,
                   const __grid_constant__ LayerMaps tm_b, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.n_stages * p.stage_bytes);
  uint64_t* empty = full + p.n_stages;
  uint64_t* tfull = empty + p.n_stages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  int unit = blockIdx.x;
  const int o = unit % p.out_tiles;
  unit /= p.out_tiles;
  const int s = unit % p.splits;
  const int c = unit / p.splits;
  const int kt0 = static_cast<int>(static_cast<long long>(s) * p.k_tiles / p.splits);
  const int kt1 = static_cast<int>(static_cast<long long>(s + 1) * p.k_tiles / p.splits);

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.n_stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
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
      const CUtensorMap* ma = o < p.a_split ? &tm_a0 : &tm_a1;
      const int arow = (o < p.a_split ? o : o - p.a_split) * 128;
      const uint32_t bytes = kATile + (1 + p.hilo) * p.chunk_rows * 128;
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      for (int kt = kt0; kt < kt1; ++kt) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) break;
        uint8_t* a = smem + stage * p.stage_bytes;
        uint8_t* bt = a + kATile;
        mbar_arrive_expect_tx(&full[stage], bytes);
        tma_load_2d(a, ma, &full[stage], kt * 64, arow, pol_w);
        const int l = (kt * 64) / p.layer_cols;
        const int col = kt * 64 - l * p.layer_cols;
        tma_load_2d(bt, &tm_b.m[l], &full[stage], col, c * p.chunk_rows, pol_x);
        if (p.hilo)
          tma_load_2d(bt + p.chunk_rows * 128, &tm_b.m[l], &full[stage], col,
                      p.n_tok + c * p.chunk_rows, pol_x);
        ++issued;
        if (++stage == static_cast<uint32_t>(p.n_stages)) {
          stage = 0;
          phase ^= 1;
        }
      }
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
      bool first = true;
      for (int kt = kt0; kt < kt1; ++kt) {
        if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t a_addr = base + stage * p.stage_bytes;
        const uint64_t adesc = umma_sdesc_sw128(a_addr);
        const uint64_t bdesc = umma_sdesc_sw128(a_addr + kATile);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          umma_bf16(tmem_base, adesc + 2 * kk, bdesc + 2 * kk, idesc, first ? 0u : 1u);
          first = false;
        }
        umma_commit(&empty[stage]);
        if (++stage == static_cast<uint32_t>(p.n_stages)) {
          stage = 0;
          phase ^= 1;
        }
      }
      umma_commit(tfull);  // also the drain point for the MMAs
      mbar_wait_drain(tfull, 0, p.status);
    }
  } else {
    // epilogue: TMEM lane = output feature, column = token (hi, then lo)
    const int q = warp & 3;
    const bool ok = mbar_wait(tfull, 0, abort_flag, p.status);
    if (__all_sync(0xffffffffu, ok) && kt1 > kt0) {
      tc_fence_after();
      const int f = o * 128 + q * 32 + lane;
      const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
      float* dst = p.part + static_cast<size_t>(s) * p.n_tok * p.ld_out + f;
      for (int c0 = 0; c0 < p.chunk_rows; c0 += 16) {
        uint32_t v[16], w[16];
        tmem_ld_32x32b_x16(tmem_base + lane_base + c0, v);
        if (p.hilo) tmem_ld_32x32b_x16(tmem_base + lane_base + p.chunk_rows + c0, w);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = c * p.chunk_rows + c0 + j;
          float val = __uint_as_float(v[j]);
          if (p.hilo) val += __uint_as_float(w[j]);
          if (tok < p.n_tok) dst[static_cast<size_t>(tok) * p.ld_out] = val;
        }
      }
      tc_fence_before();
    }
  }
  __syncthreads();
  griddep_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// ---------------------------------------------------------------------------
struct ReduceParams {
  int n_tok, hidden, splits, batch;
  float rms_eps;
  const float* part;            // [splits][n_tok][hidden]
  const uint16_t* norm_w;       // [hidden] or null
  uint16_t* yhat;               // [2][n_tok][hidden]  (hi, lo)
  const int32_t* write_pos;     // [batch]
  int32_t* pos_snapshot;        // [batch]
  dflash_kv_view cache;
  uint32_t* status;
};

__global__ void __launch_bounds__(256) fc_reduce_norm_kernel(const ReduceParams p) {
  griddep_wait();
  const int row = blockIdx.x;
  __shared__ float red[8];
  if (row == 0) {
    // bookkeeping, one thread per sequence: positions, page reservation, length
    for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
      const int pos = p.write_pos[b];
      p.pos_snapshot[b] = pos;
      const dflash_kv_view& v = p.cache;
      const int limit = v.page_table ? v.max_pages * v.page_size : v.capacity;
      if (pos < 0 || pos + kBlock > limit) {
        set_status(p.status, DFLASH_ST_CAPACITY);
        continue;
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
  }
  const int H = p.hidden;
  float ss = 0.f;
  for (int f = threadIdx.x; f < H; f += blockDim.x) {
    float y = 0.f;
    for (int s = 0; s < p.splits; ++s) y += p.part[(static_cast<size_t>(s) * p.n_tok + row) * H + f];
    ss += y * y;
  }
  float rs = 1.f;
  if (p.norm_w) {
#pragma unroll
    for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) tot += red[i];
    rs = rsqrtf(tot / H + p.rms_eps);
  }
  uint16_t* hi = p.yhat + static_cast<size_t>(row) * H;
  uint16_t* lo = p.yhat + (static_cast<size_t>(p.n_tok) + row) * H;
  for (int f = threadIdx.x; f < H; f += blockDim.x) {
    float y = 0.f;
    for (int s = 0; s < p.splits; ++s) y += p.part[(static_cast<size_t>(s) * p.n_tok + row) * H + f];
    if (p.norm_w) y = y * rs * bf16_bits_to_float(p.norm_w[f]);
    const uint16_t h = float_to_bf16_bits(y);
    hi[f] = h;
    lo[f] = float_to_bf16_bits(y - bf16_bits_to_float(h));
  }
  griddep_launch_dependents();
}

// ---------------------------------------------------------------------------
struct FinishParams {
  int n_tok, n_kv_heads, head_dim, splits, ld;   // ld = 2 * Hkv * D
  float rms_eps;
  const float* part;          // [splits][n_tok][ld]: K features then V features
  const uint16_t* k_norm_w;   // [D] or null
  const int32_t* pos_snapshot;
  dflash_kv_view cache;
  uint32_t* status;
  RopeTable rope;
};

// One CTA per (token row, KV head); thread d owns feature d of the head.
__global__ void __launch_bounds__(128) kv_finish_kernel(const FinishParams p) {
  griddep_wait();
  const int row = blockIdx.x, g = blockIdx.y, d = threadIdx.x;
  const int D = p.head_dim;
  const int b = row / kBlock, t = row - b * kBlock;
  __shared__ float kbuf[128];
  __shared__ float red[4];
  float k = 0.f, v = 0.f;
  for (int s = 0; s < p.splits; ++s) {
    const float* src = p.part + (static_cast<size_t>(s) * p.n_tok + row) * p.ld;
    k += src[g * D + d];
    v += src[p.n_kv_heads * D + g * D + d];
  }
  if (p.k_norm_w) {
    float ss = k * k;
#pragma unroll
    for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((d & 31) == 0) red[d >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int i = 0; i < D / 32; ++i) tot += red[i];
    k = k * rsqrtf(tot / D + p.rms_eps) * bf16_bits_to_float(p.k_norm_w[d]);
  }
  kbuf[d] = k;
  __syncthreads();
  const int pos = p.pos_snapshot[b] + t;
  const int half = D / 2;
  const int fi = d < half ? d : d - half;
  float sn, cs;
  sincosf(rope_angle(pos, p.rope.hi[fi], p.rope.lo[fi]), &sn, &cs);
  const float kr = d < half ? k * cs - kbuf[d + half] * sn : k * cs + kbuf[d - half] * sn;
  griddep_launch_dependents();

  const dflash_kv_view& c = p.cache;
  const int limit = c.page_table ? c.max_pages * c.page_size : c.capacity;
  if (p.pos_snapshot[b] < 0 || p.pos_snapshot[b] + kBlock > limit) return;  // flagged earlier
  size_t rowidx;
  if (c.page_table) {
    const int page = c.page_table[static_cast<size_t>(b) * c.max_pages + pos / c.page_size];
    if (page < 0) {
      if (d == 0) set_status(p.status, DFLASH_ST_PAGE_MISSING);
      return;
    }
    rowidx = static_cast<size_t>(page) * c.page_size + pos % c.page_size;
  } else {
    rowidx = static_cast<size_t>(b) * c.capacity + pos;
  }
  const size_t off = (rowidx * p.n_kv_heads + g) * D + d;
  static_cast<uint16_t*>(c.k)[off] = float_to_bf16_bits(kr);
  static_cast<uint16_t*>(c.v)[off] = float_to_bf16_bits(v);
}

int gemm_smem(int stage_bytes, int n_stages) {
  return 1024 + n_stages * (stage_bytes + 16) + 8 + 16;
}

int setup_gemm(GemmParams& g, int b_rows_per_stage) {
  g.stage_bytes = kATile + ((b_rows_per_stage * 128 + 1023) / 1024) * 1024;
  g.n_stages = (kGemmSmemBudget - 1024 - 24) / (g.stage_bytes + 16);
  if (g.n_stages > kMaxGemmStages) g.n_stages = kMaxGemmStages;
  if (g.n_stages < 2) {
    g.n_stages = 2;  // large token chunks: one CTA per SM
  }
  int cols = 32;
  while (cols < g.mma_n) cols *= 2;
  g.tmem_cols = cols;
  return gemm_smem(g.stage_bytes, g.n_stages);
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

  // ---- 1. fc GEMM ----
  {
    GemmParams g = {};
    g.k_tiles = plan.fc_k_tiles;
    g.splits = plan.fc_splits;
    g.out_tiles = plan.fc_out_tiles;
    g.a_split = plan.fc_out_tiles;
    g.layer_cols = H;
    g.n_tok = ntok;
    g.chunk_rows = ntok < 256 ? ntok : 256;
    g.n_chunks = plan.fc_tok_chunks;
    g.hilo = 0;
    g.ld_out = H;
    g.mma_n = g.chunk_rows;
    g.part = part_fc;
    g.status = status;
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
    if ((rc = set_smem_limit(reinterpret_cast<const void*>(splitk_gemm_kernel), smem))) return rc;
    const int grid = g.out_tiles * g.splits * g.n_chunks;
    if ((rc = launch(splitk_gemm_kernel, dim3(grid), dim3(kGemmThreads), smem, st, ta, ta, lm, g)))
      return rc;
  }
  // ---- 2. reduce + RMSNorm + hi/lo split; positions and pages ----
  {
    ReduceParams r = {};
    r.n_tok = ntok;
    r.hidden = H;
    r.splits = plan.fc_splits;
    r.batch = dims->batch;
    r.rms_eps = dims->rms_eps;
    r.part = part_fc;
    r.norm_w = static_cast<const uint16_t*>(hidden_norm_w);
    r.yhat = yhat;
    r.write_pos = write_pos;
    r.pos_snapshot = pos_snap;
    r.cache = *cache;
    r.status = status;
    if ((rc = launch(fc_reduce_norm_kernel, dim3(ntok), dim3(256), 0, st, r))) return rc;
  }
  // ---- 3. kv GEMM on [hi; lo] ----
  {
    GemmParams g = {};
    g.k_tiles = plan.kv_k_tiles;
    g.splits = plan.kv_splits;
    g.out_tiles = plan.kv_out_tiles;
    g.a_split = plan.kv_out_tiles / 2;
    g.layer_cols = H;
    g.n_tok = ntok;
    g.chunk_rows = ntok < 128 ? ntok : 128;
    g.n_chunks = plan.kv_tok_chunks;
    g.hilo = 1;
    g.ld_out = 2 * kvd;
    g.mma_n = 2 * g.chunk_rows;
    g.part = part_kv;
    g.status = status;
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
    if ((rc = set_smem_limit(reinterpret_cast<const void*>(splitk_gemm_kernel), smem))) return rc;
    const int grid = g.out_tiles * g.splits * g.n_chunks;
    if ((rc = launch(splitk_gemm_kernel, dim3(grid), dim3(kGemmThreads), smem, st, tk, tv, lm, g)))
      return rc;
  }
  // ---- 4. finish: reduce, k_norm, RoPE, store ----
  {
    FinishParams f = {};
    f.n_tok = ntok;
    f.n_kv_heads = dims->n_kv_heads;
    f.head_dim = dims->head_dim;
    f.splits = plan.kv_splits;
    f.ld = 2 * kvd;
    f.rms_eps = dims->rms_eps;
    f.part = part_kv;
    f.k_norm_w = static_cast<const uint16_t*>(k_norm_w);
    f.pos_snapshot = pos_snap;
    f.cache = *cache;
    f.status = status;
    fill_rope_table(f.rope.hi, f.rope.lo, dims->head_dim, dims->rope_theta);
    if ((rc = launch(kv_finish_kernel, dim3(ntok, dims->n_kv_heads), dim3(dims->head_dim), 0, st,
                     f)))
      return rc;
  }
  return DFLASH_OK;
}
