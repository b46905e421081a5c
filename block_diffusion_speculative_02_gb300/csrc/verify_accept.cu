// a3 — verification epilogue: LM-head GEMM with fused greedy argmax, then
// acceptance + commit, in one persistent kernel.
//
// "dflash-mlx" lossless speculative decoding (dpshk.com), 单次前向验证 ⑤–⑧ and
// 保证一/保证二: every verify position takes the target's greedy argmax
// (posterior); acceptance = sum(cumprod(draft == posterior)); 1 + a tokens are
// committed and the target's token at the first rejected position is the
// next staged token.
//
// Design (GB300): the LM head is a skinny GEMM (16*B token rows against V
// vocabulary rows) that streams W_lm from HBM exactly once.  It is computed
// "swap-AB" on the 5th-generation tensor cores: a vocabulary tile of 128 rows
// is the MMA's M, the token rows are its N, so the fp32 accumulator
// [128 vocab x ntok] lives in TMEM.  Each CTA owns one contiguous vocabulary
// range (balanced to 8 rows), streamed through a deep TMA pipeline of
// 128-row x 64-col swizzled tiles.  The epilogue reduces every token column
// over the tile's 128 rows with one redux.sync + ballot per column and keeps a
// 64-bit key (order-preserving fp32 bits << 32 | ~row) per token in shared
// memory, so logits never leave the SM.  The last CTA to finish (atomic
// ticket, no waiting) turns the keys into the posterior and runs the
// acceptance and the commit.
//
// Warp roles (192 threads): warp 0 issues TMA, warp 1 owns TMEM and issues the
// MMAs, warps 2-5 drain the accumulators.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "host.h"
#include "tile_gemm.cuh"

namespace dflash {
namespace {

constexpr int kThreads = 192;
constexpr int kTileRows = 128;           // vocabulary rows per MMA (M)
constexpr int kATileBytes = kTileRows * 128;
#ifndef DFLASH_LM_UNIT_ROWS
#define DFLASH_LM_UNIT_ROWS 8
#endif
constexpr int kUnitRows = DFLASH_LM_UNIT_ROWS;  // balancing granule of the vocabulary split (8..128)

// Tensor maps over W_lm with boxes of 64, 32, 16 and 8 rows: a CTA's last,
// partial tile (its range is balanced to 8 rows) is loaded as at most four
// boxes -- one per set bit of its row count -- instead of one per 8 rows.
struct PartialMaps {
  CUtensorMap m[4];
};
constexpr int kSmemBudget = 224 * 1024;
constexpr int kMaxStages = 12;
#ifndef DFLASH_LM_CHUNKS_PER_STAGE
#define DFLASH_LM_CHUNKS_PER_STAGE 4
#endif
constexpr int kLmChunksPerStage = DFLASH_LM_CHUNKS_PER_STAGE;  // power of two
#ifndef DFLASH_LM_MIN_STAGES
#define DFLASH_LM_MIN_STAGES 2
#endif
constexpr int kLmMinStages = DFLASH_LM_MIN_STAGES;

struct LmParams {
  int vocab, hidden, ntok;
  int ntok_box, n_xbox;                  // token rows per X box, X boxes per 64-col chunk
  int kb;                                // 64-column K chunks per pipeline stage
  int x_chunk;                           // bytes of the token tile of one chunk
  int n_units;                           // ceil(vocab / 8)
  int n_stages, stage_bytes;
  int n_acc, tmem_cols;
  unsigned long long* keys;              // [ntok] workspace, zero between calls
  uint32_t* ticket;
  uint32_t* status;
  int batch;
  const int32_t* block_ids;
  const int32_t* len_before;
  int32_t* posterior;
  int32_t* accept_len;
  int32_t* next_staged;
  int32_t* commit_len;
  int32_t* out_tokens;
  int out_cap;
  // drafting (dflash_draft_tokens, draft = 1): the argmaxes become the next
  // block instead of being checked against one; the prefill's staged token
  // (dflash_prefill_staged, draft = 2): one row per sequence, its argmax
  int draft;
  const int32_t* staged;                 // [B] token for block position 0, or null
  int32_t* block_out;                    // [B, 16]
};

__device__ __forceinline__ void accept_and_commit(const LmParams& p, int b) {
  int post[kBlock], blk[kBlock];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kBlock; ++i) {
    const unsigned long long k = __ldcg(&p.keys[b * kBlock + i]);
    post[i] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
    blk[i] = p.block_ids[b * kBlock + i];
    bad |= (blk[i] < 0 || blk[i] >= p.vocab);
  }
  // a = sum(cumprod(block[1:] == posterior[:15]))
  int a = 0;
  bool run = true;
#pragma unroll
  for (int i = 0; i < kBlock - 1; ++i) {
    run = run && (blk[i + 1] == post[i]);
    a += run ? 1 : 0;
  }
#pragma unroll
  for (int i = 0; i < kBlock; ++i) p.posterior[b * kBlock + i] = post[i];
  p.accept_len[b] = a;
  if (bad) set_status(p.status, DFLASH_ST_BAD_TOKEN);
  const int lb = p.len_before[b];
  if (lb < 0 || lb + 1 + a > p.out_cap) {
    set_status(p.status, DFLASH_ST_OUT_OVERFLOW);
    return;
  }
  int32_t* dst = p.out_tokens + static_cast<size_t>(b) * p.out_cap + lb;
  int staged = post[0];
#pragma unroll
  for (int i = 0; i < kBlock; ++i) {
    if (i <= a) dst[i] = blk[i];
    if (i == a) staged = post[i];
  }
  p.next_staged[b] = staged;
  p.commit_len[b] = lb + 1 + a;
}

// Drafting: every mask position's argmax is its drafted token ("dflash-mlx"
// 块扩散草稿 step 2); position 0 takes the staged token.
__device__ __forceinline__ void write_draft(const LmParams& p, int b) {
#pragma unroll
  for (int i = 0; i < kBlock; ++i) {
    const unsigned long long k = __ldcg(&p.keys[b * kBlock + i]);
    const int t = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
    if (p.posterior) p.posterior[b * kBlock + i] = t;
    if (i > 0) p.block_out[b * kBlock + i] = t;
  }
  if (p.staged) p.block_out[b * kBlock] = p.staged[b];
}

// The prefill's staged token ("dflash-mlx" 单次前向验证 ②): the argmax of
// sequence b's single row.
__device__ __forceinline__ void write_staged(const LmParams& p, int b) {
  const unsigned long long k = __ldcg(&p.keys[b]);
  p.block_out[b] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
}

__device__ __forceinline__ void finish_sequence(const LmParams& p, int b) {
  if (p.draft == 2)
    write_staged(p, b);
  else if (p.draft)
    write_draft(p, b);
  else
    accept_and_commit(p, b);
}

__global__ void __launch_bounds__(kThreads, 1)
lmhead_argmax_accept_kernel(const __grid_constant__ CUtensorMap tm_w,
                            const __grid_constant__ PartialMaps tm_part,
                            const __grid_constant__ CUtensorMap tm_x, const LmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.n_stages * p.stage_bytes);
  uint64_t* empty = full + p.n_stages;
  uint64_t* tfull = empty + p.n_stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  unsigned long long* best = reinterpret_cast<unsigned long long*>(tmem_slot + 4);

  // this CTA's vocabulary rows [r0, r1)
  const int u0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.n_units / gridDim.x);
  const int u1 =
      static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.n_units / gridDim.x);
  const int r0 = u0 * kUnitRows;
  const int r1 = min(u1 * kUnitRows, p.vocab);
  const int n_tiles = (r1 - r0 + kTileRows - 1) / kTileRows;
  const int k_stages = p.hidden / 64 / p.kb;
  const int a_stage = p.kb * kATileBytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.n_stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < p.ntok; i += kThreads) best[i] = 0ull;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // the hidden states may be produced by the previous kernel on the stream
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
#ifdef DFLASH_LM_W_EVICT_NORMAL
      const uint64_t pol_w = l2_policy_evict_normal();
#else
      const uint64_t pol_w = l2_policy_evict_first();
#endif
      const uint64_t pol_x = l2_policy_evict_last();
      const uint32_t x_bytes = static_cast<uint32_t>(p.n_xbox * p.ntok_box * 128);
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      // Every CTA walks the hidden dimension starting at its own k-stage: CTAs
      // that stream in lockstep at the same column offset of their rows hit
      // the same DRAM channels (measured: 7 % slower); rotated starts spread
      // the requests.  The accumulation order only changes fp32 rounding.
      const int k_rot = blockIdx.x % k_stages;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int row0 = r0 + t * kTileRows;
        const int rows = min(kTileRows, r1 - row0);
        const int rows8 = (rows + 7) & ~7;    // boxes past the vocabulary are zero-filled
        const uint32_t a_bytes = static_cast<uint32_t>(rows8) * 128;
        for (int ks = 0; ks < k_stages; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          uint8_t* a = smem + stage * p.stage_bytes;
          uint8_t* b = a + a_stage;
          mbar_arrive_expect_tx(&full[stage], p.kb * (a_bytes + x_bytes));
          // the kb chunks of one stage are issued back to back, so every
          // vocabulary row is requested as kb*128 contiguous bytes at once
          const int ksr = ks + k_rot < k_stages ? ks + k_rot : ks + k_rot - k_stages;
          for (int j = 0; j < p.kb; ++j) {
            const int kcol = (ksr * p.kb + j) * 64;
            uint8_t* aj = a + j * kATileBytes;
            if (rows == kTileRows) {
              tma_load_2d(aj, &tm_w, &full[stage], kcol, row0, pol_w);
            } else {
              int off = 0;
              for (int bi = 0; bi < 4; ++bi) {
                const int br = 64 >> bi;
                if (rows8 & br) {
                  tma_load_2d(aj + off * 128, &tm_part.m[bi], &full[stage], kcol, row0 + off,
                              pol_w);
                  off += br;
                }
              }
            }
            for (int c = 0; c < p.n_xbox; ++c)
              tma_load_2d(b + j * p.x_chunk + c * p.ntok_box * 128, &tm_x, &full[stage], kcol,
                          c * p.ntok_box, pol_x);
          }
          ++issued;
          if (++stage == static_cast<uint32_t>(p.n_stages)) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) {
        // let every copy still in flight land before the CTA can exit
        for (int s = 0; s < p.n_stages && s < issued; ++s) {
          const int last = s + ((issued - 1 - s) / p.n_stages) * p.n_stages;
          mbar_wait_drain(&full[s], static_cast<uint32_t>((last / p.n_stages) & 1), p.status);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t smem_base = smem_u32(smem);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int acc = t % p.n_acc;
        const uint32_t acc_phase = static_cast<uint32_t>((t / p.n_acc) & 1);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_base = tmem_base + static_cast<uint32_t>(acc * p.ntok);
        for (int ks = 0; ks < k_stages; ++ks) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_base + stage * p.stage_bytes;
          const uint32_t b_addr = a_addr + a_stage;
          for (int j = 0; j < p.kb; ++j) {
            const uint64_t adesc = umma_sdesc_sw128(a_addr + j * kATileBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              for (int c = 0; c * 256 < p.ntok; ++c) {
                const int n = min(256, p.ntok - c * 256);
                const uint64_t bdesc = umma_sdesc_sw128(b_addr + j * p.x_chunk + c * 256 * 128);
                umma_bf16(d_base + c * 256, adesc + 2 * kk, bdesc + 2 * kk,
                          umma_idesc_bf16(kTileRows, n), (ks | j | kk) != 0);
              }
            }
          }
          umma_commit(&empty[stage]);
          if (++stage == static_cast<uint32_t>(p.n_stages)) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) umma_commit(&tfull[acc]);
      }
      umma_commit(done);
      mbar_wait_drain(done, 0, p.status);
    }
  } else {
    // ---------------- epilogue: argmax over the tile's 128 rows ----------------
    const int q = warp & 3;  // TMEM lanes this warp may read: 32q .. 32q+31
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    for (int t = 0; t < n_tiles; ++t) {
      const int acc = t % p.n_acc;
      const uint32_t acc_phase = static_cast<uint32_t>((t / p.n_acc) & 1);
      const bool ok = mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status);
      if (!__all_sync(0xffffffffu, ok)) break;  // keep the warp converged for tcgen05.ld
      tc_fence_after();
      const int row0 = r0 + t * kTileRows;
      const int rows = min(kTileRows, r1 - row0);
      const bool valid = (q * 32 + lane) < rows;
      for (int c0 = 0; c0 < p.ntok; c0 += 16) {
        uint32_t v[16];
        tmem_ld_32x32b_x16(tmem_base + lane_base + static_cast<uint32_t>(acc * p.ntok + c0), v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t key = valid ? float_order_key(__uint_as_float(v[j])) : 0u;
          const uint32_t m = warp_max_u32(key);
          const uint32_t ball = __ballot_sync(0xffffffffu, valid && key == m);
          if (ball != 0u && lane == j) {
            const uint32_t row = static_cast<uint32_t>(row0 + q * 32 + (__ffs(ball) - 1));
            atomicMax(&best[c0 + j],
                      (static_cast<unsigned long long>(m) << 32) | (0xFFFFFFFFu - row));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }

  __syncthreads();
  griddep_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
  if (warp >= 2) {
    const int et = threadIdx.x - 64;
    for (int i = et; i < p.ntok; i += 128) {
      const unsigned long long b = best[i];
      if (b) atomicMax(&p.keys[i], b);
    }
    __threadfence();
    named_bar_sync(1, 128);
    if (et == 0) *last_flag = (atomicAdd(p.ticket, 1u) == gridDim.x - 1) ? 1 : 0;
    named_bar_sync(1, 128);
    if (*last_flag) {
      __threadfence();
      for (int b = et; b < p.batch; b += 128) finish_sequence(p, b);
      named_bar_sync(1, 128);
      for (int i = et; i < p.ntok; i += 128) p.keys[i] = 0ull;
      if (et == 0) *p.ticket = 0u;
    }
  }
}

// ---------------------------------------------------------------------------
// Large batches.  Past 256 token rows (batch 17 and up) the LM head is bound
// by the tensor cores rather than by the W_lm stream (2 * 16B flops per weight
// byte), and the token tile no longer fits beside a useful pipeline, so the
// logits are produced by the tiled GEMM of tile_gemm.cuh (128 token rows x
// 256 vocabulary rows per tile, clusters of two sharing each W_lm box) with an
// argmax epilogue, and one thread per sequence then finishes the verification
// (or the drafting) exactly as the skinny kernel's last CTA does.
// ---------------------------------------------------------------------------
constexpr int kWideMinRows = 257;

struct ArgmaxEpi {
  struct Params {
    unsigned long long* keys;  // [ntok] argmax keys, zero between calls
    int vocab, ntok;
  };
  static __device__ void setup(const Params&, float*, int) {}
  static __device__ void prologue(const TileCore&, const Params&) {}
  // thread = token row: the best key (order-preserving logit | ~vocabulary
  // index, so the lowest index wins an exact tie) over the tile's rows of
  // W_lm below the vocabulary size, merged into the row's key
  static __device__ void tile(const TileCore& p, const Params& e, int n, uint32_t tacc, int row,
                              const float*) {
    const int n0 = n * p.bn;
    unsigned long long best = 0ull;
    for (int c0 = 0; c0 < p.bn; c0 += 16) {
      uint32_t v[16];
      tmem_ld_32x32b_x16(tacc + c0, v);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int f = n0 + c0 + j;
        const unsigned long long k =
            (static_cast<unsigned long long>(float_order_key(__uint_as_float(v[j]))) << 32) |
            (0xFFFFFFFFu - static_cast<uint32_t>(f));
        if (f < e.vocab && k > best) best = k;
      }
    }
    if (row < e.ntok && best != 0ull) atomicMax(&e.keys[row], best);
  }
};

// One thread per sequence: acceptance and commit (or the drafted block) from
// the keys, which are then cleared for the next call.
__global__ void lm_finish_kernel(const LmParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.batch) return;
  finish_sequence(p, b);
  for (int i = 0; i < kBlock; ++i) p.keys[b * kBlock + i] = 0ull;
}

int launch_lmhead_wide(const dflash_dims& d, int budget_sms, const void* hidden,
                       const void* w_lm, LmParams& p, cudaStream_t st) {
  TileCore g = {};
  g.status = p.status;
  g.rows = p.ntok;
  g.m_tiles = (p.ntok + kTileM - 1) / kTileM;
  g.bn = 256;
  g.n_tiles = (d.vocab + g.bn - 1) / g.bn;  // the last tile's rows past V read as zeros
  g.k_tiles = d.hidden / 64;
  g.layer_cols = d.hidden;
  g.b_split = g.n_tiles;
  const uint64_t pitch = static_cast<uint64_t>(d.hidden) * 2;
  TokenMaps am;
  WeightMaps bm;
  int rc;
  if ((rc = make_tmap_2d_bf16(&am.m[0], hidden, d.hidden, p.ntok, pitch, 64, kTileM))) return rc;
  for (int l = 1; l < kMaxCtxLayers; ++l) am.m[l] = am.m[0];
  if ((rc = make_tmap_2d_bf16(&bm.m[0], w_lm, d.hidden, d.vocab, pitch, 64, g.bn / 2)))
    return rc;
  bm.m[1] = bm.m[2] = bm.m[0];
  ArgmaxEpi::Params ep = {p.keys, d.vocab, p.ntok};
  if ((rc = run_tile_gemm<ArgmaxEpi>(g, am, bm, ep, st, budget_sms))) return rc;
  return launch(lm_finish_kernel, dim3((p.batch + 127) / 128), dim3(128), 0, st, p);
}

}  // namespace

// Pipeline shape, tensor maps and launch of the LM-head kernel for `p` (whose
// workspace pointers and per-call outputs the caller has set).  Token rows:
// 16 per sequence, or -- x_rows > 0 -- x_rows rows x_pitch bytes apart (the
// MMA then takes them rounded up to 16, the rows past x_rows read as zeros).
int launch_lmhead(const dflash_dims& d, int budget_sms, const void* hidden, const void* w_lm,
                  LmParams& p, cudaStream_t st, int x_rows = 0, uint64_t x_pitch = 0) {
  p.vocab = d.vocab;
  p.hidden = d.hidden;
  p.ntok = x_rows > 0 ? (x_rows + 15) / 16 * 16 : d.batch * kBlock;
  p.batch = d.batch;
  if (x_rows == 0 && p.ntok >= kWideMinRows)
    return launch_lmhead_wide(d, budget_sms, hidden, w_lm, p, st);
  p.ntok_box = p.ntok <= 256 ? p.ntok : 256;
  p.n_xbox = (p.ntok + p.ntok_box - 1) / p.ntok_box;
  p.n_units = (p.vocab + kUnitRows - 1) / kUnitRows;
  p.x_chunk = ((p.n_xbox * p.ntok_box * 128) + 1023) / 1024 * 1024;
  const int fixed = 1024 /*alignment slack*/ + 8 * 5 + 16 + 8 * p.ntok + 64;
  // as many 64-column chunks per stage as divide K and still leave enough stages
  p.kb = kLmChunksPerStage;
  while (p.kb > 1 && ((p.hidden / 64) % p.kb ||
                      (kSmemBudget - fixed) / (p.kb * (kATileBytes + p.x_chunk) + 16) < kLmMinStages))
    p.kb >>= 1;
  p.stage_bytes = p.kb * (kATileBytes + p.x_chunk);
  p.n_stages = (kSmemBudget - fixed) / (p.stage_bytes + 16);
  if (p.n_stages > kMaxStages) p.n_stages = kMaxStages;
  if (p.n_stages < 2) return DFLASH_E_UNSUPPORTED;
  p.n_acc = (2 * p.ntok <= 512) ? 2 : 1;
  int cols = 32;
  while (cols < p.n_acc * p.ntok) cols *= 2;
  p.tmem_cols = cols;
  CUtensorMap tm_w, tm_x;
  PartialMaps tm_part;
  const uint64_t pitch = static_cast<uint64_t>(d.hidden) * 2;
  int rc;
  if ((rc = make_tmap_2d_bf16(&tm_w, w_lm, d.hidden, d.vocab, pitch, 64, kTileRows))) return rc;
  for (int bi = 0; bi < 4; ++bi)
    if ((rc = make_tmap_2d_bf16(&tm_part.m[bi], w_lm, d.hidden, d.vocab, pitch, 64, 64 >> bi)))
      return rc;
  if ((rc = make_tmap_2d_bf16(&tm_x, hidden, d.hidden, x_rows > 0 ? x_rows : p.ntok,
                              x_rows > 0 ? x_pitch : pitch, 64, p.ntok_box)))
    return rc;
  const int smem = p.n_stages * (p.stage_bytes + 16) + fixed;
  if ((rc = set_smem_limit(reinterpret_cast<const void*>(lmhead_argmax_accept_kernel), smem)))
    return rc;
  const int grid = budget_sms < p.n_units ? budget_sms : p.n_units;
  return launch(lmhead_argmax_accept_kernel, dim3(grid), dim3(kThreads), smem, st, tm_w, tm_part,
                tm_x, p);
}

}  // namespace dflash

using namespace dflash;

extern "C" int dflash_verify_accept(const dflash_dims* dims, const void* hidden,
                                    const void* w_lm, const int32_t* block_ids,
                                    const int32_t* len_before, int32_t* posterior,
                                    int32_t* accept_len, int32_t* next_staged,
                                    int32_t* commit_len, int32_t* out_tokens, int32_t out_cap,
                                    void* ws, size_t ws_bytes, dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_verify_accept");
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!hidden || !w_lm || !block_ids || !len_before || !posterior || !accept_len ||
      !next_staged || !commit_len || !out_tokens || out_cap < 1)
    return DFLASH_E_ARG;
  if (!aligned16(hidden) || !aligned16(w_lm)) return DFLASH_E_ALIGN;
  if (!ws) return DFLASH_E_WORKSPACE;
  Plan plan;
  if ((rc = make_plan(*dims, &plan))) return rc;
  if (ws_bytes < plan.total) return DFLASH_E_WORKSPACE;

  LmParams p = {};
  p.keys = ws_at<unsigned long long>(ws, plan.off_keys);
  p.ticket = ws_at<uint32_t>(ws, plan.off_tickets);
  p.status = ws_at<uint32_t>(ws, plan.off_status);
  p.batch = dims->batch;
  p.block_ids = block_ids;
  p.len_before = len_before;
  p.posterior = posterior;
  p.accept_len = accept_len;
  p.next_staged = next_staged;
  p.commit_len = commit_len;
  p.out_tokens = out_tokens;
  p.out_cap = out_cap;

  return launch_lmhead(*dims, plan.budget_sms, hidden, w_lm, p,
                       reinterpret_cast<cudaStream_t>(stream));
}

// ---------------------------------------------------------------------------
// Allocation-free variant of dflash_verify_accept.
//
// Some callers cannot hand this library a workspace: a plugin that receives
// tensors from a host framework owning every device allocation (and gives the
// plugin no allocator), a process running under a fixed device-memory budget,
// or code that must not allocate while a stream is being captured.  For them
// the LM-head/argmax/acceptance kernel's only scratch (one 64-bit argmax key
// per token row, the finishing ticket and a status word) lives in a
// library-owned array in device global memory, reserved when the library is
// loaded and kept by every GPU that loads it until the process exits.
// ---------------------------------------------------------------------------
namespace dflash {
namespace {

constexpr int kNoAllocMaxTokens = 512;   // batch * 16 at most (batch <= 32)
// every batch that check_dims accepts fits the array
static_assert(kNoAllocMaxTokens >= kMaxTokens, "the scratch array must cover every batch");
constexpr size_t kNoAllocKeyBytes = sizeof(unsigned long long) * kNoAllocMaxTokens;
constexpr size_t kNoAllocBytes = kNoAllocKeyBytes + 256;  // keys, then ticket and status

// Shared by every call on a device; holds the last call's contents.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
std::atomic<void*> g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).  In host code the array's name is
// only a host-side stand-in, so kernels must be given this address instead.
// Once a device's address is known, a call reads it with one acquire load;
// only the first lookup on a device takes the lock.
int noalloc_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH_E_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return DFLASH_E_UNSUPPORTED;
  void* p = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    p = g_noalloc_addr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return DFLASH_E_CUDA;
      g_noalloc_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return DFLASH_OK;
}

}  // namespace
}  // namespace dflash

extern "C" int dflash_verify_accept_noalloc(const dflash_dims* dims, const void* hidden,
                                            const void* w_lm, const int32_t* block_ids,
                                            const int32_t* len_before, int32_t* posterior,
                                            int32_t* accept_len, int32_t* next_staged,
                                            int32_t* commit_len, int32_t* out_tokens,
                                            int32_t out_cap, dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_verify_accept_noalloc");
  int rc = check_dims(dims);   // batch * 16 <= 512 = the array's token rows
  if (rc) return rc;
  if (!hidden || !w_lm || !block_ids || !len_before || !posterior || !accept_len ||
      !next_staged || !commit_len || !out_tokens || out_cap < 1)
    return DFLASH_E_ARG;
  if (!aligned16(hidden) || !aligned16(w_lm)) return DFLASH_E_ALIGN;
  void* scratch = nullptr;
  if ((rc = noalloc_scratch_address(&scratch))) return rc;
  Plan plan;
  if ((rc = make_plan(*dims, &plan))) return rc;

  LmParams p = {};
  char* base = static_cast<char*>(scratch);
  p.keys = reinterpret_cast<unsigned long long*>(base);
  p.ticket = reinterpret_cast<uint32_t*>(base + kNoAllocKeyBytes);
  p.status = reinterpret_cast<uint32_t*>(base + kNoAllocKeyBytes + 4);
  p.batch = dims->batch;
  p.block_ids = block_ids;
  p.len_before = len_before;
  p.posterior = posterior;
  p.accept_len = accept_len;
  p.next_staged = next_staged;
  p.commit_len = commit_len;
  p.out_tokens = out_tokens;
  p.out_cap = out_cap;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the keys and the ticket must start at zero; the status word is cleared too
  if ((rc = cuda_err(cudaMemsetAsync(scratch, 0, kNoAllocKeyBytes + 8, st)))) return rc;
  return launch_lmhead(*dims, plan.budget_sms, hidden, w_lm, p, st);
}

extern "C" int dflash_prefill_staged(const dflash_dims* dims, const void* hidden,
                                     int64_t row_pitch, const void* w_lm, int32_t* staged,
                                     void* ws, size_t ws_bytes, dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_prefill_staged");
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!hidden || !w_lm || !staged) return DFLASH_E_ARG;
  if (row_pitch < dims->hidden) return DFLASH_E_ARG;
  if (!aligned16(hidden) || !aligned16(w_lm) || (row_pitch * 2) % 16) return DFLASH_E_ALIGN;
  if (!ws) return DFLASH_E_WORKSPACE;
  Plan plan;
  if ((rc = make_plan(*dims, &plan))) return rc;
  if (ws_bytes < plan.total) return DFLASH_E_WORKSPACE;
  LmParams p = {};
  p.keys = ws_at<unsigned long long>(ws, plan.off_keys);
  p.ticket = ws_at<uint32_t>(ws, plan.off_tickets);
  p.status = ws_at<uint32_t>(ws, plan.off_status);
  p.draft = 2;
  p.block_out = staged;
  return launch_lmhead(*dims, plan.budget_sms, hidden, w_lm, p,
                       reinterpret_cast<cudaStream_t>(stream), dims->batch,
                       static_cast<uint64_t>(row_pitch) * 2);
}

extern "C" int dflash_draft_tokens(const dflash_dims* dims, const void* x,
                                   const void* final_norm_w, const void* w_lm,
                                   const int32_t* staged, int32_t* block_ids, int32_t* posterior,
                                   void* ws, size_t ws_bytes, dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_draft_tokens");
  int rc = check_dims(dims);
  if (rc) return rc;
  if (!x || !w_lm || !block_ids) return DFLASH_E_ARG;
  if (!aligned16(x) || !aligned16(w_lm)) return DFLASH_E_ALIGN;
  if (!ws) return DFLASH_E_WORKSPACE;
  DraftPlan plan;
  if ((rc = make_draft_plan(*dims, 128, &plan))) return rc;
  if (ws_bytes < plan.ffn_begin) return DFLASH_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // argmax(RMSNorm(x) * g W^T) = argmax((x * g) W^T): the norm's per-row factor
  // is positive, so only the gains reach the LM head
  void* xg = ws_at<void>(ws, plan.off_xg);
  if ((rc = launch_row_gain(x, final_norm_w, dims->hidden, plan.ntok, nullptr, nullptr, xg, st)))
    return rc;
  LmParams p = {};
  p.keys = ws_at<unsigned long long>(ws, plan.off_keys);
  p.ticket = ws_at<uint32_t>(ws, plan.off_lm_ticket);
  p.status = ws_at<uint32_t>(ws, plan.off_status);
  p.draft = 1;
  p.staged = staged;
  p.block_out = block_ids;
  p.posterior = posterior;
  return launch_lmhead(*dims, plan.budget_sms, xg, w_lm, p, st);
}
