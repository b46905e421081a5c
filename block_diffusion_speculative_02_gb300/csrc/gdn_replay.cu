// Next: rollback of the recurrent state of a hybrid target by tape replay.
//
// "dflash-mlx" (dpshk.com) 保证三 and "DFlash双实现对比" (hotelren.com) §7: a
// GatedDeltaNet layer's state is a recurrence and cannot be cut back like a
// KV cache.  The verify forward records, per block step, the innovation of
// every recurrent head (key, value, write strength beta, log-decay g); once
// the acceptance is known only the committed 1 + a steps are replayed onto
// the state saved before the verify forward:
//   S <- exp(g) * S (I - beta k k^T) + beta v k^T
//      = a S + (beta v - a beta (S k)) k^T,   a = exp(g)
//
// Rows of S [Dv, Dk] evolve independently (row i needs only S_i . k and v_i).
// One CTA of 64 threads takes 32 rows of one head of one sequence: eight
// threads span a row and each thread holds four rows.  Thread (group, l) holds
// the float4 groups at columns 32 i + 4 l of its rows, so for a fixed i the
// eight threads of a row read 128 contiguous bytes of the state, and a key
// piece read from shared memory serves four rows (shared-memory wavefronts,
// not arithmetic, bound a one-row-per-thread layout).
//
// Per step the four partial dot products are reduced across the row group
// with four shuffles, transposed so that each thread ends with the full
// S_i . k of one row; that thread forms the row's coefficient and four more
// shuffles hand every thread the coefficients of its rows.  The rows are kept
// scaled, S = c S', with c (the product of the decays so far) the same for
// every row of the head, so a step is S' += (coef / c) k: one packed fp32 FMA
// per element pair for the update and one for the dot product.  c is anchored
// in log space: with L_t the running sum of the log-decays and
// F_t = 44 ceil(L_t / 44), c_t = exp(L_t - F_t) never drops below e^-44, and
// where the anchor moves S' is rescaled once.  All per-step scalars follow
// from one prefix sum over the steps.  Several CTAs stay resident per SM, so
// one CTA's loads overlap another's arithmetic; the state is read and written
// once.
#include "common.cuh"
#include "host.h"

namespace dflash {
namespace {

constexpr int kMaxSteps = 16;
constexpr int kRows = 32;            // state rows per CTA
constexpr int kRowsPerThread = 4;
constexpr int kLanesPerRow = 8;
constexpr int kThreads = kRows / kRowsPerThread * kLanesPerRow;
constexpr float kAnchor = 44.f;      // e^-44 ~ 2^-63.5: the smallest scale c kept

template <int DK>
__global__ void __launch_bounds__(kThreads) gdn_replay_kernel(
    float* __restrict__ state, const uint16_t* __restrict__ tape_k,
    const uint16_t* __restrict__ tape_v, const float* __restrict__ tape_beta,
    const float* __restrict__ tape_g, const int32_t* __restrict__ accept_len, int n_heads, int dv,
    uint32_t* status) {
  constexpr int kGroups = DK / (4 * kLanesPerRow);   // float4 groups per row per thread
  constexpr int kKVec = DK / 8;                      // 16-byte pieces of one key
  constexpr int kVVec = kRows / 8;                   // 16-byte pieces of the CTA's values
  constexpr int kKLoads = (kMaxSteps * kKVec + kThreads - 1) / kThreads;
  constexpr int kVLoads = (kMaxSteps * kVVec + kThreads - 1) / kThreads;
  static_assert(kMaxSteps <= 32, "the per-step scan runs in one warp");
  __shared__ __align__(16) float ks[kMaxSteps][DK];
  __shared__ float vs[kMaxSteps][kRows];
  __shared__ float4 prm[kMaxSteps];                  // (beta, dot scale, 1 / c, rescale or -1)
  __shared__ float c_end;
  griddep_wait();
  const int rblocks = dv / kRows;
  const int h = blockIdx.x / rblocks, r0 = (blockIdx.x - h * rblocks) * kRows;
  const int b = blockIdx.y;
  const int a = accept_len[b];
  if (a < 0 || a >= kMaxSteps) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, DFLASH_ST_CAPACITY);
    griddep_launch_dependents();
    return;
  }
  const int n = a + 1;
  const int tid = threadIdx.x, lane = tid & 31;
  const int l = tid % kLanesPerRow, row0 = tid / kLanesPerRow * kRowsPerThread;
  // this thread's state pieces, as pairs for the packed fp32 instructions
  float* sbase = state + ((static_cast<size_t>(b) * n_heads + h) * dv + r0 + row0) * DK + 4 * l;
  float2 s[kRowsPerThread][2 * kGroups];
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r)
#pragma unroll
    for (int i = 0; i < kGroups; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(sbase + r * DK + 32 * i);
      s[r][2 * i] = make_float2(v.x, v.y);
      s[r][2 * i + 1] = make_float2(v.z, v.w);
    }
  // the tape of the committed steps, 8 bf16 per 16-byte load, issued before
  // any of them (or the state above) is waited on
  {
    uint4 kw[kKLoads], vw[kVLoads];
#pragma unroll
    for (int u = 0; u < kKLoads; ++u) {
      const int q = u * kThreads + tid, t = q / kKVec, j = q - t * kKVec;
      if (t < n)
        kw[u] = *reinterpret_cast<const uint4*>(
            tape_k + ((static_cast<size_t>(b) * kMaxSteps + t) * n_heads + h) * DK + 8 * j);
    }
#pragma unroll
    for (int u = 0; u < kVLoads; ++u) {
      const int q = u * kThreads + tid, t = q / kVVec, j = q - t * kVVec;
      if (t < n)
        vw[u] = *reinterpret_cast<const uint4*>(
            tape_v + ((static_cast<size_t>(b) * kMaxSteps + t) * n_heads + h) * dv + r0 + 8 * j);
    }
    float bt = 0.f, gt = 0.f;
    if (tid < n) {
      const size_t o = (static_cast<size_t>(b) * kMaxSteps + tid) * n_heads + h;
      bt = tape_beta[o];
      gt = tape_g[o];
    }
#pragma unroll
    for (int u = 0; u < kKLoads; ++u) {
      const int q = u * kThreads + tid, t = q / kKVec, j = q - t * kKVec;
      if (t < n) {
        const uint32_t w[4] = {kw[u].x, kw[u].y, kw[u].z, kw[u].w};
        float4* dst = reinterpret_cast<float4*>(&ks[t][8 * j]);
        dst[0] = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                             __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
        dst[1] = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                             __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
      }
    }
#pragma unroll
    for (int u = 0; u < kVLoads; ++u) {
      const int q = u * kThreads + tid, t = q / kVVec, j = q - t * kVVec;
      if (t < n) {
        const uint32_t w[4] = {vw[u].x, vw[u].y, vw[u].z, vw[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          vs[t][8 * j + 2 * e] = __uint_as_float(w[e] << 16);
          vs[t][8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
      }
    }
    if (tid < 32) {
      // L_t = g_0 + ... + g_t by an inclusive scan over the steps; anchor
      // F_t = 44 ceil(L_t / 44); c_t = exp(L_t - F_t); S' is rescaled by
      // exp(F_t - F_{t-1}) where the anchor moves
      float L = tid < n ? gt : 0.f;
#pragma unroll
      for (int o = 1; o < kMaxSteps; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, L, o);
        if (tid >= o) L += y;
      }
      const float F = kAnchor * ceilf(L / kAnchor);
      float Fp = __shfl_up_sync(0xffffffffu, F, 1);
      if (tid == 0) Fp = 0.f;
      if (tid < n)
        prm[tid] = make_float4(bt, __expf(L - Fp), __expf(F - L), F != Fp ? __expf(F - Fp) : -1.f);
      if (tid == n - 1) c_end = __expf(L - F);
    }
  }
  __syncthreads();
  griddep_launch_dependents();
  const int b1 = (l >> 1) & 1, b2 = (l >> 2) & 1;
  const int mine = 2 * b2 + b1;                 // the row whose full dot this thread ends with
  const int src = lane & ~(kLanesPerRow - 1);   // first lane of the row group
  const float* vrow = &vs[0][row0 + mine];
  for (int t = 0; t < n; ++t) {
    float2 k[2 * kGroups];
#pragma unroll
    for (int i = 0; i < kGroups; ++i) {
      const float4 kv = *reinterpret_cast<const float4*>(&ks[t][32 * i + 4 * l]);
      k[2 * i] = make_float2(kv.x, kv.y);
      k[2 * i + 1] = make_float2(kv.z, kv.w);
    }
    float p[kRowsPerThread];
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
      float2 u0 = make_float2(0.f, 0.f), u1 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < kGroups; ++i) {
        u0 = __ffma2_rn(s[r][2 * i], k[2 * i], u0);
        u1 = __ffma2_rn(s[r][2 * i + 1], k[2 * i + 1], u1);
      }
      p[r] = (u0.x + u0.y) + (u1.x + u1.y);
    }
    // transpose-reduce over the eight threads of the row group
    const float e0 = (b2 ? p[2] : p[0]) + __shfl_xor_sync(0xffffffffu, b2 ? p[0] : p[2], 4);
    const float e1 = (b2 ? p[3] : p[1]) + __shfl_xor_sync(0xffffffffu, b2 ? p[1] : p[3], 4);
    float d = (b1 ? e1 : e0) + __shfl_xor_sync(0xffffffffu, b1 ? e0 : e1, 2);
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    const float4 pr = prm[t];
    const float w = pr.x * (vrow[t * kRows] - pr.y * d) * pr.z;
    if (pr.w >= 0.f) {                          // the anchor moved (the same for every thread)
      const float2 f2 = make_float2(pr.w, pr.w);
#pragma unroll
      for (int r = 0; r < kRowsPerThread; ++r)
#pragma unroll
        for (int i = 0; i < 2 * kGroups; ++i) s[r][i] = __fmul2_rn(s[r][i], f2);
    }
#pragma unroll
    for (int r = 0; r < kRowsPerThread; ++r) {
      const float wr = __shfl_sync(0xffffffffu, w, src | (r << 1));
      const float2 w2 = make_float2(wr, wr);
#pragma unroll
      for (int i = 0; i < 2 * kGroups; ++i) s[r][i] = __ffma2_rn(w2, k[i], s[r][i]);
    }
  }
  const float2 c2 = make_float2(c_end, c_end);
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r)
#pragma unroll
    for (int i = 0; i < kGroups; ++i) {
      const float2 lo = __fmul2_rn(s[r][2 * i], c2), hi = __fmul2_rn(s[r][2 * i + 1], c2);
      *reinterpret_cast<float4*>(sbase + r * DK + 32 * i) = make_float4(lo.x, lo.y, hi.x, hi.y);
    }
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" int dflash_gdn_replay(int32_t batch, int32_t n_heads, int32_t dk, int32_t dv,
                                 float* state, const void* tape_k, const void* tape_v,
                                 const float* tape_beta, const float* tape_g,
                                 const int32_t* accept_len, void* ws, size_t ws_bytes,
                                 dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_gdn_replay");
  if (batch < 1 || n_heads < 1 || !state || !tape_k || !tape_v || !tape_beta || !tape_g ||
      !accept_len)
    return DFLASH_E_ARG;
  if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return DFLASH_E_UNSUPPORTED;
  if (batch > 65535 || static_cast<long long>(n_heads) * (dv / kRows) > 0x7fffffff)
    return DFLASH_E_UNSUPPORTED;
  if (!aligned16(state) || !aligned16(tape_k) || !aligned16(tape_v)) return DFLASH_E_ALIGN;
  if (!ws || ws_bytes < 64) return DFLASH_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = ws_at<uint32_t>(ws, 0);
  const dim3 grid(n_heads * (dv / kRows), batch), block(kThreads);
  const auto* k = static_cast<const uint16_t*>(tape_k);
  const auto* v = static_cast<const uint16_t*>(tape_v);
  return dk == 128 ? launch(gdn_replay_kernel<128>, grid, block, 0, st, state, k, v, tape_beta,
                            tape_g, accept_len, n_heads, dv, status)
                   : launch(gdn_replay_kernel<64>, grid, block, 0, st, state, k, v, tape_beta,
                            tape_g, accept_len, n_heads, dv, status);
}
