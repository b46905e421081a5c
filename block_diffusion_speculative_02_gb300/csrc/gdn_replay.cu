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
// Rows of S [Dv, Dk] evolve independently (row i needs only S_i . k and v_i),
// so one CTA of 64 threads takes 32 rows of one head of one sequence: thread
// pair (2i, 2i+1) holds row i (half a row each, fp32 in registers) and the
// tape's steps sit in shared memory as fp32.  Per step: S k by a per-thread
// partial dot product and one shuffle, then the rank-one update in place.
// Small CTAs keep several resident per SM, so one CTA's loads overlap
// another's arithmetic; the state is read and written once, and the kernel is
// bound by those bytes.
#include "common.cuh"
#include "host.h"

namespace dflash {
namespace {

constexpr int kMaxSteps = 16;
constexpr int kRows = 32;       // state rows per CTA

template <int DK>
__global__ void __launch_bounds__(2 * kRows) gdn_replay_kernel(
    float* __restrict__ state, const uint16_t* __restrict__ tape_k,
    const uint16_t* __restrict__ tape_v, const float* __restrict__ tape_beta,
    const float* __restrict__ tape_g, const int32_t* __restrict__ accept_len, int n_heads, int dv,
    uint32_t* status) {
  constexpr int kCols = DK / 2;  // state columns per thread
  __shared__ float ks[kMaxSteps][DK];
  __shared__ float vs[kMaxSteps][kRows];
  __shared__ float bs[kMaxSteps], as[kMaxSteps];
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
  // the tape of the committed steps: 8 bf16 per 16-byte load, all of a
  // thread's loads issued before any is converted
  {
    constexpr int kVec = DK / 8;                 // 16-byte pieces per key
    uint4 kv[kMaxSteps * kVec / (2 * kRows)];
#pragma unroll
    for (int u = 0; u < kMaxSteps * kVec / (2 * kRows); ++u) {
      const int i = u * 2 * kRows + threadIdx.x;
      const int t = i / kVec, j = i - t * kVec;
      if (t < n)
        kv[u] = *reinterpret_cast<const uint4*>(
            tape_k + ((static_cast<size_t>(b) * kMaxSteps + t) * n_heads + h) * DK + 8 * j);
    }
    uint2 vv[kMaxSteps * kRows / 4 / (2 * kRows)];
#pragma unroll
    for (int u = 0; u < kMaxSteps * kRows / 4 / (2 * kRows); ++u) {
      const int i = u * 2 * kRows + threadIdx.x;
      const int t = i / (kRows / 4), j = i - t * (kRows / 4);
      if (t < n)
        vv[u] = *reinterpret_cast<const uint2*>(
            tape_v + ((static_cast<size_t>(b) * kMaxSteps + t) * n_heads + h) * dv + r0 + 4 * j);
    }
#pragma unroll
    for (int u = 0; u < kMaxSteps * kVec / (2 * kRows); ++u) {
      const int i = u * 2 * kRows + threadIdx.x;
      const int t = i / kVec, j = i - t * kVec;
      if (t < n) {
        const uint32_t w[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          ks[t][8 * j + 2 * e] = __uint_as_float(w[e] << 16);
          ks[t][8 * j + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kMaxSteps * kRows / 4 / (2 * kRows); ++u) {
      const int i = u * 2 * kRows + threadIdx.x;
      const int t = i / (kRows / 4), j = i - t * (kRows / 4);
      if (t < n) {
        vs[t][4 * j] = __uint_as_float(vv[u].x << 16);
        vs[t][4 * j + 1] = __uint_as_float(vv[u].x & 0xFFFF0000u);
        vs[t][4 * j + 2] = __uint_as_float(vv[u].y << 16);
        vs[t][4 * j + 3] = __uint_as_float(vv[u].y & 0xFFFF0000u);
      }
    }
  }
  if (threadIdx.x < n) {
    const size_t o = (static_cast<size_t>(b) * kMaxSteps + threadIdx.x) * n_heads + h;
    bs[threadIdx.x] = tape_beta[o];
    as[threadIdx.x] = __expf(tape_g[o]);
  }
  __syncthreads();
  const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
  float* srow = state + ((static_cast<size_t>(b) * n_heads + h) * dv + r0 + row) * DK +
                half * kCols;
  float s[kCols];
#pragma unroll
  for (int c = 0; c < kCols; c += 4) {
    const float4 v = *reinterpret_cast<const float4*>(srow + c);
    s[c] = v.x;
    s[c + 1] = v.y;
    s[c + 2] = v.z;
    s[c + 3] = v.w;
  }
  griddep_launch_dependents();
  for (int t = 0; t < n; ++t) {
    const float* k = &ks[t][half * kCols];
    float u0 = 0.f, u1 = 0.f;
#pragma unroll
    for (int c = 0; c < kCols; c += 2) {
      u0 = fmaf(s[c], k[c], u0);
      u1 = fmaf(s[c + 1], k[c + 1], u1);
    }
    float u = u0 + u1;
    u += __shfl_xor_sync(0xffffffffu, u, 1);   // the other half of the row
    const float al = as[t], be = bs[t];
    const float coef = be * (vs[t][row] - al * u);
#pragma unroll
    for (int c = 0; c < kCols; ++c) s[c] = fmaf(al, s[c], coef * k[c]);
  }
#pragma unroll
  for (int c = 0; c < kCols; c += 4)
    *reinterpret_cast<float4*>(srow + c) = make_float4(s[c], s[c + 1], s[c + 2], s[c + 3]);
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" int dflash_gdn_replay(int32_t batch, int32_t n_heads, int32_t dk, int32_t dv,
                                 float* state, const void* tape_k, const void* tape_v,
                                 const float* tape_beta, const float* tape_g,
                                 const int32_t* accept_len, void* ws, size_t ws_bytes,
                                 dflash_stream_t stream) {
  if (batch < 1 || n_heads < 1 || !state || !tape_k || !tape_v || !tape_beta || !tape_g ||
      !accept_len)
    return DFLASH_E_ARG;
  if ((dk != 64 && dk != 128) || (dv != 64 && dv != 128)) return DFLASH_E_UNSUPPORTED;
  if (batch > 65535) return DFLASH_E_UNSUPPORTED;
  if (!aligned16(state) || !aligned16(tape_k) || !aligned16(tape_v)) return DFLASH_E_ALIGN;
  if (!ws || ws_bytes < 64) return DFLASH_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = ws_at<uint32_t>(ws, 0);
  const dim3 grid(n_heads * (dv / kRows), batch), block(2 * kRows);
  const auto* k = static_cast<const uint16_t*>(tape_k);
  const auto* v = static_cast<const uint16_t*>(tape_v);
  return dk == 128 ? launch(gdn_replay_kernel<128>, grid, block, 0, st, state, k, v, tape_beta,
                            tape_g, accept_len, n_heads, dv, status)
                   : launch(gdn_replay_kernel<64>, grid, block, 0, st, state, k, v, tape_beta,
                            tape_g, accept_len, n_heads, dv, status);
}
