// ABI plumbing: dimension checks, the split plan / workspace layout, tensor-map
// encoding, status word access.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "host.h"
#include "streamk_gemm.cuh"

namespace dflash {

namespace {

#ifndef DFLASH_TMAP_L2_PROMOTION
#define DFLASH_TMAP_L2_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

}  // namespace

int injected_failure(const char* entry) {
  const char* v = std::getenv("DFLASH_FAULT_INJECT");
  if (!v || !*v) return 0;
  const size_t n = std::strlen(entry);
  if (std::strncmp(v, entry, n) != 0 || (v[n] != '\0' && v[n] != ':')) return 0;
  if (v[n] == ':') {
    const int code = std::atoi(v + n + 1);
    if (code < 0) return code;
  }
  return DFLASH_E_CUDA;
}

namespace {

// One warp waits on an mbarrier with the same bounded wait every kernel uses.
// With arrive == 0 nothing ever arrives: the wait gives up after its time
// limit and records DFLASH_ST_TIMEOUT, and the kernel returns normally.
__global__ void selftest_wait_kernel(int arrive, uint32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && arrive) mbar_arrive(&bar);
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status);
}

}  // namespace

int check_dims(const dflash_dims* d) {
  if (!d) return DFLASH_E_ARG;
  if (d->block != kBlock) return DFLASH_E_UNSUPPORTED;
  if (d->batch < 1 || d->batch * kBlock > kMaxTokens) return DFLASH_E_UNSUPPORTED;
  if (d->hidden < 128 || d->hidden % 128) return DFLASH_E_UNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128) return DFLASH_E_UNSUPPORTED;
  if (d->n_kv_heads < 1 || d->n_q_heads < d->n_kv_heads || d->n_q_heads % d->n_kv_heads)
    return DFLASH_E_UNSUPPORTED;
  if ((d->n_q_heads / d->n_kv_heads) * kBlock > 128) return DFLASH_E_UNSUPPORTED;
  if ((d->n_kv_heads * d->head_dim) % 128) return DFLASH_E_UNSUPPORTED;
  if (d->vocab < 1) return DFLASH_E_ARG;
  if (d->n_ctx_layers < 1 || d->n_ctx_layers > kMaxCtxLayers) return DFLASH_E_UNSUPPORTED;
  if (d->max_ctx < 0 || d->sm_budget < 0) return DFLASH_E_ARG;
  if (!(d->rms_eps >= 0.0f) || !(d->rope_theta > 0.0f)) return DFLASH_E_ARG;
  return DFLASH_OK;
}

int current_num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int make_plan(const dflash_dims& d, Plan* p) {
  int rc = check_dims(&d);
  if (rc) return rc;
  Plan q = {};
  q.num_sms = current_num_sms();
  if (q.num_sms <= 0) return DFLASH_E_CUDA;
  q.budget_sms = d.sm_budget > 0 && d.sm_budget < q.num_sms ? d.sm_budget : q.num_sms;
  q.ntok = d.batch * kBlock;
  q.fc_out_tiles = d.hidden / 128;
  q.fc_k_tiles = d.n_ctx_layers * d.hidden / 64;
  q.fc_tok_chunks = (q.ntok + 255) / 256;
  q.kv_out_tiles = 2 * d.n_kv_heads * d.head_dim / 128;
  q.kv_k_tiles = d.hidden / 64;
  q.kv_tok_chunks = (q.ntok + 127) / 128;
  q.att_rows = (d.n_q_heads / d.n_kv_heads) * kBlock;
  {
    // enough (sequence, KV head, split) CTAs to fill every SM once (one
    // attention CTA per SM), and no split longer than 4096 keys so that
    // ragged batches balance
    const int pages = (d.max_ctx + 15) / 16;
    int s = q.num_sms / (d.batch * d.n_kv_heads);
    const int by_len = (d.max_ctx + 4095) / 4096;
    if (s < by_len) s = by_len;
    if (s > pages) s = pages;
    if (s > kMaxAttSplits) s = kMaxAttSplits;  // the split merge stages at most 64 splits
    if (s < 1) s = 1;
    q.att_splits = s;
  }
  size_t off = 0;
  q.off_status = off;  off += 64;
  q.off_tickets = off; off += 192;
  q.off_keys = off;    off = align_up(off + sizeof(unsigned long long) * q.ntok, 256);
  q.off_pos = off;     off = align_up(off + sizeof(int32_t) * d.batch, 256);
  q.off_ctx_tickets = off;
  off = align_up(off + sizeof(uint32_t) * (q.fc_out_tiles * q.fc_tok_chunks +
                                           q.kv_out_tiles * q.kv_tok_chunks), 256);
  q.off_ss = off;      off = align_up(off + sizeof(float) * (size_t)q.fc_out_tiles * q.ntok, 256);
  // partial tiles of the two stream-K GEMMs (sk::partial_bytes: every SM budget fits)
  q.off_fc = off;
  off = align_up(off + sk::partial_bytes(sk::gemm_dims(q.ntok, d.n_ctx_layers * d.hidden,
                                                       q.fc_out_tiles, 0), q.num_sms), 256);
  q.off_yhat = off;    off = align_up(off + 2 * sizeof(uint16_t) * (size_t)q.ntok * d.hidden, 1024);
  q.off_kv = off;
  off = align_up(off + sk::partial_bytes(sk::gemm_dims(q.ntok, d.hidden, q.kv_out_tiles, 1),
                                         q.num_sms), 256);
  const size_t att_units = (size_t)d.batch * d.n_kv_heads * q.att_splits * q.att_rows;
  q.off_att_o = off;   off = align_up(off + sizeof(float) * att_units * d.head_dim, 256);
  q.off_att_ml = off;  off = align_up(off + sizeof(float) * 2 * att_units, 256);
  q.total = off;
  *p = q;
  return DFLASH_OK;
}

int make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                      uint64_t row_pitch_bytes, uint32_t box_cols, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return DFLASH_E_CUDA;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, DFLASH_TMAP_L2_PROMOTION,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_E_ALIGN;
}

int make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                      uint64_t d2, uint64_t pitch1, uint64_t pitch2, uint32_t box0,
                      uint32_t box1, uint32_t box2) {
  auto enc = encode_fn();
  if (!enc) return DFLASH_E_CUDA;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {pitch1, pitch2};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, DFLASH_TMAP_L2_PROMOTION,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_E_ALIGN;
}

void fill_rope_table(float* hi, float* lo, int head_dim, double theta) {
  for (int d = 0; d < head_dim / 2; ++d) {
    const double f = std::pow(theta, -2.0 * d / head_dim);
    hi[d] = static_cast<float>(f);
    lo[d] = static_cast<float>(f - static_cast<double>(hi[d]));
  }
}

int set_smem_limit(const void* func, int bytes) {
  return cuda_err(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
}

}  // namespace dflash

using namespace dflash;

extern "C" size_t dflash_workspace_bytes(const dflash_dims* dims) {
  if (check_dims(dims)) return 0;
  Plan p;
  if (make_plan(*dims, &p)) return 0;
  return p.total;
}

extern "C" int dflash_cycle_sm_split(const dflash_dims* dims, int32_t* verify_sms,
                                     int32_t* project_sms) {
  if (!verify_sms || !project_sms) return DFLASH_E_ARG;
  int rc = check_dims(dims);
  if (rc) return rc;
  const int nsm = current_num_sms();
  if (nsm < 2) return DFLASH_E_CUDA;
  const double h = dims->hidden;
  const double lm = static_cast<double>(dims->vocab) * h;
  const double proj = dims->n_ctx_layers * h * h +
                      2.0 * dims->n_kv_heads * dims->head_dim * h;
  int p = static_cast<int>(std::lround(nsm * proj / (proj + lm)));
  if (p < 1) p = 1;
  if (p > nsm - 1) p = nsm - 1;
  *project_sms = p;
  *verify_sms = nsm - p;
  return DFLASH_OK;
}

extern "C" int dflash_workspace_init(void* ws, size_t ws_bytes, dflash_stream_t stream) {
  if (!ws || ws_bytes < 256) return DFLASH_E_WORKSPACE;
  return cuda_err(cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" int dflash_read_status(void* ws, uint32_t* host_status, int clear,
                                  dflash_stream_t stream) {
  if (!ws || !host_status) return DFLASH_E_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host_status, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), s);
  return cuda_err(e);
}

extern "C" const char* dflash_status_string(int code) {
  switch (code) {
    case DFLASH_OK: return "ok";
    case DFLASH_E_ARG: return "invalid argument";
    case DFLASH_E_ALIGN: return "pointer or pitch not 16-byte aligned";
    case DFLASH_E_UNSUPPORTED: return "unsupported shape";
    case DFLASH_E_WORKSPACE: return "workspace missing or too small";
    case DFLASH_E_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

extern "C" int dflash_version(void) { return 108; }

extern "C" int dflash_selftest_wait(int arrive, void* ws, size_t ws_bytes,
                                    dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_selftest_wait");
  if (!ws || ws_bytes < 64) return DFLASH_E_WORKSPACE;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      arrive, static_cast<uint32_t*>(ws));
  return cuda_err(cudaGetLastError());
}
