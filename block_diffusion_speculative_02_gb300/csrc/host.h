// Host-side plumbing shared by the ABI entry points: argument checks, the
// workspace layout, tensor-map encoding and launch helpers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include <utility>

#include "../../include/dflash.h"

namespace dflash {

constexpr int kBlock = 16;          // staged token + 15 mask positions
constexpr int kMaxCtxLayers = 8;
constexpr int kMaxTokens = 512;     // batch * 16
constexpr int kMaxViews = 4;
constexpr int kMaxAttSplits = 64;

// Shared memory of one projection GEMM CTA (one CTA per SM).
constexpr int kGemmSmemBudget = 220 * 1024;

// Launch plan for one set of shapes on one device.  The workspace layout and
// every launch derive from the same plan, so they always agree; the layout
// depends on the device only, never on dflash_dims::sm_budget.
struct Plan {
  int num_sms;          // SMs of the device
  int budget_sms;       // SMs the LM head / projection grids may occupy
  int ntok;             // batch * 16
  // context projection
  int fc_out_tiles;     // hidden / 128
  int fc_k_tiles;       // nL * hidden / 64
  int fc_tok_chunks;    // ceil(ntok / 256)
  int kv_out_tiles;     // 2 * Hkv * D / 128
  int kv_k_tiles;       // hidden / 64
  int kv_tok_chunks;    // ceil(ntok / 128)  (hi + lo columns per chunk)
  // block attention
  int att_rows;         // (Hq / Hkv) * 16 query rows per KV head
  int att_splits;
  // workspace offsets (bytes)
  size_t off_status, off_tickets, off_keys, off_pos, off_ctx_tickets, off_ss, off_fc, off_yhat,
      off_kv, off_att_o, off_att_ml, total;
};

// Workspace plan of the drafter-layer calls (dflash_draft_*).  The buffers
// that do not depend on the MLP size come first (up to ffn_begin).
struct DraftPlan {
  int num_sms, budget_sms, ntok;
  int qkv_tiles, o_tiles, gu_tiles, down_tiles;  // output tiles of 128 features
  size_t off_status, off_lm_ticket, off_tickets_qkv, off_tickets_o, off_keys, off_ss_rows,
      off_ss_x1, off_xhl, off_x1, off_xg, off_acc_a, ffn_begin, off_tickets_gu,
      off_tickets_down, off_mhl, off_acc_b, total;
};

int make_draft_plan(const dflash_dims& d, int ffn, DraftPlan* p);

// Per token row of x [n_tok, H] bf16: sum(x^2) into ss (if not null), and
// x * gain either as a hi/lo bf16 pair into hl [2, n_tok, H] or rounded once
// into out [n_tok, H] (whichever is not null).
int launch_row_gain(const void* x, const void* gain, int H, int n_tok, void* hl, float* ss,
                    void* out, cudaStream_t st);

// Failure injection for tests (host side, no GPU involved): when the
// environment variable DFLASH_FAULT_INJECT names an entry point ("name" or
// "name:code"), that call returns the code (default DFLASH_E_CUDA) before it
// checks or launches anything.  Read at every call.
int injected_failure(const char* entry);
#define DFLASH_INJECT(entry)                          \
  do {                                                \
    if (int rc_inj_ = ::dflash::injected_failure(entry)) \
      return rc_inj_;                                 \
  } while (0)

// One NVTX range per entry-point call, named after the call (seen by
// profilers; without one attached the push and pop do nothing).
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

// Opening statement of every launching entry point.
#define DFLASH_ENTRY(entry)                  \
  ::dflash::CallRange call_range_(entry);   \
  DFLASH_INJECT(entry)

int check_dims(const dflash_dims* d);
int make_plan(const dflash_dims& d, Plan* p);
int current_num_sms();

// 2-D bf16 tensor map over a row-major [rows, cols] matrix with the given row
// pitch (bytes), box = box_cols x box_rows, 128-byte swizzle.
int make_tmap_2d_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                      uint64_t row_pitch_bytes, uint32_t box_cols, uint32_t box_rows);
// 3-D bf16 tensor map over [d2][d1][d0] with pitches (bytes) for d1 and d2.
int make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                      uint64_t d2, uint64_t pitch1, uint64_t pitch2, uint32_t box0,
                      uint32_t box1, uint32_t box2);

// inv_freq table of the rotary embedding (theta^(-2d/D), d < D/2) as float
// hi/lo pairs; filled in double precision on the host.
void fill_rope_table(float* hi, float* lo, int head_dim, double theta);

// The context projection as two tiled tensor-core GEMMs (ctx_prefill.cu), for
// tokens_per_seq rows per sequence written at write_pos.  The scratch
// pointers are regions of the caller's workspace: the status word, B
// write-position snapshots, (H / 128) x rows floats, rows x H bf16 for
// bf16(g_h Y) and, unless null, rows x H bf16 for its rounding remainder
// (then the K/V GEMM reads g_h Y as that hi/lo pair, else rounded once).  At
// most max_ctas CTAs (0: the whole device).  DFLASH_E_UNSUPPORTED, before
// anything is launched, for shapes the tiles do not cover.
int tiled_projection(const dflash_dims& d, int tokens_per_seq, const void* const* layer_hidden,
                     const void* w_fc, const void* hidden_norm_w, const void* w_k,
                     const void* w_v, const void* k_norm_w, const int32_t* write_pos,
                     const dflash_kv_view& cache, uint32_t* status, int32_t* pos_snapshot,
                     float* ss, uint16_t* yhat, uint16_t* yhat_lo, int max_ctas,
                     cudaStream_t st);

// Workspace bytes of dflash_prefill_attention for this chunk length (0 on bad
// arguments); dflash_prefill_workspace_bytes covers it.
size_t prefill_attention_workspace(const dflash_dims& d, int tokens_per_seq);

// Raise the dynamic shared-memory limit of a kernel once per device.
int set_smem_limit(const void* func, int bytes);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int cuda_err(cudaError_t e) { return e == cudaSuccess ? DFLASH_OK : DFLASH_E_CUDA; }

template <typename T>
inline T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// Launch with programmatic dependent launch allowed, so that a kernel's
// prologue may overlap the tail of the previous kernel on the stream.
template <typename... KArgs, typename... Args>
inline int launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                  cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return cuda_err(e);
}

}  // namespace dflash
