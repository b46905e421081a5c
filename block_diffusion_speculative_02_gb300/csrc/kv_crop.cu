// a4 — KV-cache crop to the committed length.
//
// "DFlash双实现对比" (hotelren.com) §3: after each draft/verify cycle only the
// accepted prefix may stay in the caches, and the target and drafter caches
// are cut back together.  "dflash-mlx" (dpshk.com) 单次前向验证 ⑨ and 保证三:
// the attention KV cache is simply trimmed to the committed length.
//
// One thread per (view, sequence).  Lengths move only downwards; for a paged
// view every mapped page that starts at or after the new length is pushed on
// the free list (a stack indexed by *free_count) and unmapped.  The work is
// O(batch + released pages): the bytes of the cache are never touched.
#include "common.cuh"
#include "host.h"

namespace dflash {
namespace {

struct CropViews {
  dflash_kv_view v[kMaxViews];
  int n;
};

__global__ void kv_crop_kernel(const CropViews views, const int32_t* __restrict__ new_len,
                               int batch, uint32_t* status) {
  // the next kernel may start its prologue now: whatever it reads of ours it
  // reads after its own wait, which covers our completion
  griddep_launch_dependents();
  griddep_wait();
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= views.n * batch) return;
  const int vi = idx / batch;
  const int b = idx - vi * batch;
  const dflash_kv_view& v = views.v[vi];
  const int old = v.seq_len[b];
  const int nl = new_len[b];
  if (nl < 0 || nl > old) {
    set_status(status, DFLASH_ST_CROP_GROW);
    return;
  }
  if (v.page_table != nullptr) {
    const int ps = v.page_size;
    const int p_from = (nl + ps - 1) / ps;
    const int p_to = min((old + ps - 1) / ps, v.max_pages);
    int32_t* row = v.page_table + static_cast<size_t>(b) * v.max_pages;
    for (int pg = p_from; pg < p_to; ++pg) {
      const int page = row[pg];
      if (page < 0) continue;
      const int slot = atomicAdd(v.free_count, 1);
      if (slot < v.n_pages) {
        v.free_list[slot] = page;
        row[pg] = -1;
      } else {
        // the free list is already full (the pool's pages were counted twice
        // somewhere): the page stays mapped to this sequence, which reuses it
        // when it grows again, so no page is lost
        atomicSub(v.free_count, 1);
        set_status(status, DFLASH_ST_CAPACITY);
      }
    }
  }
  v.seq_len[b] = nl;
}

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" int dflash_kv_crop(const dflash_kv_view* views, int32_t n_views,
                              const int32_t* new_len, int32_t batch, void* ws, size_t ws_bytes,
                              dflash_stream_t stream) {
  DFLASH_ENTRY("dflash_kv_crop");
  if (!views || n_views < 1 || n_views > kMaxViews || !new_len || batch < 1)
    return DFLASH_E_ARG;
  if (!ws || ws_bytes < 64) return DFLASH_E_WORKSPACE;
  CropViews cv = {};
  cv.n = n_views;
  for (int i = 0; i < n_views; ++i) {
    const dflash_kv_view& v = views[i];
    if (!v.seq_len) return DFLASH_E_ARG;
    if (v.page_table) {
      if (!v.free_list || !v.free_count || v.page_size < 1 || v.max_pages < 1 || v.n_pages < 1)
        return DFLASH_E_ARG;
    }
    cv.v[i] = v;
  }
  const int n = n_views * batch;
  const int threads = 128;
  return launch(kv_crop_kernel, dim3((n + threads - 1) / threads), dim3(threads), 0,
                reinterpret_cast<cudaStream_t>(stream), cv, new_len, static_cast<int>(batch),
                ws_at<uint32_t>(ws, 0));
}
