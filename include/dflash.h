/*
 * dflash.h — C ABI of the DFlash per-cycle hot path on one GB300 (sm_103a).
 *
 * One draft/verify cycle of block-diffusion speculative decoding, as the
 * DFlash pages describe it:
 *   [P1] "DFlash双实现对比：PyTorch与MLX代码架构差异深度分析" (hotelren.com)
 *        §2 attention (dual-source K/V), §3 KV-cache crop, §4 target-layer
 *        hidden states concatenated by target_layer_ids.
 *   [P2] "dflash-mlx" lossless speculative decoding (dpshk.com)
 *        块扩散草稿 (block = staged token + 15 masks; drafter reads target
 *        hidden states), 单次前向验证 ①–⑨ (the cycle), 保证二 (acceptance
 *        = sum(cumprod(draft == posterior))), 保证三 (cache cut back to the
 *        committed length).
 *
 * Conventions shared by every call
 *  - All pointers are borrowed.  Device buffers are owned by the caller; the
 *    library never allocates device memory.  Scratch lives in a caller
 *    workspace of dflash_workspace_bytes() bytes, zeroed once with
 *    dflash_workspace_init(); every call leaves its part of it zeroed again.
 *    Calls that share a workspace must be ordered on the GPU (same stream or
 *    events), except dflash_ctx_project and dflash_verify_accept, which use
 *    disjoint parts of it and may run concurrently on two streams, and
 *    dflash_kv_crop, which only sets bits of the status word (atomically)
 *    and may run concurrently with any call.
 *  - Every call is asynchronous on `stream` and never synchronises the host,
 *    except dflash_read_status.  Lengths stay on the device, so a whole cycle
 *    can be captured in a CUDA graph.
 *  - A negative return value is a host-detected error (bad argument, layout,
 *    alignment, workspace too small, CUDA launch error): nothing is launched.
 *  - Errors found on the device (a length out of range, an exhausted page
 *    pool, ...) set DFLASH_ST_* bits in a status word inside the workspace,
 *    leave the offending sequence's state unchanged, and never trap.  Read
 *    them with dflash_read_status.
 *  - bf16 is IEEE bfloat16; every bf16 result is rounded to nearest even.
 *    Matrix products accumulate in fp32.
 *  - Device pointers handed to TMA (weights, hidden states, caches) must be
 *    16-byte aligned and their rows a multiple of 16 bytes.
 *  - Every wait inside a kernel (on an mbarrier, a ticket or a counter) is
 *    bounded: after about a second it records DFLASH_ST_TIMEOUT and the
 *    kernel winds down and returns; nothing traps.
 *  - Failure injection for tests: when the environment variable
 *    DFLASH_FAULT_INJECT holds the name of an entry point ("dflash_kv_crop")
 *    or a name and a negative code ("dflash_kv_crop:-5"), that entry point
 *    returns the code (default DFLASH_E_CUDA) before checking or launching
 *    anything.  The variable is read at every call.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* dflash_stream_t;

/* Host-side return codes. */
#define DFLASH_OK 0
#define DFLASH_E_ARG (-1)          /* null pointer, bad size or shape        */
#define DFLASH_E_ALIGN (-2)        /* pointer or row pitch not 16-B aligned   */
#define DFLASH_E_UNSUPPORTED (-3)  /* shape the kernels do not implement      */
#define DFLASH_E_WORKSPACE (-4)    /* workspace null or too small             */
#define DFLASH_E_CUDA (-5)         /* CUDA runtime/driver error at launch     */

/* Device status-word bits (OR-ed; read with dflash_read_status). */
#define DFLASH_ST_CROP_GROW (1u << 0)     /* crop asked to grow or go negative      */
#define DFLASH_ST_OUT_OVERFLOW (1u << 1)  /* commit would pass out_cap              */
#define DFLASH_ST_PAGE_MISSING (1u << 2)  /* unmapped page inside a used range      */
#define DFLASH_ST_POOL_EMPTY (1u << 3)    /* page pool exhausted while reserving    */
#define DFLASH_ST_BAD_TOKEN (1u << 4)     /* block id outside [0, vocab)            */
#define DFLASH_ST_CAPACITY (1u << 5)      /* length or write past the cache capacity */
#define DFLASH_ST_TIMEOUT (1u << 6)       /* a bounded in-kernel wait gave up       */

/* Model and cycle shapes.  block must be 16 (staged token + 15 masks,
 * [P2] 块扩散草稿 step 1).  Supported: head_dim in {64, 128};
 * n_q_heads % n_kv_heads == 0 with (n_q_heads / n_kv_heads) * 16 <= 128;
 * hidden % 128 == 0; (n_kv_heads * head_dim) % 128 == 0; 1 <= n_ctx_layers <= 8;
 * batch * 16 <= 512. */
typedef struct {
  int32_t batch;         /* B: sequences in the step                       */
  int32_t block;         /* T: tokens per block, 16                        */
  int32_t hidden;        /* H: target (and drafter) hidden size            */
  int32_t n_q_heads;     /* Hq                                             */
  int32_t n_kv_heads;    /* Hkv                                            */
  int32_t head_dim;      /* D                                              */
  int32_t vocab;         /* V                                              */
  int32_t n_ctx_layers;  /* nL: target layers concatenated ([P1] §4)       */
  int32_t max_ctx;       /* upper bound on any context length; sizes the
                            attention split-K scratch                       */
  float rope_theta;      /* RoPE base (Qwen3: 1e6)                          */
  float rms_eps;         /* RMSNorm epsilon (1e-6)                          */
  int32_t sm_budget;     /* SMs that dflash_verify_accept and
                            dflash_ctx_project may occupy; 0 = all.  Two
                            calls given disjoint budgets (summing to at
                            most the SM count, see dflash_cycle_sm_split)
                            run side by side on two streams instead of
                            queueing for SMs.  The other calls ignore it,
                            and it does not change the workspace size.     */
} dflash_dims;

/* A KV cache as the kernels see it.  Both layouts are head-major, so that the
 * rows of one KV head are contiguous (what one attention CTA streams):
 *  contiguous (page_table == NULL): k, v are bf16 [B, Hkv, capacity, D].
 *  paged      (page_table != NULL): k, v are bf16 [n_pages, Hkv, page_size, D];
 *             page_table is int32 [B, max_pages] (-1 = unmapped); the free
 *             pages are free_list[0 .. *free_count) (int32, device).
 *  seq_len is int32 [B] on the device: the number of valid rows.
 *  k and v may be NULL for dflash_kv_crop, which touches only lengths and pages. */
typedef struct {
  void* k;
  void* v;
  int32_t* seq_len;
  int32_t* page_table;
  int32_t* free_list;
  int32_t* free_count;
  int32_t capacity;    /* contiguous: rows per sequence; paged: max_pages * page_size */
  int32_t page_size;   /* paged: 16                                                   */
  int32_t max_pages;   /* paged: page-table columns                                   */
  int32_t n_pages;     /* paged: pool size                                            */
} dflash_kv_view;

/* Bytes of workspace needed by every call below for these shapes on the
 * current device (split counts depend on its SM count).  0 on bad dims. */
DFLASH_API size_t dflash_workspace_bytes(const dflash_dims* dims);

/* Zero a workspace (cudaMemsetAsync on `stream`). */
DFLASH_API int dflash_workspace_init(void* ws, size_t ws_bytes, dflash_stream_t stream);

/* Budgets (dflash_dims::sm_budget) for running dflash_verify_accept and
 * dflash_ctx_project side by side on two streams.  At small batch both are
 * bound by the weights they stream (W_lm; W_fc, W_k, W_v), so the device's
 * SMs are split in proportion to those bytes, each side getting at least one
 * SM (past 256 token rows both are bound by the tensor cores instead and the
 * split is only a starting point for measuring).  Writes the two budgets
 * (summing to the SM count of the current device). */
DFLASH_API int dflash_cycle_sm_split(const dflash_dims* dims, int32_t* verify_sms,
                                     int32_t* project_sms);

/*
 * a1 — context projection ([P1] §4 and §2; [P2] 块扩散草稿 step 3).
 *   X  = [h_1 | ... | h_nL]                rows = B*16 tokens, nL*H features
 *   Y  = X W_fc^T                           fp32, H features
 *   Y^ = RMSNorm(Y) * hidden_norm_w         (skipped when hidden_norm_w == NULL)
 *   K  = RoPE_pos(RMSNorm_head(Y^ W_k^T) * k_norm_w)   (head norm skipped when NULL)
 *   V  = Y^ W_v^T
 * and writes K, V (bf16) into `cache` at rows write_pos[b] + t, t = 0..15,
 * RoPE position = that row index.  For a paged cache, unmapped pages covering
 * those rows are first taken from the free list.  Finally
 * cache->seq_len[b] = write_pos[b] + 16 (the crop then trims it to the
 * committed length).  write_pos may alias cache->seq_len.
 *   layer_hidden: HOST array of nL device pointers, each bf16 [B*16, H]
 *                 (row b*16 + t), in target_layer_ids order.
 *   w_fc: bf16 [H, nL*H] (row = output feature).  w_k, w_v: bf16 [Hkv*D, H].
 *   hidden_norm_w: bf16 [H] or NULL.  k_norm_w: bf16 [D] or NULL.
 *   write_pos: int32 [B] device.
 * Errors: DFLASH_ST_CAPACITY / DFLASH_ST_PAGE_MISSING / DFLASH_ST_POOL_EMPTY
 * skip the affected rows.
 */
DFLASH_API int dflash_ctx_project(const dflash_dims* dims, const void* const* layer_hidden,
                       const void* w_fc, const void* hidden_norm_w, const void* w_k,
                       const void* w_v, const void* k_norm_w, const int32_t* write_pos,
                       const dflash_kv_view* cache, void* ws, size_t ws_bytes,
                       dflash_stream_t stream);

/*
 * a2 — dual-source block attention ([P1] §2; [P2] 块扩散草稿).
 * For sequence b (L = cache->seq_len[b]), query head h, block row i:
 *   q   = RoPE_{L+i}(q_blk[b,i,h])
 *   K   = ctx K rows 0..L-1 of KV head g = h / (Hq/Hkv)   (stored rotated)
 *         ⊕ RoPE_{L+j}(k_blk[b,j,g]), j = 0..15
 *   V   = ctx V rows 0..L-1 ⊕ v_blk[b,j,g]
 *   out[b,i,h] = softmax(q K^T * scale) V      (no mask: non-causal in the block)
 *   q_blk: bf16 [B,16,Hq,D]; k_blk, v_blk: bf16 [B,16,Hkv,D] (before RoPE);
 *   out: bf16 [B,16,Hq,D].  Lengths above cache capacity set DFLASH_ST_CAPACITY
 *   (that sequence's output is left unwritten); unmapped pages inside the
 *   length set DFLASH_ST_PAGE_MISSING and are read as zeros.
 *   The cache is only read: its rows, and its page-table slots, below L.
 *   cache->seq_len may point at any int32 [B] array of lengths, e.g. the
 *   commit_len written by dflash_verify_accept, so that the attention need
 *   not wait for the dflash_kv_crop that stores the same lengths in the view
 *   (the crop releases only pages at or past the new length).
 */
DFLASH_API int dflash_block_attention(const dflash_dims* dims, const void* q_blk, const void* k_blk,
                           const void* v_blk, const dflash_kv_view* cache, float scale,
                           void* out, void* ws, size_t ws_bytes, dflash_stream_t stream);

/*
 * Next: the target's attention in the verify forward ([P2] 单次前向验证 ⑤:
 * one forward of the target over the block; 保证三: its cache is later cut
 * back to the committed length).  Same shapes, layouts and errors as
 * dflash_block_attention, with two differences: block row i sees the
 * context rows 0..L-1 and the block rows 0..i only (causal inside the
 * block), and the block's rotated K and its V are appended to `cache` at rows
 * L..L+15 (for a paged cache the pages those rows need are first taken from
 * its free list), after which cache->seq_len[b] = L + 16.  A length with no
 * room for 16 more rows sets DFLASH_ST_CAPACITY and appends nothing.
 */
DFLASH_API int dflash_verify_attention(const dflash_dims* dims, const void* q_blk,
                                       const void* k_blk, const void* v_blk,
                                       const dflash_kv_view* cache, float scale, void* out,
                                       void* ws, size_t ws_bytes, dflash_stream_t stream);

/*
 * a3 — verification epilogue ([P2] 单次前向验证 ⑤–⑧, 保证一, 保证二).
 *   logits[b,i,:] = hidden[b,i,:] W_lm^T        (fp32, never written to memory)
 *   posterior[b,i] = argmax (lowest index on exact ties)
 *   accept_len[b] = sum_{i<15} prod_{j<=i} [block_ids[b,j+1] == posterior[b,j]]
 *   out_tokens[b, len_before[b] + i] = block_ids[b,i], i = 0..accept_len[b]
 *   next_staged[b] = posterior[b, accept_len[b]]
 *   commit_len[b]  = len_before[b] + 1 + accept_len[b]
 *   hidden: bf16 [B,16,H] (final-normed); w_lm: bf16 [V,H];
 *   block_ids, posterior: int32 [B,16]; len_before, accept_len, next_staged,
 *   commit_len: int32 [B]; out_tokens: int32 [B, out_cap].
 *   len_before may alias commit_len.  A commit that would pass out_cap sets
 *   DFLASH_ST_OUT_OVERFLOW and leaves out_tokens, next_staged and commit_len of
 *   that sequence unchanged (posterior and accept_len are still written).
 *   Block ids outside [0, vocab) set DFLASH_ST_BAD_TOKEN (they never match).
 */
DFLASH_API int dflash_verify_accept(const dflash_dims* dims, const void* hidden, const void* w_lm,
                         const int32_t* block_ids, const int32_t* len_before,
                         int32_t* posterior, int32_t* accept_len, int32_t* next_staged,
                         int32_t* commit_len, int32_t* out_tokens, int32_t out_cap,
                         void* ws, size_t ws_bytes, dflash_stream_t stream);

/*
 * Allocation-free variant of dflash_verify_accept.  The DFlash pages have no
 * counterpart to this entry point; it exists for callers that cannot give
 * the library a workspace: plugins handed tensors by a host framework that
 * owns every device allocation and offers no allocator, processes held to a
 * fixed device-memory budget, and code that must not allocate while a stream
 * is being captured.
 * Same arguments and results as dflash_verify_accept, minus ws and
 * ws_bytes.  Its scratch (one 64-bit key per token row, a ticket, a status
 * word) is a library-owned static device array sized for batch * 16 <= 512
 * token rows (about 4 KB), held by every GPU that loads the library until the
 * process exits; larger batches return DFLASH_E_UNSUPPORTED.  It calls no
 * cudaMalloc/cudaFree and no allocating library routine.  The first call on a
 * device looks up the array's device address (once per device, with that
 * device current); make that first call before any stream capture.  Each call
 * clears the keys, ticket and status word (cudaMemsetAsync on `stream`)
 * before its kernel.  All calls share the one array and it keeps the last
 * call's contents, so calls that overlap on the GPU (other streams, other
 * threads) race: order them.  Device-side status bits of this variant are not
 * reported (there is no workspace to read them from): block ids outside the
 * vocabulary still never match and a commit that would pass out_cap is still
 * skipped, but nothing tells the caller, and if an in-kernel wait gives up
 * (DFLASH_ST_TIMEOUT in the workspace variant) the outputs are undefined.
 */
DFLASH_API int dflash_verify_accept_noalloc(const dflash_dims* dims, const void* hidden,
                                            const void* w_lm, const int32_t* block_ids,
                                            const int32_t* len_before, int32_t* posterior,
                                            int32_t* accept_len, int32_t* next_staged,
                                            int32_t* commit_len, int32_t* out_tokens,
                                            int32_t out_cap, dflash_stream_t stream);

/*
 * a4 — KV-cache crop ([P1] §3; [P2] 单次前向验证 ⑨, 保证三).
 * For each of the n_views caches (target view, drafter view, ...) and each
 * sequence b: seq_len[b] <- new_len[b].  Rows below new_len are untouched.
 * Paged views: every mapped page that starts at or after new_len[b] is pushed
 * back on the free list and its table slot set to -1 (the partly used last
 * page is kept).  new_len > seq_len or new_len < 0 sets DFLASH_ST_CROP_GROW
 * and leaves that sequence unchanged.  A page that would overflow a full free
 * list (*free_count == n_pages: an inconsistent pool) stays mapped to its
 * sequence, which reuses it when it grows again, and sets DFLASH_ST_CAPACITY;
 * the length is still cut.  n_views <= 4.  views is a HOST array.
 */
DFLASH_API int dflash_kv_crop(const dflash_kv_view* views, int32_t n_views, const int32_t* new_len,
                   int32_t batch, void* ws, size_t ws_bytes, dflash_stream_t stream);

/*
 * Next: the rest of one drafter layer and the drafter's tokens.
 * [P1] §1: the drafter is built from Qwen3 components (RMSNorm, rotary
 * embedding, MLP): pre-norm decoder layers with a per-head RMSNorm of q and k
 * and a SwiGLU MLP; [P2] 块扩散草稿 steps 1-2: the block (staged token + 15
 * masks) goes through one forward and every mask position predicts its own
 * token.  x below is the layer input, bf16 [B*16, H] (row b*16 + t).
 * These calls use their own workspace (dflash_draft_workspace_bytes, zeroed
 * once with dflash_workspace_init); its status word reads with
 * dflash_read_status.  ffn = MLP width F (multiple of 128).
 */
DFLASH_API size_t dflash_draft_workspace_bytes(const dflash_dims* dims, int32_t ffn);

/* h = RMSNorm(x) * ln1_w;  q = RMSNorm_head(h W_q^T) * q_norm_w;
 * k = RMSNorm_head(h W_k^T) * k_norm_w;  v = h W_v^T   (before RoPE:
 * dflash_block_attention rotates q and k).  w_q: bf16 [Hq*D, H]; w_k, w_v:
 * bf16 [Hkv*D, H]; ln1_w [H]; q_norm_w, k_norm_w [D] or NULL (no head norm).
 * q_out: bf16 [B*16, Hq*D] (= [B,16,Hq,D]); k_out, v_out: bf16 [B*16, Hkv*D]. */
DFLASH_API int dflash_draft_qkv(const dflash_dims* dims, const void* x, const void* ln1_w,
                                const void* w_q, const void* w_k, const void* w_v,
                                const void* q_norm_w, const void* k_norm_w, void* q_out,
                                void* k_out, void* v_out, void* ws, size_t ws_bytes,
                                dflash_stream_t stream);

/* x1 = x + O W_o^T;  x_out = x1 + (silu(h2 W_gate^T) * (h2 W_up^T)) W_down^T
 * with h2 = RMSNorm(x1) * ln2_w.  attn_out O: bf16 [B*16, Hq*D] (the output of
 * dflash_block_attention); w_o: bf16 [H, Hq*D]; w_gate, w_up: bf16 [ffn, H];
 * w_down: bf16 [H, ffn]; x_out: bf16 [B*16, H] (may alias x). */
DFLASH_API int dflash_draft_mlp(const dflash_dims* dims, int32_t ffn, const void* x,
                                const void* attn_out, const void* w_o, const void* ln2_w,
                                const void* w_gate, const void* w_up, const void* w_down,
                                void* x_out, void* ws, size_t ws_bytes, dflash_stream_t stream);

/* The drafter's tokens: for every block row the greedy argmax (lowest index
 * on exact ties) of RMSNorm(x) * final_norm_w W_lm^T, logits never stored
 * (the per-row norm factor does not change an argmax, so only the gains are
 * applied).  block_ids[b, 1..15] = the argmaxes of the mask rows 1..15;
 * block_ids[b, 0] = staged[b] when staged != NULL (e.g. next_staged of
 * dflash_verify_accept), else unchanged.  posterior (int32 [B,16]) receives
 * all 16 argmaxes when not NULL.  w_lm: bf16 [V, H]; final_norm_w [H] or
 * NULL. */
DFLASH_API int dflash_draft_tokens(const dflash_dims* dims, const void* x,
                                   const void* final_norm_w, const void* w_lm,
                                   const int32_t* staged, int32_t* block_ids, int32_t* posterior,
                                   void* ws, size_t ws_bytes, dflash_stream_t stream);

/*
 * Next: the context projection of a whole prompt, for the prefill ([P2]
 * 单次前向验证 ①: the target prefills the prompt in chunks and so initialises
 * the caches; [P1] §4: the drafter's context is the projection of the
 * target's selected-layer hidden states).  The arithmetic of
 * dflash_ctx_project, for T = tokens_per_seq rows per sequence instead of 16:
 *   Y = [h_1 | ... | h_nL] W_fc^T;  Y^ = RMSNorm(Y) * hidden_norm_w;
 *   K = RoPE_pos(RMSNorm_head(Y^ W_k^T) * k_norm_w);  V = Y^ W_v^T,
 * written into `cache` at rows write_pos[b] + t, t = 0..T-1 (RoPE position =
 * that row index); pages the rows need are first taken from the free list of
 * a paged cache; then cache->seq_len[b] = write_pos[b] + T.  write_pos may
 * alias cache->seq_len.  A long prompt is projected chunk by chunk, each call
 * appending T rows.  Y^ enters the K/V GEMM rounded once to bf16 (the
 * per-cycle call keeps it as a hi + lo pair).
 *   layer_hidden: HOST array of nL device pointers, each bf16 [B*T, H]
 *                 (row b*T + t).  w_fc, hidden_norm_w, w_k, w_v, k_norm_w as
 *                 for dflash_ctx_project.  write_pos: int32 [B] device.
 *   ws: dflash_prefill_workspace_bytes(dims, T) bytes, zeroed once (it also
 *   serves dflash_prefill_attention for the same T).
 * Requires hidden % 128 == 0, n_kv_heads * head_dim % 128 == 0.
 * Errors: DFLASH_ST_CAPACITY (no room for T rows: that sequence is left
 * alone), DFLASH_ST_POOL_EMPTY / DFLASH_ST_PAGE_MISSING (rows without a page
 * are skipped).
 */
DFLASH_API size_t dflash_prefill_workspace_bytes(const dflash_dims* dims, int32_t tokens_per_seq);
DFLASH_API int dflash_ctx_prefill(const dflash_dims* dims, int32_t tokens_per_seq,
                                  const void* const* layer_hidden, const void* w_fc,
                                  const void* hidden_norm_w, const void* w_k, const void* w_v,
                                  const void* k_norm_w, const int32_t* write_pos,
                                  const dflash_kv_view* cache, void* ws, size_t ws_bytes,
                                  dflash_stream_t stream);

/*
 * Next: the target's side of the prefill ([P2] 单次前向验证 ①: the target
 * prefills the prompt in chunks, which initialises its KV cache; ②: the
 * target's greedy token after the prompt is the first staged token).
 *
 * dflash_prefill_attention — one layer's attention over a prompt chunk of
 * T = tokens_per_seq rows per sequence.  With L = cache->seq_len[b], chunk
 * row t sits at position L + t and sees the cache rows 0..L-1 and the chunk
 * rows 0..t (causal):
 *   out[b,t,h] = softmax(RoPE_{L+t}(q[b,t,h]) K^T * scale) V
 *   K = cache K rows 0..L-1 of KV head h / (Hq/Hkv) ⊕ RoPE_{L+j}(k[b,j,g]), j <= t
 *   V = cache V rows 0..L-1 ⊕ v[b,j,g], j <= t.
 * The chunk's rotated K and its V are appended to `cache` at rows L..L+T-1
 * (for a paged cache the pages they need are first taken from its free
 * list), after which cache->seq_len[b] = L + T; a prompt fed chunk by chunk
 * gives the rows of the prompt fed at once.  Any T >= 1 with ceil(T/S) *
 * batch <= 65535, S = 32 when Hq/Hkv <= 4, else 16 (the prompt rows one CTA
 * takes: S times the group fills at most 128 MMA rows); else
 * DFLASH_E_UNSUPPORTED.
 *   q: bf16 [B, T, Hq, D]; k, v: bf16 [B, T, Hkv, D] (before RoPE);
 *   out: bf16 [B, T, Hq, D].
 *   ws: dflash_prefill_workspace_bytes(dims, T) bytes, zeroed once (the same
 *   workspace serves dflash_ctx_prefill); its status word reads with
 *   dflash_read_status.  dims->max_ctx bounds L + T (it sizes the split
 *   scratch).
 * Errors: L < 0 or L + T past the capacity sets DFLASH_ST_CAPACITY and leaves
 * that sequence (cache, length, output) untouched; DFLASH_ST_POOL_EMPTY /
 * DFLASH_ST_PAGE_MISSING as for dflash_verify_attention.
 */
DFLASH_API int dflash_prefill_attention(const dflash_dims* dims, int32_t tokens_per_seq,
                                        const void* q, const void* k, const void* v,
                                        const dflash_kv_view* cache, float scale, void* out,
                                        void* ws, size_t ws_bytes, dflash_stream_t stream);

/*
 * dflash_prefill_staged — the first staged token: staged[b] = argmax over the
 * vocabulary of hidden_b W_lm^T (lowest index on exact ties; logits never
 * written), hidden_b being the final-normed hidden state of sequence b's
 * last prompt row, bf16 [H] at hidden + b * row_pitch elements (row_pitch >=
 * H, a multiple of 8: e.g. T * H to take row T-1 of a [B, T, H] array).
 * w_lm: bf16 [V, H]; staged: int32 [B].  ws: a workspace of
 * dflash_workspace_bytes(dims) bytes (the verification's), zeroed once.
 */
DFLASH_API int dflash_prefill_staged(const dflash_dims* dims, const void* hidden,
                                     int64_t row_pitch, const void* w_lm, int32_t* staged,
                                     void* ws, size_t ws_bytes, dflash_stream_t stream);

/*
 * Next: rollback of the recurrent state of a hybrid target ([P2] 保证三:
 * GatedDeltaNet states cannot be cut back; the verify forward records each
 * step's innovation and only the accepted steps are replayed; [P1] §7).
 * For every sequence b and recurrent head h (the heads of all GatedDeltaNet
 * layers, n_heads in total), for t = 0 .. accept_len[b] (1 + a steps):
 *   S <- exp(g[b,t,h]) * S (I - beta[b,t,h] k k^T) + beta[b,t,h] v k^T,
 *   k = tape_k[b,t,h], v = tape_v[b,t,h].
 * state: fp32 [B, n_heads, dv, dk], in place (the state saved before the
 * verify forward in, the state after the committed tokens out).
 * tape_k: bf16 [B, 16, n_heads, dk]; tape_v: bf16 [B, 16, n_heads, dv];
 * tape_beta, tape_g: fp32 [B, 16, n_heads]; accept_len: int32 [B] device
 * (from dflash_verify_accept).  dk, dv in {64, 128}.  accept_len outside
 * 0..15 sets DFLASH_ST_CAPACITY and leaves that sequence's state.  ws: any
 * zeroed workspace of at least 64 bytes (its status word is used).
 */
DFLASH_API int dflash_gdn_replay(int32_t batch, int32_t n_heads, int32_t dk, int32_t dv,
                                 float* state, const void* tape_k, const void* tape_v,
                                 const float* tape_beta, const float* tape_g,
                                 const int32_t* accept_len, void* ws, size_t ws_bytes,
                                 dflash_stream_t stream);

/* Copy the status word to *host_status (synchronises `stream`); if clear != 0
 * reset it to zero afterwards. */
DFLASH_API int dflash_read_status(void* ws, uint32_t* host_status, int clear, dflash_stream_t stream);

/* Text for a return code. */
DFLASH_API const char* dflash_status_string(int code);

/*
 * Self-test of the bounded wait every kernel uses: one warp waits on an
 * mbarrier; with arrive != 0 one arrival completes it at once, with
 * arrive == 0 nothing arrives and the wait gives up after its time limit
 * (about a second), records DFLASH_ST_TIMEOUT in the status word of `ws`
 * and the kernel returns; the context stays usable.  ws: at least 64 bytes.
 */
DFLASH_API int dflash_selftest_wait(int arrive, void* ws, size_t ws_bytes, dflash_stream_t stream);

/* Library ABI version (major * 100 + minor): 108. */
DFLASH_API int dflash_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */
