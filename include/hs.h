/*
 * hs.h - C ABI of a GB300 (sm_103a) library for one decode step of query-aware
 * block-sparse attention over a paged KV cache, with a HiSparse-style hot
 * device buffer.
 *
 * The operations follow these pages:
 *   [KVS] "KV 稀疏化" (KV-cache sparsity wiki): §2 attention sink + sliding
 *         window, §5 Quest (per-block min/max summary, coarse filter of the
 *         query against the summaries, top-k blocks, full attention on the
 *         chosen blocks only), §7 HiSparse (hot device buffer, host inactive KV,
 *         swap-in kernel that detects misses, updates the page table and brings
 *         KV back).
 *   [SPD] "SparDA：把KV選擇提前一層，長上下文推理顯存帶寬雙優化": §4.2 the
 *         selector keeps sink + local window + remote top-k; §4.3 the sparse
 *         index lives on top of PagedAttention blocks.
 *   [FLL] "分块稀疏注意力与KV Cache量化：长文本推理显存优化实践": §2.2 tiled
 *         attention carrying a running max and normaliser across tiles, §2.4
 *         grouped KV quantisation with a per-group scale, §3.2 group size 32.
 *
 * Conventions shared by every call
 *   - Every buffer is owned by the caller.  Device pointers must point to
 *     memory of the current CUDA device; the library never allocates, frees or
 *     synchronises (except hs_get_device_error).
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).
 *   - Arguments are checked on the host before anything is launched; a failed
 *     check returns HS_ERR_INVALID_ARG / HS_ERR_UNSUPPORTED and launches
 *     nothing.  Errors found by a kernel (a page id outside the pool, a block
 *     index outside the request, a selection larger than a capacity) set bits
 *     in a per-device error word read by hs_get_device_error(); the kernel
 *     skips the offending item and carries on.
 *   - No C++ exception crosses this interface.
 *
 * Layouts (row-major, innermost last)
 *   B = block_size tokens per block (= per page), D = head_dim,
 *   Hq / Hkv query / kv heads, g = Hq / Hkv query heads per kv head,
 *   N_b = ceil(seq_lens[b] / B) blocks of request b.
 *   k_pages, v_pages  [num_pages][B][D]   f32 | bf16 | e4m3 (one byte)
 *   k_scales,v_scales [num_pages][B][D/32] f32 (e4m3 only, else NULL)
 *   page_table        [batch][Hkv][max_blocks] int32: physical page of block j
 *                     of (b, kvh); only entries j < N_b are read.
 *   seq_lens          [batch] int32 tokens of each request, including the
 *                     token being decoded.
 *   q                 [batch][Hq][D]  f32 for f32 K/V, bf16 otherwise.
 *   smin, smax        [batch][Hkv][max_blocks][D]  f32 for f32 K/V, bf16
 *                     otherwise.
 *   sel               [batch][Hkv][capacity] int32 ascending block indices,
 *                     entries past sel_count are -1.
 *   sel_count         [batch][Hkv] int32.
 *   out               [batch][Hq][D]  bf16, or f32 when out_is_fp32.
 *   lse               [batch][Hq] f32 natural-log sum of exp of the logits.
 */
#ifndef HS_H_
#define HS_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define HS_API __attribute__((visibility("default")))
#else
#define HS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* hs_stream_t; /* cudaStream_t */

typedef enum hs_status {
  HS_OK = 0,
  HS_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad layout */
  HS_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, group size, ... */
  HS_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  HS_ERR_OUT_OF_RANGE = 4, /* device: page id or block index outside its range */
  HS_ERR_CAPACITY = 5,     /* device: selection larger than capacity / hot slots */
  HS_ERR_TIMEOUT = 6,      /* device: a bounded wait gave up */
  HS_ERR_WORKSPACE = 7,    /* workspace missing or smaller than hs_workspace_bytes */
  HS_ERR_SCRATCH_LIMIT = 8 /* needs more than the fixed scratch of the _noalloc call */
} hs_status;

/* Bits of the per-device error word. */
#define HS_EBIT_PAGE_RANGE 0x1u  /* page id < 0 or >= num_pages */
#define HS_EBIT_CAPACITY 0x2u    /* count > capacity, or > hot-buffer slots */
#define HS_EBIT_TIMEOUT 0x4u     /* a bounded device wait expired */
#define HS_EBIT_BLOCK_RANGE 0x8u /* selected block index outside [0, N_b) */

typedef enum hs_kv_dtype {
  HS_KV_F32 = 0,         /* fp32 K/V, fp32 q, fp32 summaries */
  HS_KV_BF16 = 1,        /* bf16 K/V, bf16 q, bf16 summaries */
  HS_KV_FP8E4M3_G32 = 2  /* e4m3 K/V + one fp32 scale per 32 channels per token;
                            bf16 q; bf16 summaries rounded outward */
} hs_kv_dtype;

/* Attention geometry.  head_dim in {64, 128}; num_q_heads / num_kv_heads in
 * {1, 2, 4, 8, 16}; block_size in [1, 256] (the tensor-core attention path
 * needs block_size in {16, 32, 64, 128}). */
typedef struct hs_attn_shape {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t kv_dtype; /* hs_kv_dtype */
} hs_attn_shape;

/* A paged KV cache (device memory, or mapped pinned host memory for reads). */
typedef struct hs_paged_kv {
  const void* k_pages;
  const void* v_pages;
  const float* k_scales; /* e4m3 only */
  const float* v_scales; /* e4m3 only */
  const int32_t* page_table;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t max_blocks; /* row length of page_table, smin/smax and scores */
  int64_t num_pages;  /* pages in k_pages / v_pages: valid ids are [0, num_pages) */
} hs_paged_kv;

/* Which blocks are forced and how many more are chosen by score
 * ([KVS] §2, [SPD] §4.2): a block is forced when it overlaps the first
 * sink_tokens tokens or the last window_tokens tokens of its request; k_scored
 * further blocks are the best-scoring of the rest (ties -> lower index).
 * capacity is the row length of sel and must be >= the largest possible
 * selection, ceil(sink/B) + ceil(window/B) + 1 + k_scored (or max_blocks if
 * smaller).
 * Score smoothing across decode steps ([SPD] §6.1, which blends 70% of the
 * current score with 30% of the previous one): with history_weight w in
 * (0, 1), the score a block is ranked by is (1 - w) * score + w * h, where h
 * is its entry in score_history when that is a number, else the score
 * itself; the ranked value is then stored back into score_history.
 * score_history [batch][Hkv][max_blocks] f32, device, read and written for
 * blocks j < N_b; fill it with NaN before the first step.  w = 0 turns the
 * smoothing off and score_history may be NULL. */
typedef struct hs_select_params {
  int32_t sink_tokens;
  int32_t window_tokens;
  int32_t k_scored;
  int32_t capacity;
  float history_weight;
  float* score_history;
} hs_select_params;

/* Attention options.  scale multiplies q.k (usually 1/sqrt(head_dim)).
 * blocks_per_split: selected blocks handled by one CTA before the LSE merge;
 * 0 = chosen by the library from the SMs the call may use.  algo: 0 =
 * automatic, 1 = CUDA-core kernel (every dtype), 2 = tensor-core (tcgen05)
 * kernel (bf16 and e4m3 only; HS_ERR_UNSUPPORTED otherwise).  The e4m3
 * tensor-core kernel forms each V value, code times scale, in f16 (as it does
 * the products with P), so it needs |code * scale| <= 65504 (a V scale up to
 * 146 for codes up to 448); beyond that its output is not finite.  The
 * CUDA-core kernel forms them in fp32.  max_ctas: 0 =
 * the tensor-core kernel runs one CTA on every SM; n > 0 = at most n CTAs (and
 * the automatic split for n SMs), leaving the other SMs to work launched
 * beside it, such as hs_swapin_copy.  Each of its CTAs takes a whole SM's
 * shared memory, so nothing else fits on an SM it occupies.
 * split_counters (nullable): device array of at least batch * Hkv uint32, all
 * zero before the first call that uses it.  When given, and the tensor-core
 * kernel runs every work item on a CTA of its own or cuts the work into
 * balanced chunk ranges (below), it merges the splits itself
 * ([FLL] §2.2 log-sum-exp): each split of a (request, kv head) writes its
 * partial result and counts itself in, and the split that arrives last merges
 * them all into out/lse and sets the counter back to zero; no separate merge
 * kernel is launched (otherwise one is).  Every counter is zero again when the
 * call has completed; after HS_ERR_TIMEOUT, zero the array before reusing it.
 * NULL (and the CUDA-core kernel): the merge runs as a separate kernel.
 * wait_limit_ns: bound, in nanoseconds, of every wait inside the tensor-core
 * attention (and the single-launch step) for data, a product or another role
 * of its CTA; 0 = the default of 2 s.  When a wait runs out the CTA stops all
 * of its roles, lets the copies and products it already issued finish, frees
 * its tensor memory and returns; the call's outputs are then undefined and
 * hs_get_device_error reports HS_ERR_TIMEOUT.  A limit far below a launch's
 * duration makes a wait run out on purpose (the bounded-wait test does).
 * flags: HS_ATTN_EARLY_SUMMARIES = the caller guarantees that smin/smax are
 * not written by the kernel launched just before on the same stream (they
 * were complete before it started), so the single-launch step
 * (hs_decode_step, hs_score_select_attend when fused) may start copying its
 * summary tiles while that kernel finishes, instead of after it.  Every other
 * input is still read only after it.  0 = no such guarantee.
 * Balanced chunk ranges (tensor-core kernel, split_counters given,
 * blocks_per_split 0): the 128-token chunks of every (request, kv head)'s
 * full selection are laid end to end and cut into equal runs, one per CTA,
 * so that no SM idles while another still has a whole item to go; a pair
 * whose chunks fall into several runs is merged in place as above.  The
 * library takes them when its cost estimate favours them over equal splits
 * per pair; HS_ATTN_RANGES takes them whenever they apply, HS_ATTN_NO_RANGES
 * never (hs_attn_geometry reports the choice). */
#define HS_ATTN_EARLY_SUMMARIES 1u
#define HS_ATTN_RANGES 2u
#define HS_ATTN_NO_RANGES 4u
typedef struct hs_attn_params {
  float scale;
  int32_t out_is_fp32;
  int32_t blocks_per_split;
  int32_t algo;
  int32_t max_ctas;
  uint32_t* split_counters;
  uint32_t wait_limit_ns;
  uint32_t flags;
} hs_attn_params;

/* HiSparse hot buffer ([KVS] §7).  One stream per (request, kv head) owns
 * slots_per_stream consecutive pages of the slot pool; global slot id of
 * (pair p = b*Hkv + kvh, slot s) is p*slots_per_stream + s, and that id is what
 * page_table holds, so the attention call reads the slot pool with this table.
 *   page_table  [batch][Hkv][max_blocks] device int32: slot id or -1
 *   slot_owner  [batch][Hkv][slots_per_stream] device int32: block or -1
 *   last_used   [batch][Hkv][slots_per_stream] device int32: step or -1
 *   k_slots, v_slots            device [batch*Hkv*slots_per_stream][B][D]
 *   k_slot_scales,v_slot_scales device [..][B][D/32] (e4m3 only)
 *   host_k, host_v        pinned, mapped host memory [batch][Hkv][max_blocks][B][D]
 *   host_k_scales, host_v_scales  pinned host [..][B][D/32] (e4m3 only)
 * Start state: page_table, slot_owner and last_used all -1. */
typedef struct hs_hot_buffer {
  int32_t* page_table;
  int32_t* slot_owner;
  int32_t* last_used;
  void* k_slots;
  void* v_slots;
  float* k_slot_scales;
  float* v_slot_scales;
  const void* host_k;
  const void* host_v;
  const float* host_k_scales;
  const float* host_v_scales;
  int32_t batch;
  int32_t max_blocks;
  int32_t slots_per_stream;
} hs_hot_buffer;

/* Counters accumulated (atomically added) by hs_swapin_misses; device memory. */
typedef struct hs_swap_stats {
  unsigned long long hits;
  unsigned long long misses;
  unsigned long long evictions;
  unsigned long long bytes_in;
} hs_swap_stats;

HS_API const char* hs_status_string(hs_status s);
HS_API int32_t hs_version(void);

/* Bytes of device workspace that hs_sparse_paged_decode_attn needs for this
 * geometry on the current device (split partials: per query head and split, D
 * floats of output and one float of log-sum-exp).  0 on invalid input. */
HS_API size_t hs_workspace_bytes(const hs_attn_shape* shape, int32_t batch, int32_t capacity,
                          const hs_attn_params* params);

/* How the tensor-core attention divides its work for this geometry on the
 * current device: *splits = partial results per (request, kv head) at most,
 * *chunks_per_cta = the length of a balanced chunk range (0 = equal splits
 * per pair instead).  Returns 0, or -1 on invalid input (outputs untouched).
 * Without a device it assumes 148 SMs, as hs_workspace_bytes does.  The
 * CUDA-core kernel always uses equal splits. */
HS_API int32_t hs_attn_geometry(const hs_attn_shape* shape, int32_t batch, int32_t capacity,
                                const hs_attn_params* params, int32_t* splits, int32_t* chunks_per_cta);

/* Per-block key summaries, [KVS] §5 Quest: for every request b, kv head kvh and
 * block j with first_block <= j < N_b, smin/smax[b][kvh][j][d] = min/max over
 * the block's valid tokens t in [jB, min((j+1)B, L_b)) of K[t][d].  e4m3 K is
 * dequantised (code * scale in fp32) first and the results rounded outward to
 * bf16 (min toward -inf, max toward +inf).  Other entries are not written.
 * Reading a page id outside [0, num_pages) sets HS_EBIT_PAGE_RANGE and skips
 * that block. */
HS_API hs_status hs_build_block_summaries(const hs_attn_shape* shape, const hs_paged_kv* kv,
                                   int32_t first_block, void* smin, void* smax,
                                   hs_stream_t stream);

/* Append step of a decode loop, [KVS] §5 (summaries kept current) with the
 * grouped e4m3 storage of [FLL] §2.4 + §3.2: for every (b, kvh) with
 * seq_lens[b] > 0, the token at t = seq_lens[b] - 1 (block j = t / B, row
 * t % B) is written into page page_table[b][kvh][j], and the summaries of
 * block j are widened to it, so that afterwards they equal what
 * hs_build_block_summaries computes over the block.  Row 0 starts the block's
 * summary afresh; other rows require the summary of tokens jB .. t-1 to be
 * current.  The caller updates seq_lens (to include the new token) and
 * page_table (a page for a new block) before the call.
 *   new_k, new_v  [batch][Hkv][D]  f32 for f32 K/V, bf16 otherwise; an e4m3
 *                 cache stores them quantised as hs_quantize_e4m3_g32 does
 *                 (codes into k_pages/v_pages, scales into k_scales/v_scales).
 *   The call WRITES through kv->k_pages, v_pages, k_scales and v_scales: they
 *   must point to writable device memory.
 * A block index >= max_blocks sets HS_EBIT_BLOCK_RANGE, a page id outside
 * [0, num_pages) sets HS_EBIT_PAGE_RANGE; that stream is left unchanged. */
HS_API hs_status hs_append_token(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* new_k,
                                 const void* new_v, void* smin, void* smax, hs_stream_t stream);

/* Bytes of workspace hs_score_select_topk needs when scores_opt is NULL: one
 * fp32 score per block, [batch][Hkv][max_blocks].  0 on invalid input. */
HS_API size_t hs_select_workspace_bytes(const hs_attn_shape* shape, int32_t batch, int32_t max_blocks);

/* Bound scoring and block selection, [KVS] §5 Quest + §2 sink/window:
 *   U[b][h][j] = sum_d max(q[b][h][d] * smax[b][kvh][j][d],
 *                          q[b][h][d] * smin[b][kvh][j][d])
 *   score[b][kvh][j] = max of U over the g query heads of kv head kvh
 * then sel = forced blocks + the k_scored best other blocks (score descending,
 * lower index first on ties, NaN last), ascending; all N_b blocks when that
 * covers them (ranked by the smoothed score when params->history_weight > 0).  sel_count = number selected; sel entries up to capacity past
 * the count are -1.  scores_opt (nullable) [batch][Hkv][max_blocks] f32
 * receives the scores of blocks j < N_b.  With bf16 summaries and head_dim 128
 * the bounds are computed on the tensor cores into scores_opt or, when it is
 * NULL, into workspace (hs_select_workspace_bytes bytes, else
 * HS_ERR_WORKSPACE); otherwise no workspace is needed.  Requires max_blocks
 * <= 16384. */
HS_API hs_status hs_score_select_topk(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q,
                               const void* smin, const void* smax,
                               const hs_select_params* params, int32_t* sel,
                               int32_t* sel_count, float* scores_opt, void* workspace,
                               size_t ws_bytes, hs_stream_t stream);

/* Attention over the selected blocks, [KVS] §5 (full attention on the chosen
 * blocks) with the tiled running-max/normaliser softmax of [FLL] §2.2, split
 * over CTAs and combined by a log-sum-exp merge:
 *   for query head h (kv head kvh = h / g) and the valid tokens t of the blocks
 *   in sel[b][kvh][0 .. sel_count):
 *     s_t = (q[b][h] . K[t]) * scale,  out = sum_t softmax(s)_t V[t],
 *     lse = log sum_t exp(s_t)
 * An empty selection gives out = 0 and lse = -inf.  Tokens past seq_lens[b] in
 * the last block are never read into the result.  workspace must hold
 * hs_workspace_bytes(shape, batch, capacity, params) bytes.  lse_opt nullable. */
HS_API hs_status hs_sparse_paged_decode_attn(const hs_attn_shape* shape, const hs_paged_kv* kv,
                                      const void* q, const int32_t* sel,
                                      const int32_t* sel_count, int32_t capacity,
                                      const hs_attn_params* params, void* out, float* lse_opt,
                                      void* workspace, size_t ws_bytes, hs_stream_t stream);

/* Bytes of workspace hs_score_select_attend needs: the selection's score
 * buffer (hs_select_workspace_bytes) followed by the attention's partials
 * (hs_workspace_bytes).  0 on invalid input. */
HS_API size_t hs_score_select_attend_workspace_bytes(const hs_attn_shape* shape, int32_t batch,
                                                     int32_t max_blocks, int32_t capacity,
                                                     const hs_attn_params* attn_params);

/* Selection and attention of one decode step in one call ([KVS] §5 + §2, [FLL]
 * §2.2): the same results as
 * hs_score_select_topk(shape, kv, q, smin, smax, sel_params, sel, sel_count,
 * scores_opt, ...) followed by hs_sparse_paged_decode_attn(shape, kv, q, sel,
 * sel_count, sel_params->capacity, attn_params, out, lse_opt, ...), with the
 * same argument rules, outputs and error bits as those two calls.
 * With bf16 K/V and summaries, head_dim 128, at most 8 query heads per kv
 * head, the tensor-core attention and no CTA limit (attn_params->max_ctas 0),
 * and when every (request, kv head) takes one cluster of at most 8 CTAs (its
 * 128-block score tiles and its attention splits) and all clusters fit one
 * wave, it is a single launch: each cluster scores its tiles, one CTA selects
 * and resolves the selected pages, and each CTA attends over one split of the
 * selection it received in shared memory.  Otherwise the calls' own launches
 * run in order.  workspace: hs_score_select_attend_workspace_bytes(shape,
 * batch, max_blocks, sel_params->capacity, attn_params) bytes, 16-byte
 * aligned; the selection part is used only without scores_opt. */
HS_API hs_status hs_score_select_attend(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q,
                                        const void* smin, const void* smax,
                                        const hs_select_params* sel_params, int32_t* sel,
                                        int32_t* sel_count, float* scores_opt,
                                        const hs_attn_params* attn_params, void* out, float* lse_opt,
                                        void* workspace, size_t ws_bytes, hs_stream_t stream);

/* 1 when hs_score_select_attend runs as a single launch for this geometry on
 * the current device (its clusters merge their splits themselves, with or
 * without split_counters), 0 when it runs the separate launches,
 * -1 on invalid input or without a device.  Depends on the shape, batch,
 * max_blocks, capacity and attn_params only (for page pools below 2^31
 * token rows, the tensor-core attention's own limit). */
HS_API int32_t hs_score_select_attend_fused(const hs_attn_shape* shape, int32_t batch, int32_t max_blocks,
                                            int32_t capacity, const hs_attn_params* attn_params);

/* One whole decode step of one layer: hs_append_token(shape, kv, new_k,
 * new_v, smin, smax) followed by hs_score_select_attend(shape, kv, q, smin,
 * smax, sel_params, ...), with the same argument rules, outputs and error bits
 * ([KVS] §5: the newest token's block summary covers it before the query is
 * scored; [KVS] §2 and §5 selection; [FLL] §2.2 attention).  new_k / new_v:
 * [batch][Hkv][head_dim] in the source precision (bf16, or f32 for an f32
 * cache), device, 16-byte aligned; each is written at position
 * seq_lens[b] - 1 (the caller has advanced seq_lens and given a new block its
 * page).  Where hs_score_select_attend is a single launch
 * (hs_score_select_attend_fused), the append runs inside that launch: the CTA
 * that scores the newest token's block writes the token into its page and
 * widens the block's summary in the copy it scores and in smin/smax.
 * Otherwise the append kernel runs first.  The K/V pages and smin/smax are
 * written; the page pointers of kv are used for writing here. */
HS_API hs_status hs_decode_step(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q,
                                const void* new_k, const void* new_v, void* smin, void* smax,
                                const hs_select_params* sel_params, int32_t* sel, int32_t* sel_count,
                                float* scores_opt, const hs_attn_params* attn_params, void* out,
                                float* lse_opt, void* workspace, size_t ws_bytes, hs_stream_t stream);

/* One decode step of a layer that reuses another layer's selection ([SPD]
 * §3.1: the mask chosen at a shallow layer serves the deeper ones):
 * hs_append_token(shape, kv, new_k,
 * new_v, smin, smax) followed by hs_sparse_paged_decode_attn(shape, kv, q,
 * sel, sel_count, capacity, attn_params, ...), with the same argument rules,
 * outputs and error bits; sel / sel_count are read only.  Where
 * hs_score_select_attend_fused holds for (shape, batch, max_blocks, capacity,
 * attn_params) it is one launch: the single-launch step without its scoring
 * and selection phases (the append, then the attention of each split over
 * the given selection, merged in the cluster); otherwise the append kernel and
 * the attention run in turn.  The K/V pages and smin/smax are written. */
HS_API hs_status hs_decode_step_reuse(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q,
                                      const void* new_k, const void* new_v, void* smin, void* smax,
                                      const int32_t* sel, const int32_t* sel_count, int32_t capacity,
                                      const hs_attn_params* attn_params, void* out, float* lse_opt,
                                      void* workspace, size_t ws_bytes, hs_stream_t stream);

/* HiSparse swap-in, [KVS] §7: for every (b, kvh), make each selected block
 * resident in the stream's hot slots.  Hits set last_used = step.  Misses are
 * taken in ascending block order; each goes to the lowest free slot, else to
 * the slot whose block is not in the current selection with the smallest
 * last_used (ties -> lowest slot), whose block's page_table entry becomes -1.
 * The missing page (K, V and, for e4m3, their scales) is then copied from the
 * host pool into its slot.  A selection larger than slots_per_stream sets
 * HS_EBIT_CAPACITY and leaves that stream untouched.  stats_opt (nullable,
 * device) accumulates hits, misses, evictions and bytes copied. */
HS_API hs_status hs_swapin_misses(const hs_attn_shape* shape, const hs_hot_buffer* hb,
                           const int32_t* sel, const int32_t* sel_count, int32_t capacity,
                           int32_t step, hs_swap_stats* stats_opt, hs_stream_t stream);

/* The HiSparse swap-in of hs_swapin_misses in two parts, so that the page
 * copy can overlap attention over the blocks that were already resident
 * ([KVS] §7 names the miss path as the risk to decode latency).
 * hs_swapin_plan applies the same table rule (hits stamped, misses placed in
 * ascending block order, victims chosen among slots outside the selection)
 * and writes, in the selection layout [batch][Hkv][capacity] (ascending, -1
 * padded) with counts [batch][Hkv]:
 *   hit_sel / hit_count    selected blocks that were resident on entry;
 *   miss_sel / miss_count  selected blocks just given a slot, whose pages are
 *                          not yet copied.
 * It reads no host memory; stats_opt gets hits, misses and evictions.  A
 * selection larger than slots_per_stream sets HS_EBIT_CAPACITY, leaves the
 * stream's tables untouched and writes empty lists.  The four outputs must not
 * alias sel or each other.
 * hs_swapin_copy copies the K/V pages (and e4m3 scales) of the blocks in a
 * miss list from the host pool into the slots the page table now gives them,
 * with at most max_ctas CTAs (0 = one per SM); stats_opt gets bytes_in.
 * Attention over hit_sel may run concurrently with the copy (the copy writes
 * only slots outside the selection and reads the page table); attention over
 * miss_sel must follow the copy.  Their two outputs combine with
 * hs_merge_attn_partials into the attention over the whole selection. */
HS_API hs_status hs_swapin_plan(const hs_attn_shape* shape, const hs_hot_buffer* hb, const int32_t* sel,
                                const int32_t* sel_count, int32_t capacity, int32_t step, int32_t* hit_sel,
                                int32_t* hit_count, int32_t* miss_sel, int32_t* miss_count,
                                hs_swap_stats* stats_opt, hs_stream_t stream);
/* hs_score_select_topk(shape, kv, q, smin, smax, sel_params, sel, sel_count,
 * scores_opt, workspace, ws_bytes) followed by hs_swapin_plan(shape, hb, sel,
 * sel_count, sel_params->capacity, step, hit_sel, hit_count, miss_sel,
 * miss_count, stats_opt): the same outputs, argument rules and error bits as
 * those two calls ([KVS] §5 selection, §7 hot buffer), and hb->batch must
 * equal kv->batch.  With tensor-core scoring in more than one wave and at most
 * 1024 blocks per request, each stream's plan runs in the selection's launch,
 * right after its selection. */
HS_API hs_status hs_score_select_swapin_plan(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q,
                                             const void* smin, const void* smax, const hs_select_params* sel_params,
                                             int32_t* sel, int32_t* sel_count, float* scores_opt, void* workspace,
                                             size_t ws_bytes, const hs_hot_buffer* hb, int32_t step,
                                             int32_t* hit_sel, int32_t* hit_count, int32_t* miss_sel,
                                             int32_t* miss_count, hs_swap_stats* stats_opt, hs_stream_t stream);
HS_API hs_status hs_swapin_copy(const hs_attn_shape* shape, const hs_hot_buffer* hb, const int32_t* miss_sel,
                                const int32_t* miss_count, int32_t capacity, int32_t max_ctas,
                                hs_swap_stats* stats_opt, hs_stream_t stream);

/* hs_swapin_copy, and besides the attention over the copied blocks: for each
 * (b, kvh) and each query head h of the group, over the valid tokens t (t <
 * seq_lens[b]) of the blocks in miss_sel,
 *   s_t = (q[b][h] . K[t]) * scale, out[b][h] = sum_t softmax(s)_t V[t],
 *   lse[b][h] = log sum_t exp(s_t)
 * with K/V read from the slots just filled (e4m3: code * scale).  Streams
 * with no copied token get lse = -inf and their out rows are not written.
 * q [batch][Hq][D] (f32 for f32 K/V, bf16 otherwise); out [batch][Hq][D] f32;
 * lse [batch][Hq] f32.  Together with attention over hit_sel (fp32 output)
 * and hs_merge_attn_partials this gives the attention over the selection,
 * with no separate attention launch for the misses. */
HS_API hs_status hs_swapin_copy_attend(const hs_attn_shape* shape, const hs_hot_buffer* hb, const int32_t* seq_lens,
                                       const void* q, const int32_t* miss_sel, const int32_t* miss_count,
                                       int32_t capacity, float scale, int32_t max_ctas, float* out, float* lse,
                                       hs_swap_stats* stats_opt, hs_stream_t stream);

/* Log-sum-exp merge of attention results over disjoint token sets of the same
 * queries, [FLL] §2.2 (running max and normaliser carried across tiles):
 * for each (b, h), with m = max_p lse[p][b][h],
 *   out = sum_p e^(lse_p - m) out_p / sum_p e^(lse_p - m),  lse = m + log(sum)
 * (out = 0, lse = -inf when every part is empty).
 *   outs  [parts][batch][Hq][D] f32 (each part's normalised output)
 *   lses  [parts][batch][Hq]   f32
 *   out   [batch][Hq][D] bf16, or f32 when out_is_fp32;  lse_opt [batch][Hq]. */
HS_API hs_status hs_merge_attn_partials(const hs_attn_shape* shape, int32_t batch, int32_t parts,
                                        const float* outs, const float* lses, void* out, int32_t out_is_fp32,
                                        float* lse_opt, hs_stream_t stream);

/* Grouped e4m3 quantisation of K or V rows, [FLL] §2.4 + §3.2: for each row
 * of head_dim values and each 32-channel group, scale = amax / 448 (fp32; 1
 * when amax == 0) and code = e4m3(x / scale), nearest-even, saturated to
 * +-448.  src [rows][head_dim] f32 (src_is_fp32) or bf16; codes
 * [rows][head_dim] bytes; scales [rows][head_dim/32] f32. */
HS_API hs_status hs_quantize_e4m3_g32(const void* src, int32_t src_is_fp32, int64_t rows,
                               int32_t head_dim, uint8_t* codes, float* scales,
                               hs_stream_t stream);

/* Same computation, arguments and results as hs_sparse_paged_decode_attn, for
 * callers that cannot allocate device memory.  (The pages have no counterpart
 * of this call; it exists for integration.)  Some hosts hand an operator only
 * its input and output buffers and keep the device allocator to themselves -
 * plugin and custom-operator interfaces of serving engines that plan all
 * memory ahead, or C programs that load this library without any allocator -
 * so they cannot provide the split-K workspace.  This variant keeps that
 * workspace in a fixed array of HS_NOALLOC_SCRATCH_BYTES inside the library:
 * every GPU that loads the library holds it until the process exits.
 *   - Calls whose workspace (hs_workspace_bytes for the same arguments) is
 *     larger are refused with HS_ERR_SCRATCH_LIMIT before anything runs.
 *   - The first call on a device looks up the array's device address (a
 *     cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - No cudaMalloc, cudaFree or other allocating routine is ever called.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents; the kernels overwrite every entry they read, so nothing needs
 *     clearing, but two calls that overlap on the GPU (different streams
 *     without ordering) race on it and give wrong results. */
#define HS_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
HS_API hs_status hs_sparse_paged_decode_attn_noalloc(const hs_attn_shape* shape, const hs_paged_kv* kv,
                                                     const void* q, const int32_t* sel,
                                                     const int32_t* sel_count, int32_t capacity,
                                                     const hs_attn_params* params, void* out,
                                                     float* lse_opt, hs_stream_t stream);

/* Synchronises `stream`, then reads and clears the current device's error
 * word.  Returns HS_OK when no bit was set, else, in this order of priority:
 * HS_ERR_OUT_OF_RANGE (PAGE_RANGE or BLOCK_RANGE), HS_ERR_CAPACITY,
 * HS_ERR_TIMEOUT.  bits_opt (nullable) receives the raw bits.  A failed
 * synchronisation (an earlier kernel fault) returns HS_ERR_CUDA. */
HS_API hs_status hs_get_device_error(hs_stream_t stream, uint32_t* bits_opt);

/* hs_get_device_error, also returning in timeout_opt (nullable, 11 words) the
 * first bounded wait that ran out since the last read: [0] the kernel (1 the
 * tensor-core attention, 2 the single-launch step, 3 the e4m3 attention, 4 the
 * tensor-core bound scoring; 0 = none), [1] its CTA index, [2] the wait:
 * shared-memory address of the barrier (bits 0-17), the awaited parity (bit
 * 18), the warp (bits 19-23), bit 31 set; [3..10] the progress of that CTA's
 * roles in the attention kernels (chunks issued by the copy producer, by the
 * S and by the O MMA thread, chunks done by softmax group 0 and 1, the
 * producer's work item, the softmax warps' work item and its chunk count).
 * For diagnosis only. */
HS_API hs_status hs_get_device_error_detail(hs_stream_t stream, uint32_t* bits_opt, uint32_t* timeout_opt);

#ifdef __cplusplus
}
#endif

#endif /* HS_H_ */
