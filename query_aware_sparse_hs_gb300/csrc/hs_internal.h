// Launchers implemented by the kernel translation units and called by the
// C-ABI layer (hs_api.cu) after argument checks.
#pragma once

#include "hs_common.cuh"

namespace hs {

struct SelectArgs {
  const void* q;
  const void* smin;
  const void* smax;
  int32_t* sel;
  int32_t* sel_count;
  float* scores;  // nullable
  int32_t sink_tokens, window_tokens, k_scored, capacity;
  float history_weight;  // 0: no smoothing
  float* history;        // [batch][Hkv][max_blocks] smoothed scores of the previous step (NaN = none)
};

struct AttnArgs {
  uint32_t* counters = nullptr;  // split arrival counters (tensor-core kernel merges in place)
  const void* q;
  const int32_t* sel;
  const int32_t* sel_count;
  int32_t capacity;
  float scale;
  int32_t out_is_fp32;
  void* out;
  float* lse;   // nullable
  float* ws_o;  // [batch][hq][splits][D]
  float* ws_lse;  // [batch][hq][splits]
  int32_t blocks_per_split;
  int32_t splits;
  // balanced chunk ranges (tensor-core kernels, with split counters): the
  // pairs' chunks end to end, stream_per per CTA; 0 = uniform splits
  int32_t stream_per = 0;
  int32_t stream_n = 0;  // chunks of a full selection per pair
  int32_t sms;  // multiprocessors of the current device (persistent grid size)
  int32_t merged = 0;  // set by a launcher that already wrote out / lse (fused merge)
  uint64_t wait_ns = 0;  // bound of the tensor-core kernels' waits (0: the default 2 s)
  bool early_summaries = false;  // HS_ATTN_EARLY_SUMMARIES
};

struct HotView {
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
  int32_t batch, hkv, max_blocks, slots, block, head_dim, kv_dtype;
};

// Newest token of every stream into its page + widening of its block's summary.
cudaError_t launch_append(const KvView& kv, const void* new_k, const void* new_v, void* smin, void* smax,
                          unsigned* err, cudaStream_t st);
cudaError_t launch_summaries(const KvView& kv, int first_block, void* smin, void* smax,
                             unsigned* err, int sms, cudaStream_t st);
cudaError_t launch_score_select(const KvView& kv, const SelectArgs& a, unsigned* err,
                                cudaStream_t st);
bool score_tc_supported(const KvView& kv);
// fuse (nullable): score and select in one launch, one cluster per (request,
// kv head); only where score_select_fused_supported.
cudaError_t launch_score_tc(const KvView& kv, const void* q, const void* smin, const void* smax, float* scores,
                            int sms, unsigned* err, cudaStream_t st, const SelectArgs* fuse = nullptr);
bool score_select_fused_supported(const KvView& kv, int sms);
cudaError_t launch_select_only(const KvView& kv, const SelectArgs& a, const float* scores, unsigned* err,
                               cudaStream_t st);
cudaError_t launch_attn_simt(const KvView& kv, const AttnArgs& a, unsigned* err, cudaStream_t st);
cudaError_t launch_attn_tc(const KvView& kv, AttnArgs& a, unsigned* err, cudaStream_t st);
bool attn_tc_supported(const KvView& kv);
// Bound scoring, selection and tensor-core attention in one cluster launch
// (bf16, head_dim 128, g <= 8, every pair in one wave of at most 8 CTAs).
bool score_select_attn_supported(const KvView& kv, const AttnArgs& a, int sms);
// new_k / new_v (nullable): the newest token of every pair is appended first
// (written into its page, its block's summary widened), as launch_append does.
// reuse: no scoring or selection; the attention takes the selection in
// sa.sel / sa.sel_count (capacity sa.capacity) as given.
cudaError_t launch_score_select_attn(const KvView& kv, const void* smin, const void* smax, const SelectArgs& sa,
                                     AttnArgs& a, unsigned* err, cudaStream_t st, const void* new_k = nullptr,
                                     const void* new_v = nullptr, bool reuse = false);
// LSE merge of `parts` partial results laid out [parts][rows][D] and [parts][rows].
cudaError_t launch_merge_parts(int rows, int head_dim, int parts, const float* outs, const float* lses, void* out,
                               int out_f32, float* lse_out, cudaStream_t st);
cudaError_t launch_merge(const KvView& kv, const AttnArgs& a, cudaStream_t st);
cudaError_t launch_swapin(const HotView& hb, const int32_t* sel, const int32_t* sel_count,
                          int capacity, int step, hs_swap_stats* stats, unsigned* err,
                          cudaStream_t st);
cudaError_t launch_swapin_plan(const HotView& hb, const int32_t* sel, const int32_t* sel_count, int capacity,
                               int step, int32_t* hit_sel, int32_t* hit_count, int32_t* miss_sel,
                               int32_t* miss_count, hs_swap_stats* stats, unsigned* err, cudaStream_t st);
// The hot-buffer plan run by the selection launch right after each stream's
// selection (the same outputs as launch_swapin_plan).
struct PlanArgs {
  HotView hb;
  int32_t step;
  int32_t* hit_sel;
  int32_t* hit_count;
  int32_t* miss_sel;
  int32_t* miss_count;
  hs_swap_stats* stats;  // nullable
};
// false when the geometry needs the separate launches (more than 1024 blocks
// per request or slots per stream)
bool select_plan_supported(const KvView& kv, const HotView& hb);
cudaError_t launch_select_plan(const KvView& kv, const SelectArgs& a, const float* scores, const PlanArgs& pa,
                               unsigned* err, cudaStream_t st);
// Attention over the blocks a page copy brings in (q rows of the stream's query heads).
struct MissAttnArgs {
  const void* q;
  const int32_t* seq_lens;
  float* out;
  float* lse;
  float scale;
  int hq;
};
cudaError_t launch_swapin_copy(const HotView& hb, const int32_t* miss_sel, const int32_t* miss_count,
                               int capacity, int ctas, const MissAttnArgs* attn, hs_swap_stats* stats, unsigned* err,
                               cudaStream_t st);
cudaError_t launch_quantize(const void* src, bool src_f32, int64_t rows, int head_dim,
                            uint8_t* codes, float* scales, cudaStream_t st);

}  // namespace hs
