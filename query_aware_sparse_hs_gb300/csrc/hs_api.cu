// C-ABI layer: argument checks, launch geometry, the per-device error word.
// Nothing here allocates device memory or synchronises, except
// hs_get_device_error.
#include <mutex>

#include "hs_internal.h"

namespace hs {
namespace {

// [0] HS_EBIT_* bits; [1..11] the first wait that ran out (kernel, CTA,
// wait, the CTA's progress); cleared by hs_get_device_error
__device__ unsigned int g_error_word[kErrorWords];

constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices];
int g_sm_count[kMaxDevices];
std::mutex g_mu;

struct Device {
  int id;
  unsigned* err;
  int sms;
};

hs_status current_device(Device* d) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return HS_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return HS_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return HS_ERR_CUDA;
    g_sm_count[dev] = sms;
    g_err_ptr[dev] = static_cast<unsigned*>(p);
  }
  d->id = dev;
  d->err = g_err_ptr[dev];
  d->sms = g_sm_count[dev];
  return HS_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

hs_status check_shape(const hs_attn_shape* s) {
  if (!s) return HS_ERR_INVALID_ARG;
  if (s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->num_q_heads % s->num_kv_heads != 0)
    return HS_ERR_INVALID_ARG;
  const int g = s->num_q_heads / s->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8 && g != 16) return HS_ERR_UNSUPPORTED;
  if (s->head_dim != 64 && s->head_dim != 128) return HS_ERR_UNSUPPORTED;
  if (s->block_size < 1 || s->block_size > 256) return HS_ERR_UNSUPPORTED;
  if (s->kv_dtype < HS_KV_F32 || s->kv_dtype > HS_KV_FP8E4M3_G32) return HS_ERR_INVALID_ARG;
  return HS_OK;
}

int elem_bytes(int kv_dtype) { return kv_dtype == HS_KV_F32 ? 4 : (kv_dtype == HS_KV_BF16 ? 2 : 1); }

hs_status check_kv(const hs_attn_shape* s, const hs_paged_kv* kv, bool need_v) {
  if (!kv || !kv->k_pages || !kv->page_table || !kv->seq_lens) return HS_ERR_INVALID_ARG;
  if (need_v && !kv->v_pages) return HS_ERR_INVALID_ARG;
  if (s->kv_dtype == HS_KV_FP8E4M3_G32 && (!kv->k_scales || (need_v && !kv->v_scales)))
    return HS_ERR_INVALID_ARG;
  if (kv->batch < 0 || kv->max_blocks < 1 || kv->num_pages < 0 || kv->num_pages > INT32_MAX)
    return HS_ERR_INVALID_ARG;
  if (!aligned(kv->k_pages, 16) || (need_v && !aligned(kv->v_pages, 16))) return HS_ERR_INVALID_ARG;
  if (!aligned(kv->page_table, 4) || !aligned(kv->seq_lens, 4)) return HS_ERR_INVALID_ARG;
  return HS_OK;
}

KvView make_view(const hs_attn_shape* s, const hs_paged_kv* kv) {
  KvView v;
  v.k_pages = kv->k_pages;
  v.v_pages = kv->v_pages;
  v.k_scales = kv->k_scales;
  v.v_scales = kv->v_scales;
  v.page_table = kv->page_table;
  v.seq_lens = kv->seq_lens;
  v.num_pages = kv->num_pages;
  v.batch = kv->batch;
  v.max_blocks = kv->max_blocks;
  v.hq = s->num_q_heads;
  v.hkv = s->num_kv_heads;
  v.group = s->num_q_heads / s->num_kv_heads;
  v.head_dim = s->head_dim;
  v.block = s->block_size;
  v.kv_dtype = s->kv_dtype;
  return v;
}

int max_selected(const hs_attn_shape* s, int max_blocks, int sink, int window, int k) {
  const int64_t B = s->block_size;
  const int64_t forced = (sink + B - 1) / B + (window > 0 ? (window + B - 1) / B + 1 : 0);
  const int64_t m = forced + k;
  return static_cast<int>(m < max_blocks ? m : max_blocks);
}

// Split-K geometry: how many selected blocks one CTA work item takes, a whole
// number of 128-token chunks where blocks are shorter.
void split_geometry(const hs_attn_shape* s, int batch, int capacity, const hs_attn_params* p,
                    int sms, int* bps_out, int* splits_out, AttnArgs* stream) {
  const int cap = capacity > 0 ? capacity : 1;
  int bps = p ? p->blocks_per_split : 0;
  if (stream) {
    stream->stream_per = 0;
    stream->stream_n = 0;
  }
  if (bps <= 0) {
    const int64_t pairs = static_cast<int64_t>(batch) * s->num_kv_heads;
    const int64_t n_sm = sms > 0 ? sms : 148;
    const int per_chunk = s->block_size < 128 ? 128 / s->block_size : 1;
    const int64_t chunks = (cap + per_chunk - 1) / per_chunk;  // 128-token chunks of a full selection
    // Splits per (request, kv head): the persistent CTAs take items in
    // rounds, so the busiest CTA runs ceil(items / SMs) items; each costs its
    // chunks plus about three chunks' worth of start-up, query load, state
    // combination and output (measured: halving the items of the 16-token
    // and e4m3 workloads pays more than the balance it costs).  The split
    // count with the least such time wins, the fewest splits on a tie.
    int64_t want = 1, best = -1;
    if (pairs > 0) {
      const int64_t top = chunks < 32 ? chunks : 32;
      for (int64_t sp = 1; sp <= top; ++sp) {
        const int64_t rounds = (pairs * sp + n_sm - 1) / n_sm;
        const int64_t cost = rounds * ((chunks + sp - 1) / sp + 3);
        if (best < 0 || cost < best) {
          best = cost;
          want = sp;
        }
      }
    }
    // Balanced chunk ranges (the tensor-core kernels, which then merge the
    // segments of a pair in place, so only with split counters): every CTA
    // takes an equal run of the pairs' chunks laid end to end, touching at
    // most ceil(per / chunks) + 1 pairs.  Taken only when cheaper than the
    // best uniform split, at a measured cost per item: three chunks for the
    // bf16 kernel, eight for the e4m3 one, whose item start and end (query
    // terms, state combination, in-place merge) are not overlapped with the
    // next item (the e4m3 workload, 128 pairs of 33 chunks: 53 us in ranges
    // of 28 chunks against 43 us in whole pairs).
    const uint32_t flags = p ? p->flags : 0u;
    if (stream && pairs > 0 && p && p->split_counters && !(flags & HS_ATTN_NO_RANGES)) {
      const int64_t total = pairs * chunks;
      const int64_t per = (total + n_sm - 1) / n_sm;
      const int64_t items = (per + chunks - 1) / chunks + 1;
      const int64_t segs = (chunks - 1 + per - 1) / per + 1;  // the most CTAs one pair's chunks touch
      const int64_t item_cost = s->kv_dtype == HS_KV_FP8E4M3_G32 ? 8 : 3;
      if (((flags & HS_ATTN_RANGES) || per + item_cost * items < best) && total + per < (int64_t(1) << 30)) {
        stream->stream_per = static_cast<int32_t>(per);
        stream->stream_n = static_cast<int32_t>(chunks);
        *bps_out = cap;
        *splits_out = static_cast<int>(segs);
        return;
      }
    }
    if (want > cap) want = cap;
    bps = static_cast<int>((cap + want - 1) / want);
    bps = ((bps + per_chunk - 1) / per_chunk) * per_chunk;
  }
  *bps_out = bps;
  *splits_out = (cap + bps - 1) / bps;
}

size_t workspace_for(const hs_attn_shape* s, int batch, int splits) {
  const size_t rows = static_cast<size_t>(batch) * s->num_q_heads * splits;
  const size_t bytes = rows * (s->head_dim + 1) * sizeof(float);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

// Partial workspace an attention call may need: the larger of the uniform
// splits and the tensor-core kernels' geometry (which kernel runs depends on
// the pointers given at call time).
size_t attn_workspace_need(const hs_attn_shape* s, int batch, int capacity, const hs_attn_params* p, int ctas) {
  int bps, splits;
  split_geometry(s, batch, capacity, p, ctas, &bps, &splits, nullptr);
  const size_t uniform = workspace_for(s, batch, splits);
  AttnArgs t;
  split_geometry(s, batch, capacity, p, ctas, &bps, &splits, &t);
  const size_t tc = workspace_for(s, batch, splits);
  return uniform > tc ? uniform : tc;
}

hs_status from_cuda(cudaError_t e) { return e == cudaSuccess ? HS_OK : HS_ERR_CUDA; }

// CTAs the tensor-core attention may run at once: the SM count, or fewer when
// the caller keeps SMs free for concurrent work.
int attn_ctas(int sms, const hs_attn_params* p) {
  return (p && p->max_ctas > 0 && p->max_ctas < sms) ? p->max_ctas : sms;
}

// Argument checks of the selection; fills the launch arguments.
hs_status prepare_select(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q, const void* smin,
                         const void* smax, const hs_select_params* params, int32_t* sel, int32_t* sel_count,
                         float* scores_opt, SelectArgs* out) {
  hs_status st = check_shape(shape);
  if (st != HS_OK) return st;
  if (!kv || !kv->seq_lens || kv->batch < 0 || kv->max_blocks < 1) return HS_ERR_INVALID_ARG;
  if (!q || !smin || !smax || !sel || !sel_count || !params) return HS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(smin, 16) || !aligned(smax, 16) || !aligned(sel, 4) ||
      !aligned(sel_count, 4) || (scores_opt && !aligned(scores_opt, 4)))
    return HS_ERR_INVALID_ARG;
  if (params->sink_tokens < 0 || params->window_tokens < 0 || params->k_scored < 0 ||
      params->capacity < 1)
    return HS_ERR_INVALID_ARG;
  if (!(params->history_weight >= 0.0f && params->history_weight < 1.0f)) return HS_ERR_INVALID_ARG;
  if (params->history_weight > 0.0f && (!params->score_history || !aligned(params->score_history, 4)))
    return HS_ERR_INVALID_ARG;
  if (kv->max_blocks > kMaxSelectBlocks) return HS_ERR_UNSUPPORTED;
  if (params->capacity < max_selected(shape, kv->max_blocks, params->sink_tokens,
                                      params->window_tokens, params->k_scored))
    return HS_ERR_CAPACITY;
  SelectArgs& a = *out;
  a.q = q;
  a.smin = smin;
  a.smax = smax;
  a.sel = sel;
  a.sel_count = sel_count;
  a.scores = scores_opt;
  a.sink_tokens = params->sink_tokens;
  a.window_tokens = params->window_tokens;
  a.k_scored = params->k_scored;
  a.capacity = params->capacity;
  a.history_weight = params->history_weight;
  a.history = params->history_weight > 0.0f ? params->score_history : nullptr;
  return HS_OK;
}

// The selection's launches: tensor-core bound scoring (into scores_opt or the
// workspace) and selection, fused into one launch where every tile of every
// pair fits one wave; else the CUDA-core scoring + selection clusters.
hs_status run_select(const KvView& v, const SelectArgs& a, const Device& d, void* workspace, size_t ws_bytes,
                     cudaStream_t cs) {
  if (score_tc_supported(v)) {
    float* buf = a.scores;
    if (!buf) {
      const size_t need = static_cast<size_t>(v.batch) * v.hkv * v.max_blocks * sizeof(float);
      if (!workspace || ws_bytes < need || !aligned(workspace, 16)) return HS_ERR_WORKSPACE;
      buf = static_cast<float*>(workspace);
    }
    if (score_select_fused_supported(v, d.sms))  // every tile of every pair in one wave: one launch
      return from_cuda(launch_score_tc(v, a.q, a.smin, a.smax, buf, d.sms, d.err, cs, &a));
    if (launch_score_tc(v, a.q, a.smin, a.smax, buf, d.sms, d.err, cs) != cudaSuccess) return HS_ERR_CUDA;
    return from_cuda(launch_select_only(v, a, buf, d.err, cs));
  }
  return from_cuda(launch_score_select(v, a, d.err, cs));
}

// Argument checks of the attention; fills the launch arguments and picks the
// tensor-core or the CUDA-core kernel.
hs_status prepare_attn(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q, const int32_t* sel,
                       const int32_t* sel_count, int32_t capacity, const hs_attn_params* params, void* out,
                       float* lse_opt, void* workspace, size_t ws_bytes, Device* dev, AttnArgs* out_args,
                       bool* use_tc) {
  hs_status st = check_kv(shape, kv, true);
  if (st != HS_OK) return st;
  if (!q || !sel || !sel_count || !out || !params || capacity < 1) return HS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(sel, 4) || !aligned(sel_count, 4))
    return HS_ERR_INVALID_ARG;
  if (params->algo < 0 || params->algo > 2 || params->blocks_per_split < 0 || params->max_ctas < 0)
    return HS_ERR_INVALID_ARG;
  if ((st = current_device(dev)) != HS_OK) return st;
  const Device& d = *dev;
  const KvView v = make_view(shape, kv);
  const int ctas = attn_ctas(d.sms, params);
  if (params->algo == 1) {
    *use_tc = false;
  } else if (params->algo == 2) {
    if (!attn_tc_supported(v)) return HS_ERR_UNSUPPORTED;
    *use_tc = true;
  } else {
    *use_tc = attn_tc_supported(v);
  }
  AttnArgs& a = *out_args;
  split_geometry(shape, kv->batch, capacity, params, ctas, &a.blocks_per_split, &a.splits, *use_tc ? &a : nullptr);
  const size_t need = workspace_for(shape, kv->batch, a.splits);
  if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 16))) return HS_ERR_WORKSPACE;
  a.sms = ctas;
  if (params->split_counters && !aligned(params->split_counters, 4)) return HS_ERR_INVALID_ARG;
  a.counters = params->split_counters;
  a.wait_ns = static_cast<uint64_t>(params->wait_limit_ns);
  a.early_summaries = (params->flags & HS_ATTN_EARLY_SUMMARIES) != 0;
  a.q = q;
  a.sel = sel;
  a.sel_count = sel_count;
  a.capacity = capacity;
  a.scale = params->scale;
  a.out_is_fp32 = params->out_is_fp32 ? 1 : 0;
  a.out = out;
  a.lse = lse_opt;
  a.ws_o = static_cast<float*>(workspace);
  a.ws_lse = a.ws_o + static_cast<size_t>(kv->batch) * shape->num_q_heads * a.splits * shape->head_dim;
  return HS_OK;
}

}  // namespace
}  // namespace hs

using namespace hs;

extern "C" {

const char* hs_status_string(hs_status s) {
  switch (s) {
    case HS_OK: return "ok";
    case HS_ERR_INVALID_ARG: return "invalid argument";
    case HS_ERR_UNSUPPORTED: return "unsupported configuration";
    case HS_ERR_CUDA: return "CUDA runtime error";
    case HS_ERR_OUT_OF_RANGE: return "page id or block index out of range";
    case HS_ERR_CAPACITY: return "selection larger than capacity";
    case HS_ERR_TIMEOUT: return "device wait timed out";
    case HS_ERR_WORKSPACE: return "workspace too small";
    case HS_ERR_SCRATCH_LIMIT: return "needs more than the fixed scratch of the no-allocation call";
  }
  return "unknown status";
}

int32_t hs_version(void) { return 1; }

int32_t hs_attn_geometry(const hs_attn_shape* shape, int32_t batch, int32_t capacity,
                         const hs_attn_params* params, int32_t* splits, int32_t* chunks_per_cta) {
  if (check_shape(shape) != HS_OK || batch < 0 || capacity < 1 || !params || !splits || !chunks_per_cta) return -1;
  if (params->blocks_per_split < 0 || params->max_ctas < 0) return -1;
  Device d{};
  int sms = 148;  // without a device: as hs_workspace_bytes
  if (current_device(&d) == HS_OK) sms = d.sms;
  AttnArgs a;
  split_geometry(shape, batch, capacity, params, attn_ctas(sms, params), &a.blocks_per_split, &a.splits, &a);
  *splits = a.splits;
  *chunks_per_cta = a.stream_per;
  return 0;
}

size_t hs_workspace_bytes(const hs_attn_shape* shape, int32_t batch, int32_t capacity,
                          const hs_attn_params* params) {
  if (check_shape(shape) != HS_OK || batch < 0 || capacity < 0) return 0;
  Device d{};
  int sms = 148;
  if (current_device(&d) == HS_OK) sms = d.sms;
  return attn_workspace_need(shape, batch, capacity, params, attn_ctas(sms, params));
}

hs_status hs_build_block_summaries(const hs_attn_shape* shape, const hs_paged_kv* kv,
                                   int32_t first_block, void* smin, void* smax,
                                   hs_stream_t stream) {
  hs_status st = check_shape(shape);
  if (st != HS_OK) return st;
  if ((st = check_kv(shape, kv, false)) != HS_OK) return st;
  if (!smin || !smax || !aligned(smin, 16) || !aligned(smax, 16)) return HS_ERR_INVALID_ARG;
  if (first_block < 0 || first_block > kv->max_blocks) return HS_ERR_INVALID_ARG;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  const KvView v = make_view(shape, kv);
  return from_cuda(launch_summaries(v, first_block, smin, smax, d.err, d.sms,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

hs_status hs_append_token(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* new_k,
                          const void* new_v, void* smin, void* smax, hs_stream_t stream) {
  hs_status st = check_shape(shape);
  if (st != HS_OK) return st;
  if ((st = check_kv(shape, kv, true)) != HS_OK) return st;
  if (!new_k || !new_v || !smin || !smax) return HS_ERR_INVALID_ARG;
  if (!aligned(new_k, 16) || !aligned(new_v, 16) || !aligned(smin, 16) || !aligned(smax, 16))
    return HS_ERR_INVALID_ARG;
  if (static_cast<int64_t>(kv->batch) * shape->num_kv_heads > INT32_MAX) return HS_ERR_UNSUPPORTED;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  const KvView v = make_view(shape, kv);
  return from_cuda(launch_append(v, new_k, new_v, smin, smax, d.err, reinterpret_cast<cudaStream_t>(stream)));
}

hs_status hs_score_select_topk(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q,
                               const void* smin, const void* smax,
                               const hs_select_params* params, int32_t* sel,
                               int32_t* sel_count, float* scores_opt, void* workspace,
                               size_t ws_bytes, hs_stream_t stream) {
  SelectArgs a;
  hs_status st = prepare_select(shape, kv, q, smin, smax, params, sel, sel_count, scores_opt, &a);
  if (st != HS_OK) return st;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  return run_select(make_view(shape, kv), a, d, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t hs_select_workspace_bytes(const hs_attn_shape* shape, int32_t batch, int32_t max_blocks) {
  if (check_shape(shape) != HS_OK || batch < 0 || max_blocks < 0) return 0;
  const size_t bytes = static_cast<size_t>(batch) * shape->num_kv_heads * max_blocks * sizeof(float);
  return (bytes + 255) & ~static_cast<size_t>(255);
}

hs_status hs_sparse_paged_decode_attn(const hs_attn_shape* shape, const hs_paged_kv* kv,
                                      const void* q, const int32_t* sel,
                                      const int32_t* sel_count, int32_t capacity,
                                      const hs_attn_params* params, void* out, float* lse_opt,
                                      void* workspace, size_t ws_bytes, hs_stream_t stream) {
  hs_status st = check_shape(shape);
  if (st != HS_OK) return st;
  Device d;
  AttnArgs a;
  bool use_tc = false;
  st = prepare_attn(shape, kv, q, sel, sel_count, capacity, params, out, lse_opt, workspace, ws_bytes, &d, &a,
                    &use_tc);
  if (st != HS_OK) return st;
  const KvView v = make_view(shape, kv);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = use_tc ? launch_attn_tc(v, a, d.err, s) : launch_attn_simt(v, a, d.err, s);
  if (e != cudaSuccess) return HS_ERR_CUDA;
  if (a.merged) return HS_OK;
  return from_cuda(launch_merge(v, a, s));
}

size_t hs_score_select_attend_workspace_bytes(const hs_attn_shape* shape, int32_t batch, int32_t max_blocks,
                                              int32_t capacity, const hs_attn_params* params) {
  if (check_shape(shape) != HS_OK || batch < 0 || max_blocks < 0 || capacity < 0) return 0;
  return hs_select_workspace_bytes(shape, batch, max_blocks) + hs_workspace_bytes(shape, batch, capacity, params);
}

int32_t hs_score_select_attend_fused(const hs_attn_shape* shape, int32_t batch, int32_t max_blocks,
                                     int32_t capacity, const hs_attn_params* params) {
  if (check_shape(shape) != HS_OK || batch < 0 || max_blocks < 1 || capacity < 1 || !params) return -1;
  if (params->algo < 0 || params->algo > 2 || params->blocks_per_split < 0 || params->max_ctas < 0) return -1;
  Device d;
  if (current_device(&d) != HS_OK) return -1;
  if (params->algo == 1 || attn_ctas(d.sms, params) != d.sms) return 0;
  KvView v{};
  v.batch = batch;
  v.max_blocks = max_blocks;
  v.num_pages = 1;
  v.hq = shape->num_q_heads;
  v.hkv = shape->num_kv_heads;
  v.group = shape->num_q_heads / shape->num_kv_heads;
  v.head_dim = shape->head_dim;
  v.block = shape->block_size;
  v.kv_dtype = shape->kv_dtype;
  if (!attn_tc_supported(v)) return 0;
  AttnArgs a;
  split_geometry(shape, batch, capacity, params, d.sms, &a.blocks_per_split, &a.splits, &a);
  return score_select_attn_supported(v, a, d.sms) ? 1 : 0;
}

}  // extern "C"

namespace hs {
namespace {

// Selection and attention of one step, preceded by the append of the newest
// token when new_k is given: one launch where the geometry allows, else the
// separate launches in order.
hs_status select_attend(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q, const void* new_k,
                        const void* new_v, const void* smin, const void* smax, const hs_select_params* sel_params,
                        int32_t* sel, int32_t* sel_count, float* scores_opt, const hs_attn_params* attn_params,
                        void* out, float* lse_opt, void* workspace, size_t ws_bytes, cudaStream_t s) {
  SelectArgs sa;
  hs_status st = prepare_select(shape, kv, q, smin, smax, sel_params, sel, sel_count, scores_opt, &sa);
  if (st != HS_OK) return st;
  if (new_k && (!new_v || !aligned(new_k, 16) || !aligned(new_v, 16))) return HS_ERR_INVALID_ARG;
  if (new_k && static_cast<int64_t>(kv->batch) * shape->num_kv_heads > INT32_MAX) return HS_ERR_UNSUPPORTED;
  // workspace: the selection's score buffer first, the attention's partials after it
  const size_t sw = hs_select_workspace_bytes(shape, kv->batch, kv->max_blocks);
  if (sw > 0 && (!workspace || ws_bytes < sw || !aligned(workspace, 16))) return HS_ERR_WORKSPACE;
  void* aws = workspace ? static_cast<uint8_t*>(workspace) + sw : nullptr;
  const size_t aws_bytes = workspace ? ws_bytes - sw : 0;
  Device d;
  AttnArgs a;
  bool use_tc = false;
  st = prepare_attn(shape, kv, q, sel, sel_count, sel_params->capacity, attn_params, out, lse_opt, aws, aws_bytes,
                    &d, &a, &use_tc);
  if (st != HS_OK) return st;
  const KvView v = make_view(shape, kv);
  if (use_tc && a.sms == d.sms && score_select_attn_supported(v, a, d.sms)) {
    if (launch_score_select_attn(v, smin, smax, sa, a, d.err, s, new_k, new_v) != cudaSuccess) return HS_ERR_CUDA;
  } else {
    if (new_k && launch_append(v, new_k, new_v, const_cast<void*>(smin), const_cast<void*>(smax), d.err, s) !=
                     cudaSuccess)
      return HS_ERR_CUDA;
    if ((st = run_select(v, sa, d, workspace, sw, s)) != HS_OK) return st;
    cudaError_t e = use_tc ? launch_attn_tc(v, a, d.err, s) : launch_attn_simt(v, a, d.err, s);
    if (e != cudaSuccess) return HS_ERR_CUDA;
  }
  if (a.merged) return HS_OK;
  return from_cuda(launch_merge(v, a, s));
}

}  // namespace
}  // namespace hs

extern "C" {

hs_status hs_score_select_attend(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q,
                                 const void* smin, const void* smax, const hs_select_params* sel_params,
                                 int32_t* sel, int32_t* sel_count, float* scores_opt,
                                 const hs_attn_params* attn_params, void* out, float* lse_opt, void* workspace,
                                 size_t ws_bytes, hs_stream_t stream) {
  return select_attend(shape, kv, q, nullptr, nullptr, smin, smax, sel_params, sel, sel_count, scores_opt,
                       attn_params, out, lse_opt, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

hs_status hs_decode_step(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q, const void* new_k,
                         const void* new_v, void* smin, void* smax, const hs_select_params* sel_params, int32_t* sel,
                         int32_t* sel_count, float* scores_opt, const hs_attn_params* attn_params, void* out,
                         float* lse_opt, void* workspace, size_t ws_bytes, hs_stream_t stream) {
  hs_status st = check_shape(shape);
  if (st != HS_OK) return st;
  if ((st = check_kv(shape, kv, true)) != HS_OK) return st;
  if (!new_k || !new_v) return HS_ERR_INVALID_ARG;
  return select_attend(shape, kv, q, new_k, new_v, smin, smax, sel_params, sel, sel_count, scores_opt, attn_params,
                       out, lse_opt, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

hs_status hs_decode_step_reuse(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q, const void* new_k,
                               const void* new_v, void* smin, void* smax, const int32_t* sel,
                               const int32_t* sel_count, int32_t capacity, const hs_attn_params* attn_params,
                               void* out, float* lse_opt, void* workspace, size_t ws_bytes, hs_stream_t stream) {
  using namespace hs;
  hs_status st = check_shape(shape);
  if (st != HS_OK) return st;
  if ((st = check_kv(shape, kv, true)) != HS_OK) return st;
  if (!new_k || !new_v || !aligned(new_k, 16) || !aligned(new_v, 16)) return HS_ERR_INVALID_ARG;
  if (!smin || !smax || !aligned(smin, 16) || !aligned(smax, 16)) return HS_ERR_INVALID_ARG;
  if (static_cast<int64_t>(kv->batch) * shape->num_kv_heads > INT32_MAX) return HS_ERR_UNSUPPORTED;
  Device d;
  AttnArgs a;
  bool use_tc = false;
  st = prepare_attn(shape, kv, q, sel, sel_count, capacity, attn_params, out, lse_opt, workspace, ws_bytes, &d, &a,
                    &use_tc);
  if (st != HS_OK) return st;
  const KvView v = make_view(shape, kv);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (use_tc && a.sms == d.sms && score_select_attn_supported(v, a, d.sms)) {
    SelectArgs sa{};
    sa.q = q;
    sa.smin = smin;
    sa.smax = smax;
    sa.sel = const_cast<int32_t*>(sel);  // read only: the reused selection
    sa.sel_count = const_cast<int32_t*>(sel_count);
    sa.capacity = capacity;
    if (launch_score_select_attn(v, smin, smax, sa, a, d.err, s, new_k, new_v, true) != cudaSuccess) return HS_ERR_CUDA;
  } else {
    if (launch_append(v, new_k, new_v, smin, smax, d.err, s) != cudaSuccess) return HS_ERR_CUDA;
    cudaError_t e = use_tc ? launch_attn_tc(v, a, d.err, s) : launch_attn_simt(v, a, d.err, s);
    if (e != cudaSuccess) return HS_ERR_CUDA;
  }
  if (a.merged) return HS_OK;
  return from_cuda(launch_merge(v, a, s));
}

static hs_status device_address(const void* p, const void** out) {
  if (!p) {
    *out = nullptr;
    return HS_OK;
  }
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_INVALID_ARG;
  }
  if (at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
    if (!at.devicePointer) return HS_ERR_INVALID_ARG;
    *out = at.devicePointer;
    return HS_OK;
  }
  return HS_ERR_INVALID_ARG;  // pageable memory that was never pinned
}

// Checks a hot buffer and builds the kernels' view of it (host pool pointers
// translated to their device addresses).
static hs_status hot_view(const hs_attn_shape* shape, const hs_hot_buffer* hb, HotView* v) {
  hs_status st = check_shape(shape);
  if (st != HS_OK) return st;
  if (!hb) return HS_ERR_INVALID_ARG;
  if (!hb->page_table || !hb->slot_owner || !hb->last_used || !hb->k_slots || !hb->v_slots ||
      !hb->host_k || !hb->host_v)
    return HS_ERR_INVALID_ARG;
  const bool fp8 = shape->kv_dtype == HS_KV_FP8E4M3_G32;
  if (fp8 && (!hb->k_slot_scales || !hb->v_slot_scales || !hb->host_k_scales || !hb->host_v_scales))
    return HS_ERR_INVALID_ARG;
  if (hb->batch < 0 || hb->max_blocks < 1 || hb->slots_per_stream < 1 || hb->slots_per_stream > 1024)
    return HS_ERR_INVALID_ARG;
  if (static_cast<int64_t>(hb->batch) * shape->num_kv_heads * hb->slots_per_stream > INT32_MAX)
    return HS_ERR_UNSUPPORTED;
  const int64_t page_bytes = static_cast<int64_t>(shape->block_size) * shape->head_dim * elem_bytes(shape->kv_dtype);
  if (page_bytes % 16 != 0) return HS_ERR_UNSUPPORTED;
  if (!aligned(hb->k_slots, 16) || !aligned(hb->v_slots, 16) || !aligned(hb->host_k, 16) ||
      !aligned(hb->host_v, 16))
    return HS_ERR_INVALID_ARG;
  v->page_table = hb->page_table;
  v->slot_owner = hb->slot_owner;
  v->last_used = hb->last_used;
  v->k_slots = hb->k_slots;
  v->v_slots = hb->v_slots;
  v->k_slot_scales = hb->k_slot_scales;
  v->v_slot_scales = hb->v_slot_scales;
  const void* p;
  if ((st = device_address(hb->host_k, &p)) != HS_OK) return st;
  v->host_k = p;
  if ((st = device_address(hb->host_v, &p)) != HS_OK) return st;
  v->host_v = p;
  if ((st = device_address(hb->host_k_scales, &p)) != HS_OK) return st;
  v->host_k_scales = static_cast<const float*>(p);
  if ((st = device_address(hb->host_v_scales, &p)) != HS_OK) return st;
  v->host_v_scales = static_cast<const float*>(p);
  v->batch = hb->batch;
  v->hkv = shape->num_kv_heads;
  v->max_blocks = hb->max_blocks;
  v->slots = hb->slots_per_stream;
  v->block = shape->block_size;
  v->head_dim = shape->head_dim;
  v->kv_dtype = shape->kv_dtype;
  return HS_OK;
}

hs_status hs_swapin_misses(const hs_attn_shape* shape, const hs_hot_buffer* hb,
                           const int32_t* sel, const int32_t* sel_count, int32_t capacity,
                           int32_t step, hs_swap_stats* stats_opt, hs_stream_t stream) {
  if (!sel || !sel_count || capacity < 1) return HS_ERR_INVALID_ARG;
  HotView v;
  hs_status st = hot_view(shape, hb, &v);
  if (st != HS_OK) return st;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  return from_cuda(launch_swapin(v, sel, sel_count, capacity, step, stats_opt, d.err,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

hs_status hs_swapin_plan(const hs_attn_shape* shape, const hs_hot_buffer* hb, const int32_t* sel,
                         const int32_t* sel_count, int32_t capacity, int32_t step, int32_t* hit_sel,
                         int32_t* hit_count, int32_t* miss_sel, int32_t* miss_count,
                         hs_swap_stats* stats_opt, hs_stream_t stream) {
  if (!sel || !sel_count || capacity < 1 || !hit_sel || !hit_count || !miss_sel || !miss_count)
    return HS_ERR_INVALID_ARG;
  if (hit_sel == sel || miss_sel == sel || hit_sel == miss_sel) return HS_ERR_INVALID_ARG;
  HotView v;
  hs_status st = hot_view(shape, hb, &v);
  if (st != HS_OK) return st;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  return from_cuda(launch_swapin_plan(v, sel, sel_count, capacity, step, hit_sel, hit_count, miss_sel, miss_count,
                                      stats_opt, d.err, reinterpret_cast<cudaStream_t>(stream)));
}

hs_status hs_score_select_swapin_plan(const hs_attn_shape* shape, const hs_paged_kv* kv, const void* q,
                                      const void* smin, const void* smax, const hs_select_params* sel_params,
                                      int32_t* sel, int32_t* sel_count, float* scores_opt, void* workspace,
                                      size_t ws_bytes, const hs_hot_buffer* hb, int32_t step, int32_t* hit_sel,
                                      int32_t* hit_count, int32_t* miss_sel, int32_t* miss_count,
                                      hs_swap_stats* stats_opt, hs_stream_t stream) {
  SelectArgs a;
  hs_status st = prepare_select(shape, kv, q, smin, smax, sel_params, sel, sel_count, scores_opt, &a);
  if (st != HS_OK) return st;
  if (!hit_sel || !hit_count || !miss_sel || !miss_count) return HS_ERR_INVALID_ARG;
  if (hit_sel == sel || miss_sel == sel || hit_sel == miss_sel) return HS_ERR_INVALID_ARG;
  HotView hv;
  if ((st = hot_view(shape, hb, &hv)) != HS_OK) return st;
  if (hb->batch != kv->batch) return HS_ERR_INVALID_ARG;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  const KvView v = make_view(shape, kv);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (score_tc_supported(v) && !score_select_fused_supported(v, d.sms) && select_plan_supported(v, hv)) {
    float* buf = a.scores;
    if (!buf) {
      const size_t need = static_cast<size_t>(v.batch) * v.hkv * v.max_blocks * sizeof(float);
      if (!workspace || ws_bytes < need || !aligned(workspace, 16)) return HS_ERR_WORKSPACE;
      buf = static_cast<float*>(workspace);
    }
    if (launch_score_tc(v, a.q, a.smin, a.smax, buf, d.sms, d.err, cs) != cudaSuccess) return HS_ERR_CUDA;
    const PlanArgs pa{hv, step, hit_sel, hit_count, miss_sel, miss_count, stats_opt};
    return from_cuda(launch_select_plan(v, a, buf, pa, d.err, cs));
  }
  if ((st = run_select(v, a, d, workspace, ws_bytes, cs)) != HS_OK) return st;
  return from_cuda(launch_swapin_plan(hv, sel, sel_count, a.capacity, step, hit_sel, hit_count, miss_sel, miss_count,
                                      stats_opt, d.err, cs));
}

hs_status hs_swapin_copy(const hs_attn_shape* shape, const hs_hot_buffer* hb, const int32_t* miss_sel,
                         const int32_t* miss_count, int32_t capacity, int32_t max_ctas,
                         hs_swap_stats* stats_opt, hs_stream_t stream) {
  if (!miss_sel || !miss_count || capacity < 1 || max_ctas < 0) return HS_ERR_INVALID_ARG;
  HotView v;
  hs_status st = hot_view(shape, hb, &v);
  if (st != HS_OK) return st;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  const int ctas = max_ctas > 0 ? max_ctas : d.sms;
  return from_cuda(launch_swapin_copy(v, miss_sel, miss_count, capacity, ctas, nullptr, stats_opt, d.err,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

hs_status hs_swapin_copy_attend(const hs_attn_shape* shape, const hs_hot_buffer* hb, const int32_t* seq_lens,
                                const void* q, const int32_t* miss_sel, const int32_t* miss_count, int32_t capacity,
                                float scale, int32_t max_ctas, float* out, float* lse, hs_swap_stats* stats_opt,
                                hs_stream_t stream) {
  if (!miss_sel || !miss_count || capacity < 1 || max_ctas < 0 || !seq_lens || !q || !out || !lse)
    return HS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(seq_lens, 4)) return HS_ERR_INVALID_ARG;
  HotView v;
  hs_status st = hot_view(shape, hb, &v);
  if (st != HS_OK) return st;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  MissAttnArgs a;
  a.q = q;
  a.seq_lens = seq_lens;
  a.out = out;
  a.lse = lse;
  a.scale = scale;
  a.hq = shape->num_q_heads;
  const int ctas = max_ctas > 0 ? max_ctas : d.sms;
  return from_cuda(launch_swapin_copy(v, miss_sel, miss_count, capacity, ctas, &a, stats_opt, d.err,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

hs_status hs_merge_attn_partials(const hs_attn_shape* shape, int32_t batch, int32_t parts, const float* outs,
                                 const float* lses, void* out, int32_t out_is_fp32, float* lse_opt,
                                 hs_stream_t stream) {
  hs_status st = check_shape(shape);
  if (st != HS_OK) return st;
  if (batch < 0 || parts < 1 || !outs || !lses || !out) return HS_ERR_INVALID_ARG;
  if (!aligned(outs, 4) || !aligned(lses, 4) || !aligned(out, out_is_fp32 ? 4 : 2)) return HS_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * shape->num_q_heads > INT32_MAX) return HS_ERR_UNSUPPORTED;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  return from_cuda(launch_merge_parts(batch * shape->num_q_heads, shape->head_dim, parts, outs, lses, out,
                                      out_is_fp32 ? 1 : 0, lse_opt, reinterpret_cast<cudaStream_t>(stream)));
}

hs_status hs_quantize_e4m3_g32(const void* src, int32_t src_is_fp32, int64_t rows,
                               int32_t head_dim, uint8_t* codes, float* scales,
                               hs_stream_t stream) {
  if (!src || !codes || !scales || rows < 0) return HS_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return HS_ERR_UNSUPPORTED;
  if (rows / 8 >= INT32_MAX) return HS_ERR_UNSUPPORTED;
  Device d;
  hs_status st = current_device(&d);
  if (st != HS_OK) return st;
  return from_cuda(launch_quantize(src, src_is_fp32 != 0, rows, head_dim, codes, scales,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

hs_status hs_get_device_error(hs_stream_t stream, uint32_t* bits_opt) {
  return hs_get_device_error_detail(stream, bits_opt, nullptr);
}

hs_status hs_get_device_error_detail(hs_stream_t stream, uint32_t* bits_opt, uint32_t* timeout_opt) {
  Device d;
  hs_status st = current_device(&d);
  if (st != HS_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return HS_ERR_CUDA;
  unsigned word[kErrorWords] = {};
  if (cudaMemcpyAsync(word, d.err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return HS_ERR_CUDA;
  if (cudaMemsetAsync(d.err, 0, sizeof(word), s) != cudaSuccess) return HS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return HS_ERR_CUDA;
  const unsigned bits = word[0];
  if (bits_opt) *bits_opt = bits;
  if (timeout_opt)
    for (int i = 1; i < kErrorWords; ++i) timeout_opt[i - 1] = word[i];
  if (bits & (HS_EBIT_PAGE_RANGE | HS_EBIT_BLOCK_RANGE)) return HS_ERR_OUT_OF_RANGE;
  if (bits & HS_EBIT_CAPACITY) return HS_ERR_CAPACITY;
  if (bits & HS_EBIT_TIMEOUT) return HS_ERR_TIMEOUT;
  return HS_OK;
}

}  // extern "C"

// ---- attention without caller-provided workspace ----------------------------
// For hosts that cannot allocate device memory: the split-K workspace lives in
// this fixed device array instead.  Host code must not use the array's name as
// a pointer (it is only a host-side stand-in); its device address is looked up
// once per device with cudaGetSymbolAddress and passed to the kernels.
namespace hs {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[HS_NOALLOC_SCRATCH_BYTES];
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

hs_status scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return HS_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return HS_OK;
}

}  // namespace
}  // namespace hs

extern "C" hs_status hs_sparse_paged_decode_attn_noalloc(const hs_attn_shape* shape, const hs_paged_kv* kv,
                                                         const void* q, const int32_t* sel,
                                                         const int32_t* sel_count, int32_t capacity,
                                                         const hs_attn_params* params, void* out,
                                                         float* lse_opt, hs_stream_t stream) {
  hs_status st = check_shape(shape);
  if (st != HS_OK) return st;
  if (!kv || !params || capacity < 1 || kv->batch < 0) return HS_ERR_INVALID_ARG;
  if (params->blocks_per_split < 0) return HS_ERR_INVALID_ARG;
  Device d;
  if ((st = current_device(&d)) != HS_OK) return st;
  const size_t need = attn_workspace_need(shape, kv->batch, capacity, params, attn_ctas(d.sms, params));
  if (need > HS_NOALLOC_SCRATCH_BYTES) return HS_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if ((st = scratch_address(d.id, &scratch)) != HS_OK) return st;
  return hs_sparse_paged_decode_attn(shape, kv, q, sel, sel_count, capacity, params, out, lse_opt, scratch,
                                     HS_NOALLOC_SCRATCH_BYTES, stream);
}
