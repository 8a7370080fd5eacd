// Bound scoring + block selection ("KV 稀疏化" wiki §5 Quest, §2 sink/window;
// SparDA §4.2 selector).
//
// One thread-block cluster of kSelectCluster CTAs per (request, kv head).  Each
// CTA scores a contiguous slice of the request's blocks against the g query
// heads of the kv head and stores the scores straight into the shared memory
// of CTA rank 0 (distributed shared memory), so the selection never round-trips
// through global memory.  After the cluster barrier, rank 0 finds the k-th
// largest score of the non-forced blocks with an 8-bit radix select in shared
// memory, then writes forced + chosen blocks in ascending order (select_pair.cuh).
//
// Bound:  U_h(j) = sum_d max(q_hd * smax_jd, q_hd * smin_jd)
//               = sum_d q+_hd * smax_jd + q-_hd * smin_jd,  q+ = max(q,0), q- = min(q,0)
// (term by term identical in floating point because smax >= smin and rounding
// is monotonic); the block score is the max of U over the kv head's query heads.
#include <cooperative_groups.h>

#include "hs_internal.h"
#include "select_pair.cuh"
#include "swapin_plan.cuh"

namespace cg = cooperative_groups;

namespace hs {
namespace {

using namespace sel;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int C, bool F32>
__device__ __forceinline__ void load_summary(const void* base, int64_t off, float (&x)[C]) {
  if constexpr (F32) {
    const float* p = static_cast<const float*>(base) + off;
    if constexpr (C == 4) {
      float4 v = __ldg(reinterpret_cast<const float4*>(p));
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
      float2 v = __ldg(reinterpret_cast<const float2*>(p));
      x[0] = v.x; x[1] = v.y;
    }
  } else {
    const uint16_t* p = static_cast<const uint16_t*>(base) + off;
    if constexpr (C == 4) {
      uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
      x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
      x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
    } else {
      uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(p));
      x[0] = __uint_as_float(v << 16); x[1] = __uint_as_float(v & 0xffff0000u);
    }
  }
}

template <int C, int G, bool F32>
__global__ void __cluster_dims__(kSelectCluster, 1, 1) __launch_bounds__(kThreads, (G * C <= 32) ? 2 : 1)
    score_select_kernel(KvView kv, SelectArgs a, unsigned* err) {
  extern __shared__ float s_scores[];  // [max_blocks]; rank 0's copy holds every score
  __shared__ uint32_t s_hist[3][kHistWords];
  __shared__ int s_warp[kWarps + 1];

  pdl_trigger();
  pdl_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int B = kv.block;
  const int L = max(kv.seq_lens[b], 0);
  int nb = ceil_div(L, B);
  if (nb > kv.max_blocks) {
    if (tid == 0 && rank == 0) set_error(err, HS_EBIT_BLOCK_RANGE);
    nb = kv.max_blocks;
  }
  const int64_t pair = static_cast<int64_t>(b) * kv.hkv + kvh;
  const int D = C * 32;

  // ---- scoring: this CTA's slice of blocks, one warp per block ----
  {
    float qp[G][C], qn[G][C];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int64_t qo = (static_cast<int64_t>(b) * kv.hq + kvh * G + h) * D + lane * C;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        float x = F32 ? static_cast<const float*>(a.q)[qo + c]
                      : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[qo + c]);
        qp[h][c] = fmaxf(x, 0.0f);
        qn[h][c] = fminf(x, 0.0f);
      }
    }
    float* dst = cluster.map_shared_rank(s_scores, 0);
    const int per = ceil_div(nb, kSelectCluster);
    const int jb = static_cast<int>(rank) * per, je = min(nb, jb + per);
    // Each warp scores kNB consecutive blocks per round: all their summaries are
    // loaded first (memory-level parallelism), then the kNB x G partial dot
    // products of every lane are summed across the warp by a transpose
    // reduction (each round halves the values a lane holds), so a block costs
    // about 8 shuffles instead of 5 per head.
    constexpr int kNB = (32 / G) < 4 ? ((32 / G) < 1 ? 1 : 32 / G) : 4;
    constexpr int kV = kNB * G;                    // partial sums per lane
    constexpr int kVPL = kV >= 32 ? kV / 32 : 1;   // values per lane after the reduction
    constexpr int kLPV = kV >= 32 ? 1 : 32 / kV;   // lanes holding one value
    constexpr int kLanesPerBlock = G * kLPV / kVPL;
    for (int base = jb + warp * kNB; base < je; base += kWarps * kNB) {
      float mx[kNB][C], mn[kNB][C];
#pragma unroll
      for (int u = 0; u < kNB; ++u) {
        const int j = min(base + u, je - 1);  // clamp: re-reads a valid block, result unused
        const int64_t off = (pair * kv.max_blocks + j) * D + lane * C;
        load_summary<C, F32>(a.smax, off, mx[u]);
        load_summary<C, F32>(a.smin, off, mn[u]);
      }
      float v[kV];
#pragma unroll
      for (int u = 0; u < kNB; ++u)
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float acc = 0.0f;
#pragma unroll
          for (int c = 0; c < C; ++c) {
            acc = fmaf(qp[h][c], mx[u][c], acc);
            acc = fmaf(qn[h][c], mn[u][c], acc);
          }
          v[u * G + h] = acc;
        }
      int cur = kV;
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        if (cur > 1) {
          const bool upper = (lane & o) != 0;
          const int half = cur / 2;
#pragma unroll
          for (int i = 0; i < kV / 2; ++i) {
            if (i < half) {
              const float send = upper ? v[i] : v[i + half];
              const float keep = upper ? v[i + half] : v[i];
              v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
          }
          cur = half;
        } else {
          v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
      }
      // lane now holds values [first, first + kVPL) of index u*G + h
      float best = v[0];
#pragma unroll
      for (int i = 1; i < kVPL; ++i) best = fmaxf(best, v[i]);
#pragma unroll
      for (int o = 1; o < kLanesPerBlock; o <<= 1) best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
      const int first = kV >= 32 ? lane * kVPL : lane / kLPV;
      const int u = first / G;
      if ((lane % kLanesPerBlock) == 0 && base + u < je) {
        dst[base + u] = best;
        if (a.scores) a.scores[pair * kv.max_blocks + base + u] = best;
      }
    }
  }
  for (int i = tid; i < kHistWords; i += kThreads) s_hist[0][i] = 0u;
  cluster.sync();
  if (rank != 0) return;

  smooth_scores(s_scores, nb, kv.max_blocks, a, pair);
  select_pair<kThreads>(s_scores, nb, L, B, a, pair, s_hist, s_warp, err);
}

// The selection of one (request, kv head) from its scores in global memory
// (written by the tensor-core scorer), by all THREADS threads of the CTA.
template <int THREADS, int KPT>
__device__ __forceinline__ void select_from_scores(const KvView& kv, const SelectArgs& a, const float* scores,
                                                   unsigned* err) {
  constexpr int kWarps = THREADS / 32;
  extern __shared__ float s_scores[];
  __shared__ uint32_t s_hist[3][kHistWords];
  __shared__ int s_warp[kWarps];
  __shared__ uint32_t s_range[2 * kWarps];
  const int tid = threadIdx.x;
  const int64_t pair = blockIdx.x;
  const int b = static_cast<int>(pair / kv.hkv);
  const int B = kv.block;
  const int L = max(kv.seq_lens[b], 0);
  int nb = ceil_div(L, B);
  if (nb > kv.max_blocks) {
    if (tid == 0) set_error(err, HS_EBIT_BLOCK_RANGE);
    nb = kv.max_blocks;
  }
  const float* src = scores + pair * kv.max_blocks;
  // the scores, and per warp the range of the keys of the scored (not forced) blocks
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int j0 = 0; j0 < nb; j0 += THREADS) {
    const int j = j0 + tid;
    if (j < nb) {
      const float v = src[j];
      s_scores[j] = v;
      if (!is_forced(j, L, B, a.sink_tokens, a.window_tokens)) {
        lo = min(lo, score_key(v));
        hi = max(hi, score_key(v));
      }
    }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if ((tid & 31) == 0) {
    s_range[2 * (tid >> 5)] = lo;
    s_range[2 * (tid >> 5) + 1] = hi;
  }
  for (int i = tid; i < kHistWords; i += THREADS) s_hist[0][i] = 0u;
  __syncthreads();
  const bool smoothed = a.history_weight != 0.0f && a.history != nullptr;  // the range no longer holds
  smooth_scores(s_scores, nb, kv.max_blocks, a, pair);
  select_pair_regs<THREADS, KPT>(s_scores, nb, L, B, a, pair, s_hist, s_warp, err, nullptr,
                                  smoothed ? nullptr : s_range, kWarps, true);
}

// One CTA per (request, kv head): scores -> selection.
template <int THREADS, int KPT>
__global__ __launch_bounds__(THREADS) void select_only_kernel(KvView kv, SelectArgs a, const float* scores,
                                                              unsigned* err) {
  pdl_trigger();
  pdl_wait();
  select_from_scores<THREADS, KPT>(kv, a, scores, err);
}

// The same, then the HiSparse hot-buffer plan of the stream ("KV 稀疏化" wiki
// §7) on the selection this CTA has just written: one launch instead of the
// selection and hs_swapin_plan's kernel, with the same outputs.
template <int THREADS, int KPT>
__global__ __launch_bounds__(THREADS) void select_plan_kernel(KvView kv, SelectArgs a, const float* scores,
                                                              PlanArgs pa, unsigned* err) {
  __shared__ plan::PlanSmem sm;
  pdl_trigger();
  pdl_wait();
  select_from_scores<THREADS, KPT>(kv, a, scores, err);
  __syncthreads();  // the stream's selection, written to global memory by this CTA, is complete
  const int pair = blockIdx.x;
  const int32_t* my_sel = a.sel + static_cast<int64_t>(pair) * a.capacity;
  const int cnt = plan::plan_stream(pa.hb, my_sel, a.sel_count[pair], a.capacity, pa.step, pair, sm, err);
  plan::write_lists(pa.hb, my_sel, cnt, a.capacity, pair, sm, pa.hit_sel, pa.hit_count, pa.miss_sel, pa.miss_count,
                    pa.stats);
}

template <int C, int G, bool F32>
cudaError_t launch_t(const KvView& kv, const SelectArgs& a, unsigned* err, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(kv.max_blocks) * sizeof(float);
  auto kern = score_select_kernel<C, G, F32>;
  if (cudaError_t e = allow_dynamic_smem(kern, smem); e != cudaSuccess) return e;
  dim3 grid(kSelectCluster, kv.hkv, kv.batch);
  return launch_pdl(kern, grid, dim3(kThreads), smem, st, kv, a, err);
}

template <int C, bool F32>
cudaError_t launch_g(const KvView& kv, const SelectArgs& a, unsigned* err, cudaStream_t st) {
  switch (kv.group) {
    case 1: return launch_t<C, 1, F32>(kv, a, err, st);
    case 2: return launch_t<C, 2, F32>(kv, a, err, st);
    case 4: return launch_t<C, 4, F32>(kv, a, err, st);
    case 8: return launch_t<C, 8, F32>(kv, a, err, st);
    default: return launch_t<C, 16, F32>(kv, a, err, st);
  }
}

}  // namespace

cudaError_t launch_select_only(const KvView& kv, const SelectArgs& a, const float* scores, unsigned* err,
                               cudaStream_t st) {
  const int pairs = kv.batch * kv.hkv;
  if (pairs == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(kv.max_blocks) * sizeof(float);
  // KPT consecutive blocks per thread (THREADS * KPT >= max_blocks): 256
  // threads up to 1024 blocks, 1024 threads above, with as few blocks per
  // thread as cover the request
  auto kern = kv.max_blocks <= 1024   ? select_only_kernel<kThreads, 1024 / kThreads>
              : kv.max_blocks <= 4096 ? select_only_kernel<1024, 4>
              : kv.max_blocks <= 8192 ? select_only_kernel<1024, 8>
                                      : select_only_kernel<1024, kMaxSelectBlocks / 1024>;
  const int threads = kv.max_blocks > 1024 ? 1024 : kThreads;
  if (cudaError_t e = allow_dynamic_smem(kern, smem); e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(pairs), dim3(threads), smem, st, kv, a, scores, err);
}

bool select_plan_supported(const KvView& kv, const HotView& hb) {
  return kv.max_blocks <= 1024 && hb.slots <= plan::kMaxSlots;
}

cudaError_t launch_select_plan(const KvView& kv, const SelectArgs& a, const float* scores, const PlanArgs& pa,
                               unsigned* err, cudaStream_t st) {
  const int pairs = kv.batch * kv.hkv;
  if (pairs == 0) return cudaSuccess;
  if (!select_plan_supported(kv, pa.hb)) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(kv.max_blocks) * sizeof(float);
  auto kern = select_plan_kernel<kThreads, 1024 / kThreads>;
  if (cudaError_t e = allow_dynamic_smem(kern, smem); e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(pairs), dim3(kThreads), smem, st, kv, a, scores, pa, err);
}

cudaError_t launch_score_select(const KvView& kv, const SelectArgs& a, unsigned* err,
                                cudaStream_t st) {
  if (kv.batch == 0 || kv.hkv == 0) return cudaSuccess;
  const bool f32 = kv.kv_dtype == HS_KV_F32;
  if (kv.head_dim == 128) return f32 ? launch_g<4, true>(kv, a, err, st) : launch_g<4, false>(kv, a, err, st);
  return f32 ? launch_g<2, true>(kv, a, err, st) : launch_g<2, false>(kv, a, err, st);
}

}  // namespace hs
