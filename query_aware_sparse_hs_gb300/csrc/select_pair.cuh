// Selection of the blocks of one (request, kv head) from its block scores in
// shared memory ("KV 稀疏化" wiki §2 sink/window, §5 top-k; SparDA §4.2 and
// §6.1), shared by the selection kernels and the fused scoring kernel.  Every
// function here is run by all THREADS threads of the CTA.
#pragma once

#include "hs_internal.h"

namespace hs {
namespace sel {

// Exclusive prefix sum over a CTA of THREADS threads (at most 1024); `total`
// receives the CTA-wide sum.  s_warp holds THREADS / 32 + 1 ints.
template <int THREADS>
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int& total) {
  constexpr int kWarps = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? s_warp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < kWarps) s_warp[lane] = wi - w;
    if (lane == kWarps - 1) s_warp[kWarps] = wi;
  }
  __syncthreads();
  const int excl = s_warp[warp] + incl - v;
  total = s_warp[kWarps];
  __syncthreads();
  return excl;
}

// Score smoothing across decode steps ("SparDA" article §6.1): where the
// previous step's smoothed score h of a block is a number, the score becomes
// (1 - w) * s + w * h; a block without history keeps s.  The result is stored
// as the next step's history.  All threads of the CTA call it.
__device__ __forceinline__ void smooth_scores(float* s_scores, int nb, int max_blocks, const SelectArgs& a,
                                              int64_t pair) {
  if (a.history_weight == 0.0f || a.history == nullptr) return;
  float* h = a.history + pair * max_blocks;
  const float w = a.history_weight, keep = 1.0f - a.history_weight;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) {
    const float old = h[j];
    const float v = old == old ? fmaf(w, old, keep * s_scores[j]) : s_scores[j];
    s_scores[j] = v;
    h[j] = v;
  }
  __syncthreads();
}

// Selection of one (request, kv head) from its block scores in shared memory,
// by all THREADS threads of the CTA ("KV 稀疏化" wiki §2 sink/window, §5 top-k):
// forced blocks in closed form, a 4-pass 8-bit radix select of the k-th largest
// key among the other blocks (two histogram buffers, which must be zero on
// entry), then one packed scan that places forced-or-above-threshold blocks and
// the lowest-index threshold-equal blocks in ascending order.
template <int THREADS>
__device__ __forceinline__ void select_pair(const float* s_scores, int nb, int L, int B, const SelectArgs& a,
                                            int64_t pair, uint32_t (*s_hist)[256], int* s_warp, int* s_pick,
                                            unsigned* err) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sink = a.sink_tokens, win = a.window_tokens, k = a.k_scored, cap = a.capacity;
  auto forced = [&](int j) -> bool {
    const int lo = j * B, hi = min(lo + B, L);
    return lo < sink || (win > 0 && hi > L - win);
  };
  // forced blocks in closed form: [0, sink blocks) and [first window block, nb)
  const int n_sink = min(nb, ceil_div(sink, B));
  int w_first = nb;
  if (win > 0) w_first = (L - win <= 0) ? 0 : min(nb, (L - win) / B);
  const int nf = n_sink + max(0, nb - max(w_first, n_sink));
  const bool take_all = nf + k >= nb;
  const bool use_threshold = !take_all && k > 0;
  int32_t* out = a.sel + pair * cap;

  uint32_t T = 0;
  int need_eq = 0;
  if (use_threshold) {
    // 4-pass 8-bit radix select of the k-th largest key among non-forced blocks;
    // two histogram buffers so that clearing the next one rides on this pass
    uint32_t prefix = 0, mask = 0;
    int kk = k;  // rank (1-based) of the wanted key among keys matching `prefix`
    int buf = 0;
    for (int shift = 24; shift >= 0; shift -= 8, buf ^= 1) {
      uint32_t* hist = s_hist[buf];
      for (int j = tid; j < nb; j += THREADS) {
        if (forced(j)) continue;
        const uint32_t key = score_key(s_scores[j]);
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns digits 255-8l .. 248-8l; a warp scan from the top digit
        // finds the bucket holding the kk-th largest key
        uint32_t hv[8];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          hv[i] = hist[255 - 8 * lane - i];
          sum += static_cast<int>(hv[i]);
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += n;
        }
        int above = incl - sum;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int h = static_cast<int>(hv[i]);
          if (above < kk && kk <= above + h) {
            s_pick[0] = 255 - 8 * lane - i;
            s_pick[1] = kk - above;
          }
          above += h;
        }
        uint32_t* other = s_hist[buf ^ 1];
#pragma unroll
        for (int i = 0; i < 8; ++i) other[8 * lane + i] = 0u;
      }
      __syncthreads();
      prefix |= static_cast<uint32_t>(s_pick[0]) << shift;
      mask |= 255u << shift;
      kk = s_pick[1];
    }
    T = prefix;
    need_eq = kk;
  }

  if (take_all) {
    for (int j = tid; j < cap; j += THREADS) out[j] = j < nb ? j : -1;
    if (tid == 0) {
      if (nb > cap) set_error(err, HS_EBIT_CAPACITY);
      a.sel_count[pair] = min(nb, cap);
    }
    return;
  }
  // contiguous index range per thread keeps the output ascending.  One packed
  // scan gives, for every block, how many forced-or-above-threshold blocks and
  // how many threshold-equal blocks precede it; an equal block is chosen while
  // fewer than need_eq equal blocks precede it (lower index first).
  const int per_t = ceil_div(nb, THREADS);
  const int j0 = min(nb, tid * per_t), j1 = min(nb, j0 + per_t);
  int gt_local = 0, eq_local = 0;
  for (int j = j0; j < j1; ++j) {
    if (forced(j)) {
      ++gt_local;
    } else if (use_threshold) {
      const uint32_t key = score_key(s_scores[j]);
      gt_local += key > T;
      eq_local += key == T;
    }
  }
  int packed_total;
  const int packed = block_exclusive_scan<THREADS>((gt_local << 16) | eq_local, s_warp, packed_total);
  int gt_b = packed >> 16, eq_b = packed & 0xffff;
  const int total = (packed_total >> 16) + min(packed_total & 0xffff, need_eq);
  for (int j = j0; j < j1; ++j) {
    bool is_gt = forced(j), is_eq = false;
    if (!is_gt && use_threshold) {
      const uint32_t key = score_key(s_scores[j]);
      is_gt = key > T;
      is_eq = key == T;
    }
    if (is_gt || (is_eq && eq_b < need_eq)) {
      const int pos = gt_b + min(eq_b, need_eq);  // chosen blocks before j
      if (pos < cap) out[pos] = j;
    }
    gt_b += is_gt ? 1 : 0;
    eq_b += is_eq ? 1 : 0;
  }
  for (int i = total + tid; i < cap; i += THREADS) out[i] = -1;
  if (tid == 0) {
    if (total > cap) set_error(err, HS_EBIT_CAPACITY);
    a.sel_count[pair] = min(total, cap);
  }
}

}  // namespace sel
}  // namespace hs
