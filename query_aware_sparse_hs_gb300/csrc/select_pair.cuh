// Selection of the blocks of one (request, kv head) from its block scores in
// shared memory ("KV 稀疏化" wiki §2 sink/window, §5 top-k; SparDA §4.2 and
// §6.1), shared by the selection kernels and the fused scoring kernel.  Every
// function here is run by all THREADS threads of the CTA.
#pragma once

#include "hs_internal.h"

namespace hs {
namespace sel {

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

// Histogram of one radix pass: 256 digit counters, one padding word after
// every 8 so that the digit scan below reads without bank conflicts.
constexpr int kHistWords = 256 + 32;
__device__ __forceinline__ int hist_index(uint32_t digit) { return static_cast<int>(digit + (digit >> 3)); }

// Digit scan of one radix pass, run by every warp on its own: the digit holding
// the kk-th largest counted key (digits taken from 255 down), that key's rank
// within the digit and the digit's count.  Lane l owns digits 255-8l .. 248-8l.
__device__ __forceinline__ void find_digit(const uint32_t* hist, int kk, int& digit, int& rank, int& count) {
  const int lane = threadIdx.x & 31;
  uint32_t hv[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    hv[i] = hist[hist_index(255u - 8u * lane - i)];
    sum += static_cast<int>(hv[i]);
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  int above = incl - sum, d = -1, r = 0, n = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int h = static_cast<int>(hv[i]);
    if (above < kk && kk <= above + h) {
      d = 255 - 8 * lane - i;
      r = kk - above;
      n = h;
    }
    above += h;
  }
  const int src = __ffs(__ballot_sync(0xffffffffu, d >= 0)) - 1;  // exactly one lane
  digit = __shfl_sync(0xffffffffu, d, src & 31);
  rank = __shfl_sync(0xffffffffu, r, src & 31);
  count = __shfl_sync(0xffffffffu, n, src & 31);
}

// The same smoothing with the previous step's history already staged in shared
// memory (s_prev, nb floats), for CTAs that select the same pair side by side:
// the new history is stored only when `store`.  All threads of the CTA call it.
__device__ __forceinline__ void smooth_staged(float* s_scores, const float* s_prev, int nb, int max_blocks,
                                              const SelectArgs& a, int64_t pair, bool store) {
  float* h = a.history + pair * max_blocks;
  const float w = a.history_weight, keep = 1.0f - a.history_weight;
  for (int j = threadIdx.x; j < nb; j += blockDim.x) {
    const float old = s_prev[j];
    const float v = old == old ? fmaf(w, old, keep * s_scores[j]) : s_scores[j];
    s_scores[j] = v;
    if (store) h[j] = v;
  }
  __syncthreads();
}

// Selection of one (request, kv head) from its block scores in shared memory,
// by all THREADS threads of the CTA ("KV 稀疏化" wiki §2 sink/window, §5 top-k):
// forced blocks in closed form; the k-th largest key among the other blocks by
// an 8-bit radix select (one pass per byte below the bytes that every key
// shares; three histogram buffers let the clearing of the next one ride on the
// current pass; with up to 12 warps every warp scans the histogram itself, so
// a pass takes one CTA barrier); then forced-or-above-threshold blocks and the lowest-index
// threshold-equal blocks are placed in ascending order with warp ballots and
// one barrier.
//   s_hist     three buffers of kHistWords; the first must be zero on entry,
//              all are left dirty.
//   s_warp     THREADS / 32 ints.
//   s_out      (nullable, shared memory, capacity ints) receives the selected
//              indices as well.
//   key_range  (nullable) n_range pairs (min, max) of score_key over sets of
//              blocks that together cover blocks [0, nb); with it the passes
//              start at the first byte where the smallest and the largest key
//              differ.
//   store      false: nothing is written to global memory (sel, sel_count,
//              error bits); another CTA stores the same selection.
// Returns the number stored (min(selected, capacity)) to every thread.
template <int THREADS>
__device__ __forceinline__ int select_pair(const float* s_scores, int nb, int L, int B, const SelectArgs& a,
                                           int64_t pair, uint32_t (*s_hist)[kHistWords], int* s_warp,
                                           unsigned* err, int* s_out = nullptr, const uint32_t* key_range = nullptr,
                                           int n_range = 0, bool store = true) {
  constexpr int kWarps = THREADS / 32;
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
  int32_t* out = a.sel + pair * cap;

  if (nf + k >= nb) {  // every block is selected
    for (int j = tid; j < cap; j += THREADS) {
      if (store) out[j] = j < nb ? j : -1;
      if (s_out && j < nb) s_out[j] = j;
    }
    if (tid == 0 && store) {
      if (nb > cap) set_error(err, HS_EBIT_CAPACITY);
      a.sel_count[pair] = min(nb, cap);
    }
    return min(nb, cap);
  }

  uint32_t T = 0;
  int need_eq = 0;
  if (k > 0) {
    uint32_t lo = 0u, hi = 0xffffffffu;
    if (key_range) {
      lo = 0xffffffffu;
      hi = 0u;
      for (int i = 0; i < n_range; ++i) {
        lo = min(lo, key_range[2 * i]);
        hi = max(hi, key_range[2 * i + 1]);
      }
    }
    const uint32_t diff = lo ^ hi;
    int shift = diff == 0u ? -8 : ((31 - __clz(diff)) & ~7);  // highest byte that differs
    uint32_t mask = shift >= 24 ? 0u : (0xffffffffu << (shift + 8));
    uint32_t prefix = hi & mask;
    int kk = k;  // rank (1-based) of the wanted key among the keys matching prefix
    for (int pass = 0; shift >= 0; shift -= 8, ++pass) {
      uint32_t* hist = s_hist[pass % 3];
      uint32_t* next = s_hist[(pass + 1) % 3];  // last read two passes ago
      for (int i = tid; i < kHistWords; i += THREADS) next[i] = 0u;
      for (int j = tid; j < nb; j += THREADS) {
        if (forced(j)) continue;
        const uint32_t key = score_key(s_scores[j]);
        if ((key & mask) == prefix) atomicAdd(&hist[hist_index((key >> shift) & 255u)], 1u);
      }
      __syncthreads();
      int digit, rank, count;
      if constexpr (kWarps <= 12) {
        find_digit(hist, kk, digit, rank, count);  // every warp on its own: no second barrier
      } else {
        // many warps: warp 0 scans and the others read its result
        if (warp == 0) {
          find_digit(hist, kk, digit, rank, count);
          if (lane == 0) {
            s_warp[0] = digit;
            s_warp[1] = rank;
          }
        }
        __syncthreads();
        digit = s_warp[0];
        rank = s_warp[1];
        __syncthreads();  // s_warp is rewritten by the next pass or the placement
      }
      prefix |= static_cast<uint32_t>(digit) << shift;
      mask |= 255u << shift;
      kk = rank;
    }
    T = prefix;
    need_eq = kk;
  }

  // Placement: warp w takes the contiguous index range [w*R, (w+1)*R) in rounds
  // of 32; per round, ballots of "forced or above T" and "equal to T" give each
  // lane its position.  An equal block is chosen while fewer than need_eq
  // equal blocks precede it (lower index first).
  const int rounds = ceil_div(nb, 32 * kWarps);
  const int base = warp * rounds * 32;
  const unsigned below = (1u << lane) - 1u;
  auto flags = [&](int j, bool& gt, bool& eq) {
    gt = false;
    eq = false;
    if (j >= nb) return;
    if (forced(j)) {
      gt = true;
    } else if (k > 0) {
      const uint32_t key = score_key(s_scores[j]);
      gt = key > T;
      eq = key == T;
    }
  };
  int gt_w = 0, eq_w = 0;
  for (int r = 0; r < rounds; ++r) {
    bool gt, eq;
    flags(base + r * 32 + lane, gt, eq);
    gt_w += __popc(__ballot_sync(0xffffffffu, gt));
    eq_w += __popc(__ballot_sync(0xffffffffu, eq));
  }
  if (lane == 0) s_warp[warp] = (gt_w << 16) | eq_w;
  __syncthreads();
  int gt_b = 0, eq_b = 0, gt_t = 0, eq_t = 0;
#pragma unroll 4
  for (int w = 0; w < kWarps; ++w) {
    const int v = s_warp[w];
    if (w < warp) {
      gt_b += v >> 16;
      eq_b += v & 0xffff;
    }
    gt_t += v >> 16;
    eq_t += v & 0xffff;
  }
  for (int r = 0; r < rounds; ++r) {
    const int j = base + r * 32 + lane;
    bool gt, eq;
    flags(j, gt, eq);
    const unsigned bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    const int eq_before = eq_b + __popc(be & below);
    if (gt || (eq && eq_before < need_eq)) {
      const int pos = gt_b + __popc(bg & below) + min(eq_before, need_eq);  // chosen blocks before j
      if (pos < cap) {
        if (store) out[pos] = j;
        if (s_out) s_out[pos] = j;
      }
    }
    gt_b += __popc(bg);
    eq_b += __popc(be);
  }
  const int total = gt_t + min(eq_t, need_eq);
  if (store) {
    for (int i = total + tid; i < cap; i += THREADS) out[i] = -1;
    if (tid == 0) {
      if (total > cap) set_error(err, HS_EBIT_CAPACITY);
      a.sel_count[pair] = min(total, cap);
    }
  }
  return min(total, cap);
}

// Whether block j of a request of L tokens is forced (sink or window).
__device__ __forceinline__ bool is_forced(int j, int L, int B, int sink, int win) {
  const int lo = j * B, hi = min(lo + B, L);
  return lo < sink || (win > 0 && hi > L - win);
}

// The same selection with the keys held in registers: thread t owns blocks
// t*KPT .. t*KPT+KPT-1 (nb <= THREADS * KPT), keys are computed once, forced
// blocks are [0, sink blocks) and [first window block, nb), and placement is
// one warp scan of per-thread counts plus one barrier.  Same arguments, result
// and tie rule as select_pair.
//
// The k-th largest candidate key is found by counting passes over the
// candidates' own key range [lo, hi] rather than fixed bytes: a pass counts
// the keys of the current range in 256 bins of width 2^sh (the smallest
// power of two that covers the range in 256 bins) and keeps the bin that holds
// the wanted key.  The search ends as soon as that bin's keys are all taken
// (its count equals the rank still wanted: every key from the bin's lower
// bound up is selected) or the bins are single keys (then ties take the lowest
// indices).  Bound scores of one request sit in a narrow band, so the bins
// spread them out (few shared-memory atomics meet on one counter) and one or
// two passes usually settle the threshold.  With up to 12 warps every warp
// scans the histogram itself; with more, warp 0 scans and broadcasts.
//   key_range  (nullable) n_range pairs (min, max) of score_key covering every
//              candidate (scored, not forced) block; without it the range is
//              found here (one more barrier).
template <int THREADS, int KPT>
__device__ __forceinline__ int select_pair_regs(const float* s_scores, int nb, int L, int B, const SelectArgs& a,
                                                int64_t pair, uint32_t (*s_hist)[kHistWords], int* s_warp,
                                                unsigned* err, int* s_out, const uint32_t* key_range, int n_range,
                                                bool store) {
  constexpr int kWarps = THREADS / 32;
  static_assert(KPT <= 32, "per-thread block masks are 32 bits");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sink = a.sink_tokens, win = a.window_tokens, k = a.k_scored, cap = a.capacity;
  const int n_sink = min(nb, ceil_div(sink, B));
  int w_first = nb;
  if (win > 0) w_first = (L - win <= 0) ? 0 : min(nb, (L - win) / B);
  w_first = max(w_first, n_sink);
  const int nf = n_sink + (nb - w_first);
  int32_t* out = a.sel + pair * cap;

  if (nf + k >= nb) {  // every block is selected
    for (int j = tid; j < cap; j += THREADS) {
      if (store) out[j] = j < nb ? j : -1;
      if (s_out && j < nb) s_out[j] = j;
    }
    if (tid == 0 && store) {
      if (nb > cap) set_error(err, HS_EBIT_CAPACITY);
      a.sel_count[pair] = min(nb, cap);
    }
    return min(nb, cap);
  }

  const int j0 = tid * KPT;
  uint32_t key[KPT];
  unsigned cand = 0u, forc = 0u;  // per owned block: a candidate (scored) / forced
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const int j = j0 + i;
    key[i] = 0u;
    if (j < nb) {
      if (j < n_sink || j >= w_first) {
        forc |= 1u << i;
      } else {
        cand |= 1u << i;
        key[i] = score_key(s_scores[j]);
      }
    }
  }

  uint32_t T = 0;   // selected: key > T, then the first need_eq keys == T
  int need_eq = 0;
  if (k > 0) {
    uint32_t lo = 0xffffffffu, hi = 0u;
    if (key_range) {
      for (int i = 0; i < n_range; ++i) {
        lo = min(lo, key_range[2 * i]);
        hi = max(hi, key_range[2 * i + 1]);
      }
    } else {
      // the candidates' range through the third histogram buffer, which the
      // first pass does not touch (the second clears it after the first's barrier)
      uint32_t l = 0xffffffffu, h = 0u;
#pragma unroll
      for (int i = 0; i < KPT; ++i)
        if ((cand >> i) & 1u) {
          l = min(l, key[i]);
          h = max(h, key[i]);
        }
      l = __reduce_min_sync(0xffffffffu, l);
      h = __reduce_max_sync(0xffffffffu, h);
      uint32_t* scratch = s_hist[2];
      if (lane == 0) {
        scratch[2 * warp] = l;
        scratch[2 * warp + 1] = h;
      }
      __syncthreads();
#pragma unroll 4
      for (int i = 0; i < kWarps; ++i) {
        lo = min(lo, scratch[2 * i]);
        hi = max(hi, scratch[2 * i + 1]);
      }
    }
    uint32_t base = lo, span = hi - lo;  // the current range: [base, base + span]
    int kk = k;  // rank (1-based, from the top) of the wanted key within the range
    for (int pass = 0;; ++pass) {
      const int sh = max(0, 24 - __clz(span));  // bins of 2^sh keys: span >> sh < 256
      uint32_t* hist = s_hist[pass % 3];
      uint32_t* next = s_hist[(pass + 1) % 3];  // last read two passes ago
      for (int i = tid; i < kHistWords; i += THREADS) next[i] = 0u;
#pragma unroll
      for (int i = 0; i < KPT; ++i)
        if (((cand >> i) & 1u) && key[i] - base <= span) atomicAdd(&hist[hist_index((key[i] - base) >> sh)], 1u);
      __syncthreads();
      int digit, rank, count;
      if constexpr (kWarps <= 12) {
        find_digit(hist, kk, digit, rank, count);
      } else {
        if (warp == 0) {
          find_digit(hist, kk, digit, rank, count);
          if (lane == 0) {
            s_warp[0] = digit;
            s_warp[1] = rank;
            s_warp[2] = count;
          }
        }
        __syncthreads();
        digit = s_warp[0];
        rank = s_warp[1];
        count = s_warp[2];
        __syncthreads();  // s_warp is rewritten by the next pass or the placement
      }
      const uint32_t bin_lo = base + (static_cast<uint32_t>(digit) << sh);
      if (sh == 0) {  // single keys: ties take the lowest indices
        T = bin_lo;
        need_eq = rank;
        break;
      }
      if (count == rank && bin_lo > 0u) {  // the whole bin is taken: every key >= bin_lo
        T = bin_lo - 1u;
        need_eq = 0;
        break;
      }
      base = bin_lo;
      span = (1u << sh) - 1u;
      kk = rank;
    }
  }

  // placement: forced-or-above-threshold, then the lowest-index equal blocks
  unsigned gt = forc, eq = 0u;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    if (k > 0 && ((cand >> i) & 1u)) {
      gt |= (key[i] > T ? 1u : 0u) << i;
      eq |= (key[i] == T ? 1u : 0u) << i;
    }
  }
  const int mine = (__popc(gt) << 16) | __popc(eq);
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int before = incl - mine, total_packed = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int v = s_warp[w];
    before += w < warp ? v : 0;
    total_packed += v;
  }
  int gt_b = before >> 16, eq_b = before & 0xffff;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const bool is_gt = (gt >> i) & 1u, is_eq = (eq >> i) & 1u;
    if (is_gt || (is_eq && eq_b < need_eq)) {
      const int pos = gt_b + min(eq_b, need_eq);
      if (pos < cap) {
        if (store) out[pos] = j0 + i;
        if (s_out) s_out[pos] = j0 + i;
      }
    }
    gt_b += is_gt ? 1 : 0;
    eq_b += is_eq ? 1 : 0;
  }
  const int total = (total_packed >> 16) + min(total_packed & 0xffff, need_eq);
  if (store) {
    for (int i = total + tid; i < cap; i += THREADS) out[i] = -1;
    if (tid == 0) {
      if (total > cap) set_error(err, HS_EBIT_CAPACITY);
      a.sel_count[pair] = min(total, cap);
    }
  }
  return min(total, cap);
}

// Per-warp (min, max) of score_key over the blocks of the calling warp's
// lanes (valid = the lane holds a block): lane 0 stores the pair at
// range[2 * slot].  All 32 lanes call it.
__device__ __forceinline__ void warp_key_range(float score, bool valid, uint32_t* range, int slot) {
  const uint32_t key = score_key(score);
  const uint32_t lo = __reduce_min_sync(0xffffffffu, valid ? key : 0xffffffffu);
  const uint32_t hi = __reduce_max_sync(0xffffffffu, valid ? key : 0u);
  if ((threadIdx.x & 31) == 0) {
    range[2 * slot] = lo;
    range[2 * slot + 1] = hi;
  }
}

}  // namespace sel
}  // namespace hs
