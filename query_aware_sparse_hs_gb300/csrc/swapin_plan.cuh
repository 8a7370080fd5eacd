// HiSparse hot-buffer table rule ("KV 稀疏化" wiki §7) for one stream, run by
// all threads of a CTA: hits stamped and protected, misses placed in
// ascending block order on the free slot, else the least recently used slot
// outside the selection; and the hit / miss lists in the selection layout.
// Shared by the plan kernel and the selection kernel that plans in the same
// launch.
#pragma once

#include "hs_internal.h"

namespace hs {
namespace plan {

constexpr int kMaxSlots = 1024;

__device__ __forceinline__ unsigned long long umin64(unsigned long long a, unsigned long long b) {
  return a < b ? a : b;
}

struct PlanSmem {
  int owner[kMaxSlots];
  int last[kMaxSlots];
  int sel[kMaxSlots];  // the stream's selection
  unsigned char prot[kMaxSlots];
  // per selection entry: 1 = resident at entry, 2 = a page-table entry out of
  // the stream's slots (skipped by the victim walk), 0 = to be brought in
  unsigned char hit[kMaxSlots];
  int copy_j[kMaxSlots];
  int copy_s[kMaxSlots];
  int ncopy, hits, evict;
};

// Runs the victim rule of one stream and updates its tables.  Returns the
// stream's selection count (entries of `my_sel`), or -1 when the selection
// does not fit (HS_EBIT_CAPACITY; the stream is left untouched).  Afterwards
// sm.copy_j/copy_s hold the sm.ncopy (block, slot) pairs to fill and sm.hit[i]
// says whether entry i was a hit.  All threads of the CTA call it.
static __device__ int plan_stream(const HotView& hb, const int32_t* my_sel, int cnt, int capacity, int step, int pair,
                           PlanSmem& sm, unsigned* err) {
  const int S = hb.slots;
  const int base = pair * S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (cnt > capacity || cnt > S) {
    if (tid == 0) set_error(err, HS_EBIT_CAPACITY);
    return -1;
  }
  if (cnt < 0) cnt = 0;
  int32_t* pt = hb.page_table + static_cast<int64_t>(pair) * hb.max_blocks;

  for (int s = tid; s < S; s += blockDim.x) {
    sm.owner[s] = hb.slot_owner[base + s];
    sm.last[s] = hb.last_used[base + s];
    sm.prot[s] = 0;
  }
  if (tid == 0) { sm.ncopy = 0; sm.hits = 0; sm.evict = 0; }
  __syncthreads();

  // hits: stamp and protect
  for (int i = tid; i < cnt; i += blockDim.x) {
    const int j = my_sel[i];
    sm.sel[i] = j;
    sm.hit[i] = 0;
    if (j < 0 || j >= hb.max_blocks) continue;
    const int g = pt[j];
    if (g >= 0) {
      const int s = g - base;
      if (s < 0 || s >= S) {
        set_error(err, HS_EBIT_PAGE_RANGE);
        sm.hit[i] = 2;
        continue;
      }
      sm.prot[s] = 1;
      sm.last[s] = step;
      sm.hit[i] = 1;
      atomicAdd(&sm.hits, 1);
    }
  }
  __syncthreads();

  // misses, in ascending block order (from shared memory only: a miss's
  // page-table entry is -1 until this walk assigns it a slot)
  if (warp == 0) {
    for (int i = 0; i < cnt; ++i) {
      const int j = sm.sel[i];
      if (j < 0 || j >= hb.max_blocks) {
        if (lane == 0) set_error(err, HS_EBIT_BLOCK_RANGE);
        continue;
      }
      if (sm.hit[i]) continue;  // resident (or an entry out of the stream's slots)
      // victim key: (class, last_used, slot); class 0 = free, 1 = evictable, 3 = protected
      unsigned long long best = ~0ull;
      for (int s = lane; s < S; s += 32) {
        unsigned long long key;
        if (sm.owner[s] < 0)
          key = static_cast<unsigned long long>(s);
        else if (sm.prot[s])
          key = (3ull << 62) | static_cast<unsigned long long>(s);
        else
          key = (1ull << 62) |
                (static_cast<unsigned long long>(static_cast<uint32_t>(sm.last[s]) ^ 0x80000000u) << 20) |
                static_cast<unsigned long long>(s);
        best = umin64(best, key);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) best = umin64(best, __shfl_xor_sync(0xffffffffu, best, o));
      const int s = static_cast<int>(best & 0xFFFFFull);
      if ((best >> 62) == 3ull) {  // cannot happen when cnt <= S
        if (lane == 0) set_error(err, HS_EBIT_CAPACITY);
        break;
      }
      if (lane == 0) {
        const int old = sm.owner[s];
        if (old >= 0) {
          pt[old] = -1;
          ++sm.evict;
        }
        sm.owner[s] = j;
        sm.last[s] = step;
        sm.prot[s] = 1;
        pt[j] = base + s;
        sm.copy_j[sm.ncopy] = j;
        sm.copy_s[sm.ncopy] = s;
        ++sm.ncopy;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int s = tid; s < S; s += blockDim.x) {
    hb.slot_owner[base + s] = sm.owner[s];
    hb.last_used[base + s] = sm.last[s];
  }
  return cnt;
}

// Hit and miss lists of the stream in the selection layout (ascending, -1
// padded) with their counts, and the stream's statistics; after plan_stream
// (cnt = its result).  All threads of the CTA call it.
static __device__ void write_lists(const HotView& hb, const int32_t* my_sel, int cnt, int capacity, int pair,
                                   PlanSmem& sm, int32_t* hit_sel, int32_t* hit_count, int32_t* miss_sel,
                                   int32_t* miss_count, hs_swap_stats* stats) {
  const int64_t row = static_cast<int64_t>(pair) * capacity;
  int nh = 0, nm = 0;
  if (cnt > 0 && threadIdx.x < 32) {  // warp 0 compacts hits and misses in selection order
    const int lane = threadIdx.x;
    for (int i0 = 0; i0 < cnt; i0 += 32) {
      const int i = i0 + lane;
      const int j = i < cnt ? my_sel[i] : -1;
      const bool valid = i < cnt && j >= 0 && j < hb.max_blocks;
      const bool h = valid && sm.hit[i] == 1;
      const bool m = valid && sm.hit[i] != 1;
      const unsigned bh = __ballot_sync(0xffffffffu, h), bm = __ballot_sync(0xffffffffu, m);
      const unsigned below = (1u << lane) - 1u;
      if (h) hit_sel[row + nh + __popc(bh & below)] = j;
      if (m) miss_sel[row + nm + __popc(bm & below)] = j;
      nh += __popc(bh);
      nm += __popc(bm);
    }
  }
  __shared__ int s_nh, s_nm;
  if (threadIdx.x == 0) { s_nh = nh; s_nm = nm; }  // warp 0's lanes all hold the totals
  __syncthreads();
  for (int i = s_nh + threadIdx.x; i < capacity; i += blockDim.x) hit_sel[row + i] = -1;
  for (int i = s_nm + threadIdx.x; i < capacity; i += blockDim.x) miss_sel[row + i] = -1;
  if (threadIdx.x == 0) {
    hit_count[pair] = s_nh;
    miss_count[pair] = s_nm;
    if (stats && cnt >= 0) {
      atomicAdd(&stats->hits, static_cast<unsigned long long>(s_nh));
      atomicAdd(&stats->misses, static_cast<unsigned long long>(sm.ncopy));
      atomicAdd(&stats->evictions, static_cast<unsigned long long>(sm.evict));
    }
  }
}

}  // namespace plan
}  // namespace hs
