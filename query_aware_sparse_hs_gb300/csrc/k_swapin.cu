// HiSparse swap-in ("KV 稀疏化" wiki §7): on the decode path, detect the
// selected blocks that are not in the hot device buffer, pick victims by the
// current access set, update the page table, and pull the missing pages back
// from the pinned host pool.
//
// One CTA per (request, kv head) stream.  The table logic is sequential by
// definition (each miss sees the state left by the previous one), so warp 0
// runs it in ascending block order with a warp-wide argmin over the slots;
// then the whole CTA streams the missing pages from mapped host memory into
// their slots with 16-byte vector loads (zero-copy over the CPU-GPU link).
#include "hs_internal.h"

namespace hs {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxSlots = 1024;

__device__ __forceinline__ unsigned long long umin64(unsigned long long a, unsigned long long b) {
  return a < b ? a : b;
}

__global__ __launch_bounds__(kThreads) void swapin_kernel(HotView hb, const int32_t* __restrict__ sel,
                                                          const int32_t* __restrict__ sel_count,
                                                          int capacity, int step,
                                                          hs_swap_stats* stats, unsigned* err) {
  __shared__ int s_owner[kMaxSlots];
  __shared__ int s_last[kMaxSlots];
  __shared__ unsigned char s_prot[kMaxSlots];
  __shared__ int s_copy_j[kMaxSlots];
  __shared__ int s_copy_s[kMaxSlots];
  __shared__ int s_ncopy, s_hits, s_evict;

  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x;
  const int S = hb.slots;
  const int base = pair * S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int cnt = sel_count[pair];
  if (cnt > capacity || cnt > S) {
    if (tid == 0) set_error(err, HS_EBIT_CAPACITY);
    return;  // the stream is left untouched
  }
  if (cnt < 0) cnt = 0;
  const int32_t* my_sel = sel + static_cast<int64_t>(pair) * capacity;
  int32_t* pt = hb.page_table + static_cast<int64_t>(pair) * hb.max_blocks;

  for (int s = tid; s < S; s += kThreads) {
    s_owner[s] = hb.slot_owner[base + s];
    s_last[s] = hb.last_used[base + s];
    s_prot[s] = 0;
  }
  if (tid == 0) { s_ncopy = 0; s_hits = 0; s_evict = 0; }
  __syncthreads();

  // hits: stamp and protect
  for (int i = tid; i < cnt; i += kThreads) {
    const int j = my_sel[i];
    if (j < 0 || j >= hb.max_blocks) continue;
    const int g = pt[j];
    if (g >= 0) {
      const int s = g - base;
      if (s < 0 || s >= S) { set_error(err, HS_EBIT_PAGE_RANGE); continue; }
      s_prot[s] = 1;
      s_last[s] = step;
      atomicAdd(&s_hits, 1);
    }
  }
  __syncthreads();

  // misses, in ascending block order
  if (warp == 0) {
    for (int i = 0; i < cnt; ++i) {
      const int j = my_sel[i];
      if (j < 0 || j >= hb.max_blocks) {
        if (lane == 0) set_error(err, HS_EBIT_BLOCK_RANGE);
        continue;
      }
      if (pt[j] >= 0) continue;  // a hit (or a block placed earlier in this loop)
      // victim key: (class, last_used, slot); class 0 = free, 1 = evictable, 3 = protected
      unsigned long long best = ~0ull;
      for (int s = lane; s < S; s += 32) {
        unsigned long long key;
        if (s_owner[s] < 0)
          key = static_cast<unsigned long long>(s);
        else if (s_prot[s])
          key = (3ull << 62) | static_cast<unsigned long long>(s);
        else
          key = (1ull << 62) |
                (static_cast<unsigned long long>(static_cast<uint32_t>(s_last[s]) ^ 0x80000000u) << 20) |
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
        const int old = s_owner[s];
        if (old >= 0) {
          pt[old] = -1;
          ++s_evict;
        }
        s_owner[s] = j;
        s_last[s] = step;
        s_prot[s] = 1;
        pt[j] = base + s;
        s_copy_j[s_ncopy] = j;
        s_copy_s[s_ncopy] = s;
        ++s_ncopy;
      }
      __syncwarp();
    }
  }
  __syncthreads();
  for (int s = tid; s < S; s += kThreads) {
    hb.slot_owner[base + s] = s_owner[s];
    hb.last_used[base + s] = s_last[s];
  }

  // copy the missing pages host -> slots
  const int ncopy = s_ncopy;
  const int elem = hb.kv_dtype == HS_KV_F32 ? 4 : (hb.kv_dtype == HS_KV_BF16 ? 2 : 1);
  const int64_t page_bytes = static_cast<int64_t>(hb.block) * hb.head_dim * elem;
  const int vec_per_page = static_cast<int>(page_bytes / 16);
  const int64_t total_vec = static_cast<int64_t>(ncopy) * vec_per_page;
  const int64_t pool_pair = static_cast<int64_t>(pair) * hb.max_blocks;
  for (int64_t v = tid; v < 2 * total_vec; v += kThreads) {
    const int which = v >= total_vec;  // 0 = K, 1 = V
    const int64_t w = v - which * total_vec;
    const int c = static_cast<int>(w / vec_per_page);
    const int64_t off = w % vec_per_page;
    const int64_t src_page = pool_pair + s_copy_j[c];
    const int64_t dst_page = base + s_copy_s[c];
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(which ? hb.host_v : hb.host_k) + src_page * page_bytes) + off;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<char*>(which ? hb.v_slots : hb.k_slots) + dst_page * page_bytes) + off;
    *dst = *src;
  }
  if (hb.kv_dtype == HS_KV_FP8E4M3_G32) {
    const int sc_per_page = hb.block * (hb.head_dim / kQuantGroup);
    const int64_t total_sc = static_cast<int64_t>(ncopy) * sc_per_page;
    for (int64_t v = tid; v < 2 * total_sc; v += kThreads) {
      const int which = v >= total_sc;
      const int64_t w = v - which * total_sc;
      const int c = static_cast<int>(w / sc_per_page);
      const int64_t off = w % sc_per_page;
      const int64_t src_page = pool_pair + s_copy_j[c];
      const int64_t dst_page = base + s_copy_s[c];
      const float* src = (which ? hb.host_v_scales : hb.host_k_scales) + src_page * sc_per_page + off;
      float* dst = (which ? hb.v_slot_scales : hb.k_slot_scales) + dst_page * sc_per_page + off;
      *dst = *src;
    }
  }
  if (stats && tid == 0) {
    const int64_t sc_bytes = hb.kv_dtype == HS_KV_FP8E4M3_G32
                                 ? static_cast<int64_t>(hb.block) * (hb.head_dim / kQuantGroup) * 4
                                 : 0;
    atomicAdd(&stats->hits, static_cast<unsigned long long>(s_hits));
    atomicAdd(&stats->misses, static_cast<unsigned long long>(ncopy));
    atomicAdd(&stats->evictions, static_cast<unsigned long long>(s_evict));
    atomicAdd(&stats->bytes_in, static_cast<unsigned long long>(ncopy) * 2ull *
                                    static_cast<unsigned long long>(page_bytes + sc_bytes));
  }
}

}  // namespace

cudaError_t launch_swapin(const HotView& hb, const int32_t* sel, const int32_t* sel_count,
                          int capacity, int step, hs_swap_stats* stats, unsigned* err,
                          cudaStream_t st) {
  const int pairs = hb.batch * hb.hkv;
  if (pairs == 0) return cudaSuccess;
  return launch_pdl(swapin_kernel, dim3(pairs), dim3(kThreads), 0, st, hb, sel, sel_count, capacity, step,
                    stats, err);
}

}  // namespace hs
