// HiSparse swap-in ("KV 稀疏化" wiki §7): on the decode path, detect the
// selected blocks that are not in the hot device buffer, pick victims by the
// current access set, update the page table, and pull the missing pages back
// from the pinned host pool.
//
// The table logic ("plan") is sequential by definition (each miss sees the
// state left by the previous one): one CTA per (request, kv head) stream, warp
// 0 walks the misses in ascending block order with a warp-wide argmin over the
// slots.  The page copy streams the missing pages from mapped host memory into
// their slots with 16-byte vector loads (zero-copy over the CPU-GPU link).
//
// Kernels: swapin_kernel plans and copies one stream per CTA;
// swapin_plan_kernel only plans, and lists the selection's hits (resident
// before the call) and misses in the selection layout; swapin_copy_kernel
// copies the pages of such a miss list on a few SMs, and
// copied_blocks_attn_kernel computes the attention over the copied blocks,
// so that both can run beside an attention launch over the hit list on the
// other SMs (they touch disjoint slots: victims are never in the current
// selection).
#include "hs_internal.h"

namespace hs {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxSlots = 1024;
// The copy kernel runs on a few SMs of its own (the attention CTAs beside it
// fill the SMs' shared memory): large CTAs keep many host loads in flight.
constexpr int kCopyThreads = 1024;
constexpr int kCopyUnroll = 4;
constexpr int kCopyBatch = 1024;  // (block, slot) pairs staged per round
constexpr int kAttnThreads = 256;

__device__ __forceinline__ unsigned long long umin64(unsigned long long a, unsigned long long b) {
  return a < b ? a : b;
}

struct PlanSmem {
  int owner[kMaxSlots];
  int last[kMaxSlots];
  unsigned char prot[kMaxSlots];
  unsigned char hit[kMaxSlots];  // per selection entry: resident at entry
  int copy_j[kMaxSlots];
  int copy_s[kMaxSlots];
  int ncopy, hits, evict;
};

// Runs the victim rule of one stream and updates its tables.  Returns the
// stream's selection count (entries of `my_sel`), or -1 when the selection
// does not fit (HS_EBIT_CAPACITY; the stream is left untouched).  Afterwards
// sm.copy_j/copy_s hold the sm.ncopy (block, slot) pairs to fill and sm.hit[i]
// says whether entry i was a hit.  All threads of the CTA call it.
__device__ int plan_stream(const HotView& hb, const int32_t* my_sel, int cnt, int capacity, int step, int pair,
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
    sm.hit[i] = 0;
    if (j < 0 || j >= hb.max_blocks) continue;
    const int g = pt[j];
    if (g >= 0) {
      const int s = g - base;
      if (s < 0 || s >= S) { set_error(err, HS_EBIT_PAGE_RANGE); continue; }
      sm.prot[s] = 1;
      sm.last[s] = step;
      sm.hit[i] = 1;
      atomicAdd(&sm.hits, 1);
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
      if (pt[j] >= 0) continue;  // a hit
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

__device__ __forceinline__ int64_t page_bytes_of(const HotView& hb) {
  const int elem = hb.kv_dtype == HS_KV_F32 ? 4 : (hb.kv_dtype == HS_KV_BF16 ? 2 : 1);
  return static_cast<int64_t>(hb.block) * hb.head_dim * elem;
}

__device__ __forceinline__ int64_t scale_bytes_of(const HotView& hb) {
  return hb.kv_dtype == HS_KV_FP8E4M3_G32 ? static_cast<int64_t>(hb.block) * (hb.head_dim / kQuantGroup) * 4 : 0;
}

// Copies `n` pages of one stream (pool page pool_pair + js[c] -> slot
// base + ss[c]), K and V and, for e4m3, their scales, with all threads of the
// CTA; each thread keeps kCopyUnroll 16-byte loads in flight.
template <typename JS, typename SS>
__device__ void copy_pages(const HotView& hb, int pair, int n, JS js, SS ss) {
  const int64_t pool_pair = static_cast<int64_t>(pair) * hb.max_blocks;
  const int64_t base = static_cast<int64_t>(pair) * hb.slots;
  const int64_t page_bytes = page_bytes_of(hb);
  const int64_t vpp = page_bytes / 16;
  const int64_t total = static_cast<int64_t>(n) * vpp * 2;  // K then V
  for (int64_t v0 = threadIdx.x; v0 < total; v0 += static_cast<int64_t>(blockDim.x) * kCopyUnroll) {
    uint4 buf[kCopyUnroll];
    uint4* dst[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t v = v0 + static_cast<int64_t>(u) * blockDim.x;
      dst[u] = nullptr;
      if (v < total) {
        const int which = v >= n * vpp;  // 0 = K, 1 = V
        const int64_t w = v - which * n * vpp;
        const int c = static_cast<int>(w / vpp);
        const int64_t off = w - c * vpp;
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const char*>(which ? hb.host_v : hb.host_k) +
                                                          (pool_pair + js(c)) * page_bytes) + off;
        dst[u] = reinterpret_cast<uint4*>(static_cast<char*>(which ? hb.v_slots : hb.k_slots) +
                                          (base + ss(c)) * page_bytes) + off;
        buf[u] = __ldcs(src);
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (dst[u]) *dst[u] = buf[u];
  }
  if (hb.kv_dtype == HS_KV_FP8E4M3_G32) {
    const int sc_per_page = hb.block * (hb.head_dim / kQuantGroup);
    const int64_t total_sc = static_cast<int64_t>(n) * sc_per_page;
    for (int64_t v = threadIdx.x; v < 2 * total_sc; v += blockDim.x) {
      const int which = v >= total_sc;
      const int64_t w = v - which * total_sc;
      const int c = static_cast<int>(w / sc_per_page);
      const int64_t off = w % sc_per_page;
      const float* src = (which ? hb.host_v_scales : hb.host_k_scales) + (pool_pair + js(c)) * sc_per_page + off;
      float* dst = (which ? hb.v_slot_scales : hb.k_slot_scales) + (base + ss(c)) * sc_per_page + off;
      *dst = __ldcs(src);
    }
  }
}

__global__ __launch_bounds__(kThreads) void swapin_kernel(HotView hb, const int32_t* __restrict__ sel,
                                                          const int32_t* __restrict__ sel_count,
                                                          int capacity, int step,
                                                          hs_swap_stats* stats, unsigned* err) {
  __shared__ PlanSmem sm;
  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x;
  const int32_t* my_sel = sel + static_cast<int64_t>(pair) * capacity;
  if (plan_stream(hb, my_sel, sel_count[pair], capacity, step, pair, sm, err) < 0) return;
  const int ncopy = sm.ncopy;
  copy_pages(hb, pair, ncopy, [&](int c) { return sm.copy_j[c]; }, [&](int c) { return sm.copy_s[c]; });
  if (stats && threadIdx.x == 0) {
    atomicAdd(&stats->hits, static_cast<unsigned long long>(sm.hits));
    atomicAdd(&stats->misses, static_cast<unsigned long long>(ncopy));
    atomicAdd(&stats->evictions, static_cast<unsigned long long>(sm.evict));
    atomicAdd(&stats->bytes_in, static_cast<unsigned long long>(ncopy) * 2ull *
                                    static_cast<unsigned long long>(page_bytes_of(hb) + scale_bytes_of(hb)));
  }
}

// Plan only: tables updated, hit and miss lists written in the selection
// layout ([pair][capacity], ascending, -1 padded) with their counts.
__global__ __launch_bounds__(kThreads) void swapin_plan_kernel(HotView hb, const int32_t* __restrict__ sel,
                                                               const int32_t* __restrict__ sel_count,
                                                               int capacity, int step, int32_t* hit_sel,
                                                               int32_t* hit_count, int32_t* miss_sel,
                                                               int32_t* miss_count, hs_swap_stats* stats,
                                                               unsigned* err) {
  __shared__ PlanSmem sm;
  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x;
  const int64_t row = static_cast<int64_t>(pair) * capacity;
  const int32_t* my_sel = sel + row;
  const int cnt = plan_stream(hb, my_sel, sel_count[pair], capacity, step, pair, sm, err);
  int nh = 0, nm = 0;
  if (cnt > 0 && threadIdx.x < 32) {  // warp 0 compacts hits and misses in selection order
    const int lane = threadIdx.x;
    for (int i0 = 0; i0 < cnt; i0 += 32) {
      const int i = i0 + lane;
      const int j = i < cnt ? my_sel[i] : -1;
      const bool valid = i < cnt && j >= 0 && j < hb.max_blocks;
      const bool h = valid && sm.hit[i];
      const bool m = valid && !sm.hit[i];
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

// Attention of one stream's query heads over the blocks it has just copied:
// the part of the selection's attention that the attention over the hits
// leaves out.  Normalised output and natural-log lse per query head, to be
// combined with the hits' part by the LSE merge.
struct MissAttn {
  const void* q;            // [batch][Hq][D]: f32 for f32 K/V, bf16 otherwise
  const int32_t* seq_lens;  // [batch]
  float* out;               // [batch][Hq][D]
  float* lse;               // [batch][Hq]
  float scale_log2;         // scale * log2(e)
  int hq, group;
};

constexpr int kMaxGroup = 16;
constexpr int kSub = 64;  // token rows of a block staged in shared memory at a time

template <int KIND>
constexpr int elem_size() { return KIND == HS_KV_F32 ? 4 : (KIND == HS_KV_BF16 ? 2 : 1); }

// Dynamic shared memory of the copied-blocks attention: K and V rows of a
// sub-block (+ e4m3 scales) and q of the group.
// K/V rows are staged with a stride of one row plus four elements, so that
// threads reading four consecutive elements of consecutive rows hit distinct
// banks.
template <int C, int KIND>
struct AttendSmem {
  static constexpr int D = C * 32;
  static constexpr int kRowBytes = D * elem_size<KIND>();
  static constexpr int kStride = kRowBytes + 4 * elem_size<KIND>();
  static constexpr int kScaleRow = KIND == HS_KV_FP8E4M3_G32 ? (D / kQuantGroup) * 4 : 0;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kSub * kStride;
  static constexpr int kOffKs = (kOffV + kSub * kStride + 15) / 16 * 16;
  static constexpr int kOffVs = kOffKs + kSub * kScaleRow;
  static constexpr int kOffQ = (kOffVs + kSub * kScaleRow + 15) / 16 * 16;
  static constexpr int kBytes = kOffQ + kMaxGroup * D * 4;
};

// Channel d of staged row t, as the attention sees it (e4m3: code * scale).
template <int C, int KIND>
__device__ __forceinline__ float staged_val(const uint8_t* rows, const float* scales, int t, int d) {
  constexpr int D = C * 32;
  const uint8_t* r = rows + t * AttendSmem<C, KIND>::kStride;
  if constexpr (KIND == HS_KV_F32) {
    return reinterpret_cast<const float*>(r)[d];
  } else if constexpr (KIND == HS_KV_BF16) {
    return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(r)[d]);
  } else {
    return e4m3x2_to_float2(static_cast<uint16_t>(r[d])).x * scales[t * (D / kQuantGroup) + d / kQuantGroup];
  }
}

// Channels d0 .. d0+3 of staged row t (d0 a multiple of 4), one load.
template <int C, int KIND>
__device__ __forceinline__ float4 staged_val4(const uint8_t* rows, const float* scales, int t, int d0) {
  constexpr int D = C * 32;
  const uint8_t* r = rows + t * AttendSmem<C, KIND>::kStride;
  if constexpr (KIND == HS_KV_F32) {
    return *reinterpret_cast<const float4*>(r + d0 * 4);
  } else if constexpr (KIND == HS_KV_BF16) {
    const uint2 u = *reinterpret_cast<const uint2*>(r + d0 * 2);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xffff0000u));
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(r + d0);
    const float sc = scales[t * (D / kQuantGroup) + d0 / kQuantGroup];
    const float2 a = e4m3x2_to_float2(static_cast<uint16_t>(u & 0xffffu));
    const float2 b = e4m3x2_to_float2(static_cast<uint16_t>(u >> 16));
    return make_float4(a.x * sc, a.y * sc, b.x * sc, b.y * sc);
  }
}

// Copy only: the pages of the miss lists written by swapin_plan_kernel, whose
// slots the page table now names.  The misses of all streams, in stream
// order, are cut into one equal share per CTA, so that every CTA keeps its
// 16-byte host loads in flight however the misses fall on the streams (a CTA
// per stream in turn would wait out a host round trip per stream).  Each CTA
// finds its share with two passes over the miss counts (total, then the
// prefix of the streams it touches), resolves up to kCopyBatch misses at a
// time to (stream, block, slot) and copies them with all its threads.
__device__ __forceinline__ int clamp_misses(int n, int capacity, int S) {
  n = n < 0 ? 0 : (n > capacity ? capacity : n);
  return n > S ? S : n;
}

__global__ __launch_bounds__(kCopyThreads, 1) void swapin_copy_kernel(HotView hb, const int32_t* __restrict__ miss_sel,
                                                                      const int32_t* __restrict__ miss_count,
                                                                      int capacity, hs_swap_stats* stats,
                                                                      unsigned* err) {
  __shared__ int s_p[kCopyBatch];  // stream of each miss of the window (-1: skipped)
  __shared__ int s_j[kCopyBatch];  // its block, then (resolved) its pool page offset
  __shared__ int s_s[kCopyBatch];  // its slot
  __shared__ int s_warp[kCopyThreads / 32];
  // No early trigger: CTAs of a dependent launched early would wait on SMs
  // that the attention running beside the copy needs.
  pdl_wait();  // (a no-op unless launched as a programmatic dependent)
  const int pairs = hb.batch * hb.hkv;
  const int S = hb.slots;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kW = kCopyThreads / 32;
  // inclusive block scan of one value per thread (the tile's running sum is in *tot)
  auto block_scan = [&](int v, long long* tot) -> int {
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int wv = lane < kW ? s_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wv, o);
        if (lane >= o) wv += y;
      }
      if (lane < kW) s_warp[lane] = wv;
    }
    __syncthreads();
    const int incl = x + (warp > 0 ? s_warp[warp - 1] : 0);
    *tot = s_warp[kW - 1];
    __syncthreads();  // s_warp is reused by the next tile
    return incl;
  };
  // pass 1: all misses
  long long total = 0;
  for (int p0 = 0; p0 < pairs; p0 += kCopyThreads) {
    const int p = p0 + tid;
    long long t;
    block_scan(p < pairs ? clamp_misses(miss_count[p], capacity, S) : 0, &t);
    total += t;
  }
  const long long lo = total * blockIdx.x / gridDim.x, hi = total * (blockIdx.x + 1) / gridDim.x;
  const int64_t page_bytes = page_bytes_of(hb);
  const int vpp = static_cast<int>(page_bytes / 16);
  unsigned long long pages = 0;
  for (long long w0 = lo; w0 < hi; w0 += kCopyBatch) {
    const long long w1 = min(hi, w0 + kCopyBatch);
    const int m = static_cast<int>(w1 - w0);
    // pass 2: the streams whose misses fall in [w0, w1) list them
    long long carry = 0;
    for (int p0 = 0; p0 < pairs && carry < w1; p0 += kCopyThreads) {
      const int p = p0 + tid;
      const int n = p < pairs ? clamp_misses(miss_count[p], capacity, S) : 0;
      long long t;
      const long long pre = carry + block_scan(n, &t) - n;  // misses before stream p
      for (long long k = max(pre, w0); k < min(pre + n, w1); ++k) {
        s_p[k - w0] = p;
        s_j[k - w0] = static_cast<int>(k - pre);  // index in the stream's miss list
      }
      carry += t;
    }
    __syncthreads();
    // resolve: block and slot of each miss of the window
    for (int e = tid; e < m; e += kCopyThreads) {
      const int p = s_p[e];
      const int j = miss_sel[static_cast<int64_t>(p) * capacity + s_j[e]];
      int sl = -1;
      if (j < 0 || j >= hb.max_blocks) {
        set_error(err, HS_EBIT_BLOCK_RANGE);
      } else {
        sl = hb.page_table[static_cast<int64_t>(p) * hb.max_blocks + j] - p * S;
        if (sl < 0 || sl >= S) {
          set_error(err, HS_EBIT_PAGE_RANGE);
          sl = -1;
        }
      }
      s_j[e] = j;
      s_s[e] = sl;
      if (sl < 0) s_p[e] = -1;
    }
    __syncthreads();
    // copy: K then V of every miss, kCopyUnroll 16-byte host loads in flight per thread
    const int64_t vtot = static_cast<int64_t>(m) * vpp * 2;
    for (int64_t v0 = tid; v0 < vtot; v0 += static_cast<int64_t>(kCopyThreads) * kCopyUnroll) {
      uint4 buf[kCopyUnroll];
      uint4* dst[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t v = v0 + static_cast<int64_t>(u) * kCopyThreads;
        dst[u] = nullptr;
        if (v < vtot) {
          const int which = v >= static_cast<int64_t>(m) * vpp;  // 0 = K, 1 = V
          const int w = static_cast<int>(v - which * static_cast<int64_t>(m) * vpp);
          const int e = w / vpp, off = w - e * vpp;
          const int p = s_p[e];
          if (p >= 0) {
            const uint4* src = reinterpret_cast<const uint4*>(
                                   static_cast<const char*>(which ? hb.host_v : hb.host_k) +
                                   (static_cast<int64_t>(p) * hb.max_blocks + s_j[e]) * page_bytes) + off;
            dst[u] = reinterpret_cast<uint4*>(static_cast<char*>(which ? hb.v_slots : hb.k_slots) +
                                              (static_cast<int64_t>(p) * S + s_s[e]) * page_bytes) + off;
            buf[u] = __ldcs(src);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u)
        if (dst[u]) *dst[u] = buf[u];
    }
    if (hb.kv_dtype == HS_KV_FP8E4M3_G32) {
      const int spp = hb.block * (hb.head_dim / kQuantGroup);  // scales per page
      for (int v = tid; v < 2 * m * spp; v += kCopyThreads) {
        const int which = v >= m * spp;
        const int w = v - which * m * spp;
        const int e = w / spp, off = w - e * spp;
        const int p = s_p[e];
        if (p < 0) continue;
        const float* src = (which ? hb.host_v_scales : hb.host_k_scales) +
                           (static_cast<int64_t>(p) * hb.max_blocks + s_j[e]) * spp + off;
        float* dst = (which ? hb.v_slot_scales : hb.k_slot_scales) + (static_cast<int64_t>(p) * S + s_s[e]) * spp + off;
        *dst = __ldcs(src);
      }
    }
    if (stats && tid == 0)
      for (int e = 0; e < m; ++e) pages += s_p[e] >= 0 ? 1 : 0;
    __syncthreads();  // the window's lists are refilled next
  }
  if (stats && pages)
    atomicAdd(&stats->bytes_in, pages * 2ull * static_cast<unsigned long long>(page_bytes + scale_bytes_of(hb)));
}

// Attention of one stream's query heads over the blocks of its miss list,
// read from the slots the copy filled.  One CTA per stream (streams without
// misses only write lse = -inf).  Per block, in pieces of up to kSub valid
// tokens, the rows are staged in shared memory (16-byte loads, padded rows);
// then each warp takes whole heads (warp w: heads w, w + 8) with no further
// barrier: lane t scores tokens t and t + 32, the warp's shuffles give the
// running max and sum, and lane t accumulates p * v for channels
// [C t, C t + C).
template <int C, int KIND>
__global__ __launch_bounds__(kAttnThreads) void copied_blocks_attn_kernel(HotView hb,
                                                                         const int32_t* __restrict__ miss_sel,
                                                                         const int32_t* __restrict__ miss_count,
                                                                         int capacity, MissAttn ma, unsigned* err) {
  using Ly = AttendSmem<C, KIND>;
  constexpr int D = C * 32;
  constexpr int kWarps = kAttnThreads / 32;
  constexpr int kHpw = (kMaxGroup + kWarps - 1) / kWarps;  // heads per warp
  static_assert(kSub == 64, "two token rows per lane");
  extern __shared__ __align__(16) uint8_t dyn[];
  float* s_q = reinterpret_cast<float*>(dyn + Ly::kOffQ);
  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x;
  const int S = hb.slots;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = ma.group;
  const int b = pair / hb.hkv, kvh = pair - b * hb.hkv;
  const int64_t qrow0 = static_cast<int64_t>(b) * ma.hq + static_cast<int64_t>(kvh) * g;
  int n = miss_count[pair];
  n = n < 0 ? 0 : (n > capacity ? capacity : n);
  n = n > S ? S : n;
  if (n == 0) {
    if (tid < g) ma.lse[qrow0 + tid] = -INFINITY;
    return;
  }
  const int64_t row = static_cast<int64_t>(pair) * capacity;
  const int32_t* pt = hb.page_table + static_cast<int64_t>(pair) * hb.max_blocks;
  const int L = ma.seq_lens[b];
  const int B = hb.block;
  for (int i = tid; i < g * D; i += kAttnThreads) {
    const int64_t e = qrow0 * D + i;  // heads of the group are consecutive rows
    s_q[i] = KIND == HS_KV_F32 ? static_cast<const float*>(ma.q)[e]
                               : bf16_bits_to_float(static_cast<const uint16_t*>(ma.q)[e]);
  }
  // per head of this warp: running max and sum (log2 units), p * v of its C channels
  float m[kHpw], l[kHpw], acc[kHpw][C];
#pragma unroll
  for (int k = 0; k < kHpw; ++k) {
    m[k] = -INFINITY;
    l[k] = 0.0f;
#pragma unroll
    for (int c = 0; c < C; ++c) acc[k][c] = 0.0f;
  }
  const float* ksc = reinterpret_cast<const float*>(dyn + Ly::kOffKs);
  const float* vsc = reinterpret_cast<const float*>(dyn + Ly::kOffVs);
  for (int c = 0; c < n; ++c) {
    const int j = miss_sel[row + c];
    if (j < 0 || j >= hb.max_blocks) continue;  // reported by the copy
    const int sl = pt[j] - pair * S;
    if (sl < 0 || sl >= S) continue;
    const int nv = min(B, L - j * B);  // valid tokens of the block (uniform)
    const int64_t row0 = (static_cast<int64_t>(pair) * S + sl) * B;
    for (int r0 = 0; r0 < nv; r0 += kSub) {
      const int rows = min(kSub, nv - r0);
      __syncthreads();  // every warp is done with the previous piece (and q is in)
      {  // stage K and V rows (and scales): 16-byte loads, 4-byte stores into the padded rows
        constexpr int kVecRow = Ly::kRowBytes / 16;
        const int vec = rows * kVecRow;
        const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(hb.k_slots) +
                                                         (row0 + r0) * Ly::kRowBytes);
        const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(hb.v_slots) +
                                                         (row0 + r0) * Ly::kRowBytes);
        for (int v = tid; v < 2 * vec; v += kAttnThreads) {
          const int w = v < vec ? v : v - vec;
          const uint4 x = v < vec ? ks[w] : vs[w];
          uint32_t* dst = reinterpret_cast<uint32_t*>(dyn + (v < vec ? Ly::kOffK : Ly::kOffV) +
                                                      (w / kVecRow) * Ly::kStride + (w % kVecRow) * 16);
          dst[0] = x.x;
          dst[1] = x.y;
          dst[2] = x.z;
          dst[3] = x.w;
        }
        if constexpr (KIND == HS_KV_FP8E4M3_G32) {
          constexpr int G = D / kQuantGroup;
          for (int v = tid; v < 2 * rows * G; v += kAttnThreads) {
            if (v < rows * G)
              reinterpret_cast<float*>(dyn + Ly::kOffKs)[v] = hb.k_slot_scales[(row0 + r0) * G + v];
            else
              reinterpret_cast<float*>(dyn + Ly::kOffVs)[v - rows * G] = hb.v_slot_scales[(row0 + r0) * G + v - rows * G];
          }
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < kHpw; ++k) {
        const int h = warp + k * kWarps;
        if (h >= g) break;  // the same for the whole warp
        const float4* qv = reinterpret_cast<const float4*>(s_q + h * D);
        // scores of tokens lane and lane + 32 (two chains each)
        const int t0 = min(lane, rows - 1), t1 = min(lane + 32, rows - 1);
        float a0 = 0.0f, a1 = 0.0f, b0 = 0.0f, b1 = 0.0f;
#pragma unroll 8
        for (int d4 = 0; d4 < D / 4; ++d4) {
          const float4 q4 = qv[d4];
          const float4 x = staged_val4<C, KIND>(dyn + Ly::kOffK, ksc, t0, d4 * 4);
          const float4 y = staged_val4<C, KIND>(dyn + Ly::kOffK, ksc, t1, d4 * 4);
          a0 = fmaf(q4.x, x.x, a0);
          a1 = fmaf(q4.y, x.y, a1);
          a0 = fmaf(q4.z, x.z, a0);
          a1 = fmaf(q4.w, x.w, a1);
          b0 = fmaf(q4.x, y.x, b0);
          b1 = fmaf(q4.y, y.y, b1);
          b0 = fmaf(q4.z, y.z, b0);
          b1 = fmaf(q4.w, y.w, b1);
        }
        const float s0 = lane < rows ? (a0 + a1) * ma.scale_log2 : -INFINITY;
        const float s1 = lane + 32 < rows ? (b0 + b1) * ma.scale_log2 : -INFINITY;
        const float mn = fmaxf(m[k], warp_max(fmaxf(s0, s1)));
        const float alpha = m[k] == -INFINITY ? 0.0f : exp2f(m[k] - mn);
        const float p0 = s0 == -INFINITY ? 0.0f : exp2f(s0 - mn);
        const float p1 = s1 == -INFINITY ? 0.0f : exp2f(s1 - mn);
        l[k] = l[k] * alpha + warp_sum(p0 + p1);
        m[k] = mn;
#pragma unroll
        for (int cc = 0; cc < C; ++cc) acc[k][cc] *= alpha;
        // p * v: token t's probability from lane t % 32
        for (int t = 0; t < rows; ++t) {
          const float pt_ = __shfl_sync(0xffffffffu, t < 32 ? p0 : p1, t & 31);
          if constexpr (C == 4) {
            const float4 v4 = staged_val4<C, KIND>(dyn + Ly::kOffV, vsc, t, lane * 4);
            acc[k][0] = fmaf(pt_, v4.x, acc[k][0]);
            acc[k][1] = fmaf(pt_, v4.y, acc[k][1]);
            acc[k][2] = fmaf(pt_, v4.z, acc[k][2]);
            acc[k][3] = fmaf(pt_, v4.w, acc[k][3]);
          } else {
#pragma unroll
            for (int cc = 0; cc < C; ++cc)
              acc[k][cc] = fmaf(pt_, staged_val<C, KIND>(dyn + Ly::kOffV, vsc, t, lane * C + cc), acc[k][cc]);
          }
        }
      }
    }
  }
  // normalised output and lse of this warp's heads
#pragma unroll
  for (int k = 0; k < kHpw; ++k) {
    const int h = warp + k * kWarps;
    if (h >= g) break;
    const float lk = l[k];
    if (lk > 0.0f) {
#pragma unroll
      for (int cc = 0; cc < C; ++cc) ma.out[(qrow0 + h) * D + lane * C + cc] = acc[k][cc] / lk;
    }
    if (lane == 0) ma.lse[qrow0 + h] = lk > 0.0f ? (m[k] + log2f(lk)) * 0.6931471805599453f : -INFINITY;
  }
  (void)err;
}

}  // namespace

template <int C, int KIND>
cudaError_t launch_attend(const HotView& hb, const int32_t* miss_sel, const int32_t* miss_count, int capacity,
                          const MissAttn& ma, unsigned* err, cudaStream_t st) {
  constexpr int kBytes = AttendSmem<C, KIND>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(copied_blocks_attn_kernel<C, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(copied_blocks_attn_kernel<C, KIND>, dim3(hb.batch * hb.hkv), dim3(kAttnThreads), kBytes, st, hb,
                    miss_sel, miss_count, capacity, ma, err);
}

cudaError_t launch_swapin(const HotView& hb, const int32_t* sel, const int32_t* sel_count,
                          int capacity, int step, hs_swap_stats* stats, unsigned* err,
                          cudaStream_t st) {
  const int pairs = hb.batch * hb.hkv;
  if (pairs == 0) return cudaSuccess;
  return launch_pdl(swapin_kernel, dim3(pairs), dim3(kThreads), 0, st, hb, sel, sel_count, capacity, step,
                    stats, err);
}

cudaError_t launch_swapin_plan(const HotView& hb, const int32_t* sel, const int32_t* sel_count, int capacity,
                               int step, int32_t* hit_sel, int32_t* hit_count, int32_t* miss_sel,
                               int32_t* miss_count, hs_swap_stats* stats, unsigned* err, cudaStream_t st) {
  const int pairs = hb.batch * hb.hkv;
  if (pairs == 0) return cudaSuccess;
  return launch_pdl(swapin_plan_kernel, dim3(pairs), dim3(kThreads), 0, st, hb, sel, sel_count, capacity, step,
                    hit_sel, hit_count, miss_sel, miss_count, stats, err);
}

cudaError_t launch_swapin_copy(const HotView& hb, const int32_t* miss_sel, const int32_t* miss_count,
                               int capacity, int ctas, const MissAttnArgs* attn, hs_swap_stats* stats, unsigned* err,
                               cudaStream_t st) {
  const int pairs = hb.batch * hb.hkv;
  if (pairs == 0) return cudaSuccess;
  const int grid = ctas < pairs ? ctas : pairs;
  // A plain launch: the copy usually follows a wait on another stream's plan,
  // which it must not overtake.
  swapin_copy_kernel<<<grid, kCopyThreads, 0, st>>>(hb, miss_sel, miss_count, capacity, stats, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !attn) return e;
  MissAttn ma{};
  ma.q = attn->q;
  ma.seq_lens = attn->seq_lens;
  ma.out = attn->out;
  ma.lse = attn->lse;
  ma.scale_log2 = attn->scale * 1.4426950408889634f;
  ma.hq = attn->hq;
  ma.group = attn->hq / hb.hkv;
  if (hb.head_dim == 128) {
    if (hb.kv_dtype == HS_KV_F32) return launch_attend<4, HS_KV_F32>(hb, miss_sel, miss_count, capacity, ma, err, st);
    if (hb.kv_dtype == HS_KV_BF16) return launch_attend<4, HS_KV_BF16>(hb, miss_sel, miss_count, capacity, ma, err, st);
    return launch_attend<4, HS_KV_FP8E4M3_G32>(hb, miss_sel, miss_count, capacity, ma, err, st);
  }
  if (hb.kv_dtype == HS_KV_F32) return launch_attend<2, HS_KV_F32>(hb, miss_sel, miss_count, capacity, ma, err, st);
  if (hb.kv_dtype == HS_KV_BF16) return launch_attend<2, HS_KV_BF16>(hb, miss_sel, miss_count, capacity, ma, err, st);
  return launch_attend<2, HS_KV_FP8E4M3_G32>(hb, miss_sel, miss_count, capacity, ma, err, st);
}

}  // namespace hs
