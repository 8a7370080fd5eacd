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
#include "swapin_plan.cuh"
#include "tc_ptx.cuh"

namespace hs {
namespace {

constexpr int kThreads = 256;
// The copy kernel runs on a few SMs of its own (the attention CTAs beside it
// fill the SMs' shared memory): large CTAs keep many host loads in flight.
constexpr int kCopyThreads = 1024;
constexpr int kCopyUnroll = 4;
constexpr int kCopyBatch = 1024;  // (block, slot) pairs staged per round
constexpr int kAttnThreads = 256;

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
  __shared__ plan::PlanSmem sm;
  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x;
  const int32_t* my_sel = sel + static_cast<int64_t>(pair) * capacity;
  if (plan::plan_stream(hb, my_sel, sel_count[pair], capacity, step, pair, sm, err) < 0) return;
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
  __shared__ plan::PlanSmem sm;
  pdl_trigger();
  pdl_wait();
  const int pair = blockIdx.x;
  const int64_t row = static_cast<int64_t>(pair) * capacity;
  const int32_t* my_sel = sel + row;
  const int cnt = plan::plan_stream(hb, my_sel, sel_count[pair], capacity, step, pair, sm, err);
  plan::write_lists(hb, my_sel, cnt, capacity, pair, sm, hit_sel, hit_count, miss_sel, miss_count, stats);
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
constexpr int kMissWin = 64;  // misses of a stream resolved at a time by the copied-blocks attention

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
  {  // q of the group (consecutive rows): every load of a thread in flight before its first store
    constexpr int kQPer = (kMaxGroup * D + kAttnThreads - 1) / kAttnThreads;
    float qv[kQPer];
#pragma unroll
    for (int u = 0; u < kQPer; ++u) {
      const int i = tid + u * kAttnThreads;
      const int64_t e = qrow0 * D + i;
      qv[u] = i >= g * D ? 0.0f
                         : (KIND == HS_KV_F32 ? static_cast<const float*>(ma.q)[e]
                                              : bf16_bits_to_float(static_cast<const uint16_t*>(ma.q)[e]));
    }
#pragma unroll
    for (int u = 0; u < kQPer; ++u)
      if (tid + u * kAttnThreads < g * D) s_q[tid + u * kAttnThreads] = qv[u];
  }
  // the stream's misses resolved up front, kMissWin at a time: block and slot
  // (-1: skipped, reported by the copy)
  __shared__ int s_mj[kMissWin], s_ms[kMissWin];
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
    if (c % kMissWin == 0) {
      __syncthreads();  // the previous window is used up
      if (tid < kMissWin && c + tid < n) {
        const int j = miss_sel[row + c + tid];
        int sl = -1;
        if (j >= 0 && j < hb.max_blocks) {
          sl = pt[j] - pair * S;
          if (sl >= S) sl = -1;
        }
        s_mj[tid] = j;
        s_ms[tid] = sl < 0 ? -1 : sl;
      }
      __syncthreads();
    }
    const int j = s_mj[c % kMissWin], sl = s_ms[c % kMissWin];
    if (sl < 0) continue;  // the same for every thread
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
        constexpr int kPer = (2 * kSub * kVecRow + kAttnThreads - 1) / kAttnThreads;
        uint4 xs[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {  // every load of a thread in flight before its first store
          const int v = tid + u * kAttnThreads;
          const int w = v < vec ? v : v - vec;
          if (v < 2 * vec) xs[u] = v < vec ? ks[w] : vs[w];
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int v = tid + u * kAttnThreads;
          if (v >= 2 * vec) break;
          const int w = v < vec ? v : v - vec;
          uint32_t* dst = reinterpret_cast<uint32_t*>(dyn + (v < vec ? Ly::kOffK : Ly::kOffV) +
                                                      (w / kVecRow) * Ly::kStride + (w % kVecRow) * 16);
          dst[0] = xs[u].x;
          dst[1] = xs[u].y;
          dst[2] = xs[u].z;
          dst[3] = xs[u].w;
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

// The same for bf16 K/V and head_dim 128 on the tensor cores (warp-level
// mma.sync m16n8k16, bf16 products exact, fp32 accumulation): the copied
// blocks are a few hundred scattered tiles, too small for a tcgen05 pipeline.
// One CTA of 4 warps per stream; warp w takes tokens [16 w, 16 w + 16) of
// every 64-token piece of every missed block: S (16 padded heads x 16 tokens)
// = Q.K^T over 8 k-steps of 16 channels, the online softmax per head row
// (quad shuffles), then O (16 heads x 128 channels) += P.V with P as bf16
// high part + remainder (the S accumulators are the A fragments of P).  The
// warps' states are combined through shared memory at the end.
constexpr int kMmaWarps = 4;
constexpr int kMmaRow = 128 * 2 + 16;  // staged row: 128 bf16 + 16 bytes (ldmatrix rows hit distinct banks)
constexpr int kMmaStage = 16 * kMmaRow;  // one warp's 16 rows of K (or V)
constexpr int kMmaSmem = 16 * kMmaRow + kMmaWarps * 2 * kMmaStage;  // Q, then per warp K and V
static_assert(kMmaSmem >= kMmaWarps * (16 * 128 + 32) * 4, "the warps' states fit the staging area");

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// D += A.B, m16n8k16, bf16 inputs, fp32 accumulators
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
               "{%0, %1, %2, %3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// 16-byte global -> shared copy, the bytes past src_bytes zero-filled
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ __launch_bounds__(kMmaWarps * 32) void copied_blocks_attn_mma_kernel(HotView hb,
                                                                               const int32_t* __restrict__ miss_sel,
                                                                               const int32_t* __restrict__ miss_count,
                                                                               int capacity, MissAttn ma,
                                                                               unsigned* err) {
  constexpr int D = 128;
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ int s_mj[kMissWin], s_ms[kMissWin];
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
  const uint32_t sq = tc::smem_u32(dyn);
  uint8_t* kst = dyn + 16 * kMmaRow + warp * 2 * kMmaStage;  // this warp's K rows, then its V rows
  uint8_t* vst = kst + kMmaStage;
  {  // Q of the group, 16 rows (zero past g), bf16
    const int r = tid >> 3, seg = tid & 7;  // 128 threads: row r (0..15), 16-byte segments seg and seg + 8
    uint4 x0 = make_uint4(0, 0, 0, 0), x1 = x0;
    if (r < g) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(ma.q) + (qrow0 + r) * D);
      x0 = src[seg];
      x1 = src[seg + 8];
    }
    *reinterpret_cast<uint4*>(dyn + r * kMmaRow + seg * 16) = x0;
    *reinterpret_cast<uint4*>(dyn + r * kMmaRow + (seg + 8) * 16) = x1;
  }
  const int q4 = lane & 3, r8 = lane >> 2;  // fragment coordinates
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};  // rows r8, r8 + 8
  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  for (int c = 0; c < n; ++c) {
    if (c % kMissWin == 0) {
      __syncthreads();  // the previous window is used up (and Q is in)
      if (tid < kMissWin && c + tid < n) {
        const int j = miss_sel[row + c + tid];
        int sl = -1;
        if (j >= 0 && j < hb.max_blocks) {
          sl = pt[j] - pair * S;
          if (sl >= S) sl = -1;
        }
        s_mj[tid] = j;
        s_ms[tid] = sl < 0 ? -1 : sl;
      }
      __syncthreads();
    }
    const int j = s_mj[c % kMissWin], sl = s_ms[c % kMissWin];
    if (sl < 0) continue;  // reported by the copy; the same for every thread
    const int nv = min(B, L - j * B);  // valid tokens of the block
    const int64_t row0 = (static_cast<int64_t>(pair) * S + sl) * B;
    for (int r0 = 0; r0 < nv; r0 += 64) {
      const int t0 = r0 + 16 * warp;  // this warp's first token of the piece
      const int rows = min(16, nv - t0);
      if (rows <= 0) continue;  // the same for the whole warp
      {  // stage this warp's 16 K and V rows by asynchronous copies (zero fill past the valid tokens)
        const uint8_t* kg = static_cast<const uint8_t*>(hb.k_slots) + (row0 + t0) * (D * 2);
        const uint8_t* vg = static_cast<const uint8_t*>(hb.v_slots) + (row0 + t0) * (D * 2);
        __syncwarp();  // every lane is done with the previous piece's rows
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // 16 rows x 16 segments; lane takes segment lane & 15 of rows 2u + (lane >> 4)
          const int rr = 2 * u + (lane >> 4), seg = lane & 15;
          const int bytes = rr < rows ? 16 : 0;
          const int rs = rr < rows ? rr : 0;  // (a valid address even when nothing is read)
          cp_async16(tc::smem_u32(kst + rr * kMmaRow + seg * 16), kg + rs * (D * 2) + seg * 16, bytes);
          cp_async16(tc::smem_u32(vst + rr * kMmaRow + seg * 16), vg + rs * (D * 2) + seg * 16, bytes);
        }
        cp_async_wait_all();
        __syncwarp();
      }
      // S = Q.K^T: 16 heads x 16 tokens (two n-tiles of 8 tokens)
      float sc[2][4];
#pragma unroll
      for (int i = 0; i < 2; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.0f;
      const uint32_t kbase = tc::smem_u32(kst);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
        ldsm_x4(sq + ((lane & 7) + ((lane >> 3) & 1) * 8) * kMmaRow + (16 * ks + (lane >> 4) * 8) * 2, a0, a1, a2, a3);
        ldsm_x4(kbase + ((lane & 7) + (lane >> 4) * 8) * kMmaRow + (16 * ks + ((lane >> 3) & 1) * 8) * 2, b0, b1, b2,
                b3);
        mma_bf16_16816(sc[0], a0, a1, a2, a3, b0, b1);
        mma_bf16_16816(sc[1], a0, a1, a2, a3, b2, b3);
      }
      // online softmax per head row (rows r8 and r8 + 8; tokens 8 i + 2 q4 + {0, 1})
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float x[4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int tok = 8 * i + 2 * q4 + e;
            x[2 * i + e] = tok < rows ? sc[i][2 * h + e] * ma.scale_log2 : -INFINITY;
          }
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn = fmaxf(m[h], mx);
        alpha[h] = m[h] == -INFINITY ? (mn == -INFINITY ? 1.0f : 0.0f) : exp2f(m[h] - mn);
        float sum = 0.0f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[k] = x[k] == -INFINITY ? 0.0f : exp2f(x[k] - mn);
          sum += x[k];
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        l[h] = l[h] * alpha[h] + sum;
        m[h] = mn;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          sc[i][2 * h] = x[2 * i];
          sc[i][2 * h + 1] = x[2 * i + 1];
        }
      }
      // P as A fragments (bf16 high part + remainder)
      uint32_t ph[4], pl[4];
      {
        const float pv[4][2] = {{sc[0][0], sc[0][1]}, {sc[0][2], sc[0][3]}, {sc[1][0], sc[1][1]}, {sc[1][2], sc[1][3]}};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __nv_bfloat162 hi = __floats2bfloat162_rn(pv[k][0], pv[k][1]);
          const float2 hf = __bfloat1622float2(hi);
          ph[k] = *reinterpret_cast<const uint32_t*>(&hi);
          pl[k] = pack_bf16(pv[k][0] - hf.x, pv[k][1] - hf.y);
        }
      }
      // O = O * alpha + P.V over the 16 channel tiles
      const uint32_t vbase = tc::smem_u32(vst);
#pragma unroll
      for (int dt = 0; dt < 16; dt += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + ((lane & 7) + ((lane >> 3) & 1) * 8) * kMmaRow + (8 * dt + (lane >> 4) * 8) * 2, b0, b1, b2,
                  b3);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float (&od)[4] = o[dt + e];
          od[0] *= alpha[0];
          od[1] *= alpha[0];
          od[2] *= alpha[1];
          od[3] *= alpha[1];
          const uint32_t bb0 = e ? b2 : b0, bb1 = e ? b3 : b1;
          mma_bf16_16816(od, ph[0], ph[1], ph[2], ph[3], bb0, bb1);
          mma_bf16_16816(od, pl[0], pl[1], pl[2], pl[3], bb0, bb1);
        }
      }
    }
  }
  // combine the four warps' states through shared memory: per warp o [16][128], m [16], l [16]
  __syncthreads();  // every warp is done with its staging rows
  float* xo = reinterpret_cast<float*>(dyn);
  float* xm = xo + kMmaWarps * 16 * 128;
  float* xl = xm + kMmaWarps * 16;
#pragma unroll
  for (int dt = 0; dt < 16; ++dt) {
    const int d = 8 * dt + 2 * q4;
    float* w0 = xo + (warp * 16 + r8) * 128 + d;
    w0[0] = o[dt][0];
    w0[1] = o[dt][1];
    w0[8 * 128] = o[dt][2];
    w0[8 * 128 + 1] = o[dt][3];
  }
  if (q4 == 0) {
    xm[warp * 16 + r8] = m[0];
    xm[warp * 16 + r8 + 8] = m[1];
    xl[warp * 16 + r8] = l[0];
    xl[warp * 16 + r8 + 8] = l[1];
  }
  __syncthreads();
  // thread t: channel t of every head of the group
  for (int h = 0; h < g; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMmaWarps; ++w) M = fmaxf(M, xm[w * 16 + h]);
    float lt = 0.0f, acc = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kMmaWarps; ++w) {
        const float mw = xm[w * 16 + h];
        const float sw = mw == -INFINITY ? 0.0f : exp2f(mw - M);
        lt = fmaf(xl[w * 16 + h], sw, lt);
        acc = fmaf(xo[(w * 16 + h) * 128 + tid], sw, acc);
      }
    }
    if (lt > 0.0f) ma.out[(qrow0 + h) * D + tid] = acc / lt;
    if (tid == 0) ma.lse[qrow0 + h] = lt > 0.0f ? (M + log2f(lt)) * 0.6931471805599453f : -INFINITY;
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
    if (hb.kv_dtype == HS_KV_BF16) {
      cudaError_t e2 = cudaFuncSetAttribute(copied_blocks_attn_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            kMmaSmem);
      if (e2 != cudaSuccess) return e2;
      return launch_pdl(copied_blocks_attn_mma_kernel, dim3(hb.batch * hb.hkv), dim3(kMmaWarps * 32), kMmaSmem, st,
                        hb, miss_sel, miss_count, capacity, ma, err);
    }
    return launch_attend<4, HS_KV_FP8E4M3_G32>(hb, miss_sel, miss_count, capacity, ma, err, st);
  }
  if (hb.kv_dtype == HS_KV_F32) return launch_attend<2, HS_KV_F32>(hb, miss_sel, miss_count, capacity, ma, err, st);
  if (hb.kv_dtype == HS_KV_BF16) return launch_attend<2, HS_KV_BF16>(hb, miss_sel, miss_count, capacity, ma, err, st);
  return launch_attend<2, HS_KV_FP8E4M3_G32>(hb, miss_sel, miss_count, capacity, ma, err, st);
}

}  // namespace hs
