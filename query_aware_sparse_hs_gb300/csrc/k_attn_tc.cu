// Tensor-core gather-attention over the selected blocks (bf16 or e4m3 K/V,
// head_dim 128): "KV 稀疏化" wiki §5 (full attention on the chosen blocks only) with the
// tiled running-max / normaliser softmax of "分块稀疏注意力与KV Cache量化" §2.2.
//
// The g query heads that share a kv head make the decode step a real small GEMM
// per 128-token chunk:
//   S^T[128 tok x 16]   = K[128 tok x 128 d] . Qpad^T[128 d x 16]     (tcgen05, M=128 N=16)
//   O^T[128 d x 2*NH]   = V^T[128 d x 128 tok] . [P_hi | P_lo][128 tok x 2*NH]
// P is split into a bf16 high part and a bf16 remainder so the probabilities
// keep ~16 significant bits through the bf16 MMA; both accumulate in fp32 TMEM.
//
// Persistent, warp-specialised CTA (one per SM):
//   TMA producer warp: cp.async.bulk.tensor of each selected page's K and V
//               rows (two 64-channel halves, 128-byte swizzle) into a 3-stage
//               ring, completion tracked by mbarrier transaction bytes.
//   two MMA issuer warps (one thread each): S = K.Q^T and O = V^T.P; TMEM
//               double-buffers S and O.
//   softmax / correction warps: thread t owns TMEM lane t = token t of the
//               chunk for S, and channel t for O; running max and sum per head,
//               P written to shared memory for GEMM2, O accumulated in registers
//               with the online-softmax rescale.  The bf16 kernel has two such
//               groups working on alternate chunks, merged per work item.
// Every wait is bounded (2 s); on a time-out the CTA sets HS_EBIT_TIMEOUT,
// stops all roles, lets in-flight copies land and frees its TMEM.
#include <cooperative_groups.h>
#include <type_traits>
#include <cuda.h>

#include "bound_tile.cuh"
#include "hs_internal.h"
#include "select_pair.cuh"
#include "tc_ptx.cuh"

namespace cg = cooperative_groups;

namespace hs {
namespace {

using namespace tc;

constexpr int kD = 128;
constexpr int kChunk = 128;
constexpr int kStages = 3;
// e4m3 kernel roles: warps 0-3 and 15-18 the two softmax groups, 4-11 V code
// conversion, 12 TMA producer, 13 S' = K.Q'^T issuer (and TMEM owner),
// 14 and 19 the O' = V^T.P' issuers of the even and the odd chunks (an MMA
// takes its issuing thread ~70 cycles, so a chunk's eight P.V products are
// issued while the other group's are)
constexpr int kThreads = 640;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kMma2Warp = 14;
constexpr int kMma3Warp = 19;
constexpr int kHalfBytes = kChunk * 128;   // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kHalfBytes;  // one K or V chunk
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kQHalfBytes = 16 * 128;       // 16 (padded) head rows x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct TcArgs {
  const int32_t* sel;
  const int32_t* sel_count;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const __nv_bfloat16* q;
  const float* k_scales;  // e4m3 only
  const float* v_scales;
  float* ws_o;
  float* ws_lse;
  void* out;       // one split per pair: the final output and lse are written directly
  float* lse_out;
  unsigned* counters;  // split arrivals per pair (null: a separate merge kernel runs)
  int64_t num_pages;
  int hkv, hq, group, block, max_blocks, capacity, bps, splits, items;
  // balanced chunk ranges (stream_per > 0): the pairs' chunks (stream_n per
  // pair, a full selection) laid end to end and cut into one range of
  // stream_per chunks per CTA; an item is then a pair (items = pairs), its
  // part inside the CTA's range one segment, and splits the most segments a
  // pair can have (the partial workspace stride)
  int stream_per, stream_n;
  int out_f32;
  float scale_log2;
  uint64_t wait_ns;  // bound of every wait of the CTA's roles
};

template <int NH>
struct Layout {
  static constexpr int kPBytes = kChunk * 2 * NH * 2;
  // P buffers: two per softmax group where they fit (a group writes P of its
  // next chunk while the P.V product of its previous one may still read the
  // other), else one per group, and the group then waits for that product
  // before rewriting P
  static constexpr int kPBufs = NH <= 8 ? 4 : 2;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffP = kOffQ + 2 * kQHalfBytes;
  static constexpr int kOffX = kOffP + kPBufs * kPBytes;  // group hand-over: o[NH][128], m[NH], 2 words
  static constexpr int kOffBar = kOffX + ((NH * 128 + 2 * NH) * 4 + 15) / 16 * 16;
  static constexpr int kNumBars = 2 * kStages + 16;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffRed = kOffMisc + 16;
  static constexpr int kOffMeta = kOffRed + 2 * 3 * 4 * NH * 4;  // red: [group][3][4 warps][NH]; meta: [stage][8] (page, valid tokens)
  static constexpr int kOffProg = kOffMeta + kStages * 8 * 8;     // progress words of the roles (for a time-out record)
  static constexpr int kBytes = kOffProg + 32;
  // the layout plus 1 KB to align its base; what is left of the SM's shared
  // memory can hold a small CTA of another kernel (the overlapped page copy)
  static constexpr int kAlloc = (kBytes + 1024 + 127) / 128 * 128;
  static_assert(kAlloc <= 232448, "shared memory layout too large");
  static constexpr int kTmemCols = NH == 8 ? 64 : 128;
  static constexpr int kColO = 32;  // S uses columns [0, 32)
};

struct Item {
  int pair, split, b, kvh, s0, s1, nch, L, nb;
  int nseg;  // the pair's splits (segments): 1 = this item writes the output itself
};

// The work items of one CTA and where their selected blocks come from.  A
// persistent launch takes items first, first + stride, ... (below end) and
// resolves the global selection through the page table; a CTA of the fused
// scoring + selection + attention launch takes one item, whose (page, valid
// tokens) list rank 0 of its cluster has already resolved into this CTA's
// shared memory: list[i] is position s0 + i of the pair's selection,
// positions [s0, s1) are the item's, and L is the request's length.
struct Work {
  int first, stride;
  const int2* list;
  int s0, s1, L;
  int end;
  static constexpr bool kRanges = false;
};
// The same with balanced chunk ranges (a compile-time mode, so that each
// kernel carries the item geometry of one mode only).
struct RangeWork : Work {
  static constexpr bool kRanges = true;
};

// With balanced chunk ranges the CTA takes the pairs its range touches, in
// order; otherwise every gridDim.x-th item.
template <class W>
__device__ __forceinline__ W persistent_work(const TcArgs& a) {
  W w;
  w.list = nullptr;
  w.s0 = w.s1 = w.L = 0;
  if constexpr (W::kRanges) {  // (the chunk total stays below 2^30, so int holds every index)
    const int lo = static_cast<int>(blockIdx.x) * a.stream_per;
    const int hi = min(lo + a.stream_per, a.items * a.stream_n);
    w.first = lo / a.stream_n;
    w.stride = 1;
    w.end = hi > lo ? (hi - 1) / a.stream_n + 1 : w.first;
  } else {
    w.first = static_cast<int>(blockIdx.x);
    w.stride = static_cast<int>(gridDim.x);
    w.end = a.items;
  }
  return w;
}

template <class W>
__device__ __forceinline__ int item_pair(const TcArgs& a, int item) {
  if constexpr (W::kRanges) return item;
  return item / a.splits;
}

// Selected blocks per split of a pair with cnt selected blocks: its whole
// 128-token chunks spread evenly over the splits, at most bps.
__device__ __forceinline__ int split_len(int cnt, int bpc, int splits, int bps) {
  const int per = ((cnt + bpc - 1) / bpc + splits - 1) / splits * bpc;
  return min(per, bps);
}

// The two global reads an item's geometry depends on (its pair's selection
// count and request length), separate from the arithmetic on them, so that a
// loop can issue them an item ahead and use them an item later.
struct ItemPre {
  int cnt, L;
};
template <class W>
__device__ __forceinline__ ItemPre item_pre(const TcArgs& a, int item, const W& w) {
  if (w.list) return ItemPre{0, 0};
  const int pair = item_pair<W>(a, item);
  return ItemPre{a.sel_count[pair], a.seq_lens[pair / a.hkv]};
}

template <class W>
__device__ __forceinline__ Item item_geom_from(const TcArgs& a, int item, int bpc, const W& w, ItemPre pre) {
  Item it;
  it.pair = item_pair<W>(a, item);
  it.split = item - it.pair * a.splits;
  it.nseg = a.splits;
  it.b = it.pair / a.hkv;
  it.kvh = it.pair - it.b * a.hkv;
  if (w.list) {
    it.s0 = w.s0;
    it.s1 = w.s1;
    it.L = w.L;
  } else {
    int cnt = pre.cnt;
    cnt = max(0, min(cnt, a.capacity));
    if constexpr (W::kRanges) {
      // the part of the pair's chunks [base, base + stream_n) inside this
      // CTA's range; the pair's segments are the ranges it touches
      const int base = it.pair * a.stream_n;
      const int lo = static_cast<int>(blockIdx.x) * a.stream_per;
      const int c_lo = max(lo - base, 0);
      const int c_hi = min(lo + a.stream_per - base, a.stream_n);
      const int first_cta = base / a.stream_per;
      it.split = static_cast<int>(blockIdx.x) - first_cta;
      it.nseg = (base + a.stream_n - 1) / a.stream_per - first_cta + 1;
      it.s0 = min(cnt, c_lo * bpc);
      it.s1 = min(cnt, c_hi * bpc);
    } else {
      const int per = split_len(cnt, bpc, a.splits, a.bps);
      it.s0 = it.split * per;
      it.s1 = min(cnt, it.s0 + per);
    }
    it.L = pre.L;
  }
  const int nblk = it.s1 - it.s0;
  it.nch = nblk > 0 ? (nblk + bpc - 1) / bpc : 0;
  it.nb = min((max(it.L, 0) + a.block - 1) / a.block, a.max_blocks);
  return it;
}

template <class W>
__device__ __forceinline__ Item item_geom(const TcArgs& a, int item, int bpc, const W& w) {
  return item_geom_from(a, item, bpc, w, item_pre(a, item, w));
}


// A split's result: with one split per (request, kv head) it is the final
// output (written directly, no merge pass); otherwise it goes to the partial
// workspace for the log-sum-exp merge.
__device__ __forceinline__ void put_partial(const TcArgs& a, const Item& it, int h, int t, float o, float lse) {
  const int64_t orow = static_cast<int64_t>(it.b) * a.hq + static_cast<int64_t>(it.kvh) * a.group + h;
  if (it.nseg == 1) {
    if (a.out_f32)
      static_cast<float*>(a.out)[orow * kD + t] = o;
    else
      static_cast<__nv_bfloat16*>(a.out)[orow * kD + t] = __float2bfloat16_rn(o);
    if (a.lse_out && t == 0) a.lse_out[orow] = lse;
  } else {
    const int64_t row = orow * a.splits + it.split;
    a.ws_o[row * kD + t] = o;
    if (t == 0) a.ws_lse[row] = lse;
  }
}

// Split-K completion without a merge launch ("分块稀疏注意力与KV Cache量化"
// §2.2 log-sum-exp): once the 128 writer threads of an item have stored its
// partials (a CTA barrier), one thread counts the item in on its pair's
// counter with an acquire-release atomic, which publishes the CTA's partials
// and, for the split that arrives last, makes every other split's visible.
// That split merges them into the output and re-arms the counter.  No thread
// waits for another CTA.  Thread t merges 8 channels of head t / 16 (heads in
// rounds of 8), in the same order and arithmetic as the merge kernel.
// bar_id = the writers' named barrier; s_last = a shared-memory word.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void merge_if_last(const TcArgs& a, const Item& it, int t, int bar_id,
                                              volatile int* s_last) {
  named_barrier(bar_id, 128);  // every writer's partial stores are issued
  if (t == 0) *s_last = atom_add_acq_rel_gpu(a.counters + it.pair, 1u) == static_cast<unsigned>(it.nseg - 1);
  named_barrier(bar_id, 128);
  const bool last = *s_last != 0;
  named_barrier(bar_id, 128);  // s_last may be rewritten by the next item
  if (!last) return;
  const int g = a.group, S = it.nseg;
  const int c0 = (t & 15) * 8;
  for (int h0 = 0; h0 < g; h0 += 8) {
    const int h = h0 + (t >> 4);
    if (h >= g) continue;
    const int64_t orow = static_cast<int64_t>(it.b) * a.hq + static_cast<int64_t>(it.kvh) * g + h;
    const int64_t r0 = orow * a.splits;  // the pair's segments, stride splits
    float M = -INFINITY;
#pragma unroll 1
    for (int s = 0; s < S; ++s) M = fmaxf(M, __ldcg(a.ws_lse + r0 + s));
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    float lse = -INFINITY;
    if (M != -INFINITY) {
      float tot = 0.0f;
#pragma unroll 1
      for (int s = 0; s < S; ++s) {
        const float w = expf(__ldcg(a.ws_lse + r0 + s) - M);
        const float4* src = reinterpret_cast<const float4*>(a.ws_o + (r0 + s) * kD + c0);
        const float4 x0 = __ldcg(src), x1 = __ldcg(src + 1);
        const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        tot += w;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = w > 0.0f ? fmaf(w, x[i], acc[i]) : acc[i];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = acc[i] / tot;
      lse = M + logf(tot);
    }
    if (a.out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow * kD + c0);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      uint32_t w4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        w4[i] = *reinterpret_cast<const uint32_t*>(&v);
      }
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow * kD + c0) =
          make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    if (a.lse_out && (t & 15) == 0) a.lse_out[orow] = lse;
  }
  if (t == 0) a.counters[it.pair] = 0u;
}

// First item at or after `item` (stepping by w.stride) that has chunks; w.end or past if none.
template <class W>
__device__ __forceinline__ int find_item(const TcArgs& a, int bpc, int item, Item* it, const W& w) {
  for (; item < w.end; item += w.stride) {
    *it = item_geom(a, item, bpc, w);
    if (it->nch > 0) break;
  }
  return item;
}

// Lane's block of the group of 32 selected positions starting at `gbase`:
// (page, valid tokens), page -1 past the item or for a bad entry.  The
// selection entry is read without waiting for the item's count.
__device__ __forceinline__ int2 resolve_group(const TcArgs& a, const Item& it, int gbase, unsigned* bad,
                                              const Work& w) {
  const int lane = threadIdx.x & 31;
  if (w.list) return it.s0 + gbase + lane < it.s1 ? w.list[gbase + lane] : make_int2(-1, 0);
  const int pos = it.s0 + gbase + lane;
  const int64_t row = static_cast<int64_t>(it.pair) * a.capacity;
  const int j = pos < a.capacity ? a.sel[row + pos] : -1;
  if (pos >= it.s1) return make_int2(-1, 0);
  if (j < 0 || j >= it.nb) {
    *bad |= HS_EBIT_BLOCK_RANGE;
    return make_int2(-1, 0);
  }
  const int page = a.page_table[static_cast<int64_t>(it.pair) * a.max_blocks + j];
  if (page < 0 || page >= a.num_pages) {
    *bad |= HS_EBIT_PAGE_RANGE;
    return make_int2(-1, 0);
  }
  return make_int2(page, min(a.block, it.L - j * a.block));
}

// TMA producer warp (all 32 lanes).  An item's selected blocks are resolved 32
// at a time (lane i: block i of the group) and the next group - of this item or
// of the next one - is looked up while the current group's chunks are issued,
// so page-table lookups stay off the copy stream.  Each chunk's pages and
// valid-token counts are published in meta[stage][8] for the softmax warps and
// every lane issues the copies of its own block.
// prog[0] / prog[5]: chunks issued so far / the item being issued.
template <int STAGES, class W, typename IssueFn>
__device__ __forceinline__ void run_producer(const TcArgs& a, const W& w, int bpc, uint32_t full0, uint32_t empty0,
                                             int2* meta, uint32_t bytes_per_block, volatile int* abort_flag,
                                             unsigned* err, volatile int* prog, IssueFn issue) {
  const int lane = threadIdx.x & 31;
  unsigned bad = 0;
  Item it;
  int item = find_item(a, bpc, w.first, &it, w);
  int2 cur = item < w.end ? resolve_group(a, it, 0, &bad, w) : make_int2(-1, 0);
  int c = 0;
  bool stop = false;
  while (item < w.end && !stop) {
    const int nblk = it.s1 - it.s0;
    const int ngroups = (nblk + 31) / 32;
    int next_item = item;
    Item nit = it;
    for (int g = 0; g < ngroups && !stop; ++g) {
      // the next group (of this item, or the first of the next item) is
      // looked up once this group's first chunks fill the ring, so that its
      // dependent loads overlap the copies in flight instead of delaying them
      int2 nxt = make_int2(-1, 0);
      bool looked = false;
      auto look_ahead = [&]() {
        if (g + 1 < ngroups) {
          nxt = resolve_group(a, it, (g + 1) * 32, &bad, w);
        } else {
          next_item = find_item(a, bpc, item + w.stride, &nit, w);
          if (next_item < w.end) nxt = resolve_group(a, nit, 0, &bad, w);
        }
        looked = true;
      };
      const int gchunks = min(32 / bpc, (nblk - g * 32 + bpc - 1) / bpc);
      const int look_at = min(gchunks, STAGES) - 1;
      for (int k = 0; k < gchunks; ++k, ++c) {
        int go = 0;
        if (lane == 0)
          go = !*abort_flag &&
               (c < STAGES || mbar_wait(empty0 + 8 * (c % STAGES), ((c / STAGES) + 1) & 1, abort_flag, a.wait_ns));
        if (!__shfl_sync(0xffffffffu, go, 0)) {
          stop = true;
          break;
        }
        const int s = c % STAGES;
        const int bi = lane - k * bpc;
        const bool mine = bi >= 0 && bi < bpc;
        if (mine) meta[s * 8 + bi] = cur;
        const uint32_t tx = __reduce_add_sync(0xffffffffu, (mine && cur.x >= 0) ? bytes_per_block : 0u);
        __syncwarp();
        if (lane == 0) mbar_arrive_tx(full0 + 8 * s, tx);
        __syncwarp();
        if (mine && cur.x >= 0) issue(s, bi, cur.x);
        if (lane == 0) {
          prog[0] = c + 1;
          prog[5] = item;
        }
        if (k == look_at) look_ahead();
      }
      if (!looked && !stop) look_ahead();  // a group shorter than the ring
      cur = nxt;
    }
    item = next_item;
    it = nit;
  }
  bad = __reduce_or_sync(0xffffffffu, bad);
  if (lane == 0) {
    if (bad) set_error(err, bad);
    // let every copy this CTA issued land before the CTA can exit
    for (int s = 0; s < STAGES && s < c; ++s) {
      const int last = c - 1 - ((c - 1 - s) % STAGES);
      mbar_drain(full0 + 8 * s, (last / STAGES) & 1);
    }
  }
}

// bf16 kernel: warps 0-7 are two softmax groups of 4 warps (group g takes the
// chunks c with c % 2 == g, so two chunks are in the softmax stage at once),
// warp 8 is the TMA producer, warp 9 issues S = K.Q^T, warps 10 and 11 issue
// O = V^T.P of the even and the odd chunks.
constexpr int kThreadsB = 384;
constexpr int kProdB = 8, kMma1B = 9, kMma2B = 10, kMma3B = 11;

// Lazy running max of the online softmax: a chunk moves a head's running max
// m only when one of its logits (log2 units) exceeds m by more than this;
// otherwise its probabilities 2^(x - m) stay <= 2^kLazyMax (within the range
// of the bf16 / f16 P parts) and nothing is rescaled.  The result is the same
// softmax: the offset cancels in the normalisation.
constexpr float kLazyMax = 8.0f;

// float -> unsigned key with the same order (-0 below +0; no NaN here), and back
__device__ __forceinline__ uint32_t float_order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// per-warp max (or sum) of each of the NH values a lane holds, over the warp's
// 32 lanes, by halving exchanges: afterwards lane l holds the result of value
// l / (32 / NH) (NH <= 32)
template <int NH, bool MAX>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[NH]) {
  const int lane = threadIdx.x & 31;
  int cur = NH;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    if (cur > 1) {
      const bool upper = (lane & o) != 0;
      const int half = cur / 2;
#pragma unroll
      for (int i = 0; i < NH / 2; ++i) {
        if (i < half) {
          const float send = upper ? v[i] : v[i + half];
          const float keep = upper ? v[i + half] : v[i];
          const float got = __shfl_xor_sync(0xffffffffu, send, o);
          v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
      }
      cur = half;
    } else {
      const float got = __shfl_xor_sync(0xffffffffu, v[0], o);
      v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
    }
  }
  return v[0];
}

// Barrier of P buffer b (the bf16 kernel has up to four P buffers; the first
// two barriers keep their original slots).  One barrier per buffer: a buffer
// is written again only after the product that read it has completed, so its
// barrier is never two phases ahead of the MMA thread that waits on it (a
// parity wait cannot tell phase n from phase n + 2).
__host__ __device__ constexpr int p_full_index(int b) { return b < 2 ? 2 * kStages + 4 + b : 2 * kStages + 9 + b; }

// Barrier initialisation (thread 0) and TMEM allocation (warp kMma1B) of a
// bf16 attention CTA; the caller synchronises the CTA before any role starts.
template <int NH>
__device__ __forceinline__ void attn_bf16_setup(uint8_t* smem) {
  using Ly = Layout<NH>;
  const uint32_t bar0 = smem_u32(smem) + Ly::kOffBar;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar0 + 8 * s, 1);              // full
      mbar_init(bar0 + 8 * (kStages + s), 1);  // empty
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar0 + 8 * (2 * kStages + b), 1);      // s_full
      mbar_init(bar0 + 8 * (2 * kStages + 2 + b), 128);  // s_free
      mbar_init(bar0 + 8 * (2 * kStages + 6 + b), 1);    // o_full
      mbar_init(bar0 + 8 * (2 * kStages + 8 + b), 128);  // o_free
    }
    for (int b = 0; b < 4; ++b) mbar_init(bar0 + 8 * p_full_index(b), 128);  // p_full, one per P buffer
    mbar_init(bar0 + 8 * (2 * kStages + 10), 128);  // q_full
    mbar_init(bar0 + 8 * (2 * kStages + 13), 1);    // q_free
    mbar_init(bar0 + 8 * (2 * kStages + 14), 128);  // x_full
    mbar_init(bar0 + 8 * (2 * kStages + 15), 128);  // x_free
    *reinterpret_cast<volatile int*>(smem + Ly::kOffMisc + 4) = 0;   // abort flag
    *reinterpret_cast<volatile int*>(smem + Ly::kOffMisc + 12) = 0;  // which wait ran out
    for (int i = 0; i < 8; ++i) reinterpret_cast<volatile int*>(smem + Ly::kOffProg)[i] = 0;
    fence_barrier_init();
  }
  if (warp == kMma1B) {
    tmem_alloc(smem_u32(smem + Ly::kOffMisc), Ly::kTmemCols);
    tmem_relinquish();
  }
}

struct NoEmit {};

// The whole life of one bf16 attention CTA over the items of w: set-up
// (unless SETUP is false: the caller ran attn_bf16_setup, synchronised the
// CTA and waited for its predecessor), roles, tear-down.  An item's result
// goes to the output (one split) or the partial workspace, or, with an Emit
// other than NoEmit, to emit(h, channel, o, lse) for the caller's merge.  Run
// by all kThreadsB threads.
template <int NH, bool SETUP = true, class Emit = NoEmit, class W = Work>
__device__ __forceinline__ void attn_bf16_cta(const CUtensorMap* tm_k_, const CUtensorMap* tm_v_, const TcArgs& a,
                                              const W& w, unsigned* err, const Emit& emit = Emit{}) {
  constexpr bool PART_SMEM = !std::is_same<Emit, NoEmit>::value;
  using Ly = Layout<NH>;
  const CUtensorMap& tm_k = *tm_k_;
  const CUtensorMap& tm_v = *tm_v_;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Ly::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (kStages + s); };
  auto s_full = [&](int b) { return bar0 + 8 * (2 * kStages + b); };
  auto s_free = [&](int b) { return bar0 + 8 * (2 * kStages + 2 + b); };
  auto p_full = [&](int b) { return bar0 + 8 * p_full_index(b); };  // b = P buffer
  auto o_full = [&](int b) { return bar0 + 8 * (2 * kStages + 6 + b); };
  auto o_free = [&](int b) { return bar0 + 8 * (2 * kStages + 8 + b); };
  const uint32_t q_full = bar0 + 8 * (2 * kStages + 10);
  // q_free: every S product of an item is complete (the Q operand may be
  // rewritten); x_full / x_free: an item's state handed from one softmax
  // group to the other / read by it
  const uint32_t q_free = bar0 + 8 * (2 * kStages + 13);
  const uint32_t x_full = bar0 + 8 * (2 * kStages + 14);
  const uint32_t x_free = bar0 + 8 * (2 * kStages + 15);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kOffMisc + 4);
  // progress of the roles, copied into the record of a wait that runs out:
  // [0] chunks issued by the producer, [1] / [2] chunks issued by the S / O
  // MMA thread, [3] / [4] chunks done by softmax group 0 / 1, [5] the
  // producer's item, [6] the softmax groups' item, [7] its chunk count
  volatile int* prog = reinterpret_cast<volatile int*>(smem + Ly::kOffProg);
  auto k_half = [&](int s, int h) { return sbase + s * kStageBytes + h * kHalfBytes; };
  auto v_half = [&](int s, int h) { return sbase + s * kStageBytes + kTileBytes + h * kHalfBytes; };
  auto q_half = [&](int h) { return sbase + Ly::kOffQ + h * kQHalfBytes; };
  auto p_buf = [&](int b) { return sbase + Ly::kOffP + b * Ly::kPBytes; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.block;
  const int bpc = kChunk / B;

  if constexpr (SETUP) {
    pdl_trigger();
    // ---- set-up: barriers, TMEM, tensor maps (overlaps the previous kernel) ----
    if (warp == kProdB && lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    attn_bf16_setup<NH>(smem);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();  // the selection and q of this step are complete from here on
  }
  const uint32_t tmem = *tmem_slot;

  int2* meta = reinterpret_cast<int2*>(smem + Ly::kOffMeta);
  if (warp == kProdB) {
    // ================= TMA producer =================
    run_producer<kStages>(a, w, bpc, full_bar(0), empty_bar(0), meta, 4u * B * 128u, abort_flag, err, prog,
                          [&](int s, int bi, int page) {
                            const uint32_t row_off = bi * B * 128;
                            const int y = page * B;
                            tma_load_2d(k_half(s, 0) + row_off, &tm_k, 0, y, full_bar(s));
                            tma_load_2d(k_half(s, 1) + row_off, &tm_k, 64, y, full_bar(s));
                            tma_load_2d(v_half(s, 0) + row_off, &tm_v, 0, y, full_bar(s));
                            tma_load_2d(v_half(s, 1) + row_off, &tm_v, 64, y, full_bar(s));
                          });
  } else if (warp == kMma1B || warp == kMma2B || warp == kMma3B) {
    // ================= MMA issuers: one thread for S = K.Q^T, two for O = V^T.P =================
    // (an MMA takes its issuing thread ~70 cycles, a GEMM's eight a few hundred
    // ns, so S and O are issued from different threads, and the O products of
    // the two softmax groups' chunks from one thread each)
    if (lane == 0) {
      const bool first = warp == kMma1B;
      const int par = warp == kMma2B ? 0 : 1;  // an O issuer's chunk parity
      constexpr uint32_t idesc1 = idesc_bf16(128, 16, false, false);
      constexpr uint32_t idesc2 = idesc_bf16(128, 2 * NH, true, true);
      constexpr uint32_t kPLbo = 8 * 2 * NH * 2;  // bytes between 8-token groups of P
      const uint64_t kdesc = smem_desc(k_half(0, 0), 16, 1024, 2);
      const uint64_t qdesc = smem_desc(q_half(0), 16, 1024, 2);
      const uint64_t vdesc = smem_desc(v_half(0, 0), kHalfBytes, 1024, 2);
      const uint64_t pdesc = smem_desc(p_buf(0), kPLbo, 128, 0);
      int c = 0, qi = 0, qc = 0;
      int item = w.first;
      Item it = item < w.end ? item_geom(a, item, bpc, w) : Item{};
      bool ok = true;
      while (ok && item < w.end && !*abort_flag) {
        const int next = item + w.stride;
        const Item nit = next < w.end ? item_geom(a, next, bpc, w) : Item{};  // in flight meanwhile
        if (it.nch > 0 && first) {
          ok = mbar_wait(q_full, qi & 1, abort_flag, a.wait_ns);
          ++qi;
        }
        for (int ci = 0; ok && ci < it.nch; ++ci, ++c) {
          const int st = c % kStages, bb = c & 1;
          if (first) {
            ok = mbar_wait(full_bar(st), (c / kStages) & 1, abort_flag, a.wait_ns) &&
                 (c < 2 || mbar_wait(s_free(bb), ((c >> 1) + 1) & 1, abort_flag, a.wait_ns));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < kD / 16; ++k) {
              const uint32_t koff = st * kStageBytes + (k >> 2) * kHalfBytes + (k & 3) * 32;
              const uint32_t qoff = (k >> 2) * kQHalfBytes + (k & 3) * 32;
              mma_f16(tmem + bb * 16, kdesc + (koff >> 4), qdesc + (qoff >> 4), idesc1, k > 0 ? 1u : 0u);
            }
            mma_commit(s_full(bb));
            prog[1] = c + 1;
            if (ci == it.nch - 1) {
              mma_commit(q_free);  // the item's last S product: its Q operand is free
              ++qc;
            }
          } else {
            if (bb != par) continue;
            ok = mbar_wait(p_full(c % Ly::kPBufs), (c / Ly::kPBufs) & 1, abort_flag, a.wait_ns) &&
                 (c < 2 || mbar_wait(o_free(bb), ((c >> 1) + 1) & 1, abort_flag, a.wait_ns));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < kChunk / 16; ++k) {
              const uint32_t voff = st * kStageBytes + k * 2048;
              const uint32_t poff = (c % Ly::kPBufs) * Ly::kPBytes + k * 2 * kPLbo;
              mma_f16(tmem + Ly::kColO + bb * 2 * NH, vdesc + (voff >> 4), pdesc + (poff >> 4), idesc2,
                      k > 0 ? 1u : 0u);
            }
            mma_commit(o_full(bb));
            mma_commit(empty_bar(st));
            prog[2] = c + 1;
          }
        }
        item = next;
        it = nit;
      }
      // every product this thread issued is complete before TMEM is released
      // (a commit arrives once all of the thread's earlier MMAs are done)
      if (first && c > 0) mbar_drain(s_full((c - 1) & 1), ((c - 1) >> 1) & 1);
      if (first && qc > 0) mbar_drain(q_free, (qc - 1) & 1);
      if (!first) {
        const int last = ((c - 1) & 1) == par ? c - 1 : c - 2;  // this issuer's last chunk
        if (last >= 0) mbar_drain(empty_bar(last % kStages), (last / kStages) & 1);
      }
    }
  } else if (warp < 8) {
    // ================= softmax / correction: two groups of 4 warps =================
    const int grp = warp >> 2;       // group: owns the chunks with c % 2 == grp, S/P/O buffer grp
    const int wq = warp & 3;         // TMEM lane quarter
    const int t = tid & 127;         // token row of S, channel of O
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const int bar = 1 + grp;         // named barrier of the group
    const int g = a.group;
    float* red = reinterpret_cast<float*>(smem + Ly::kOffRed) + grp * 12 * NH;  // [3][4 warps][NH]
    float* rs = red + 8 * NH;                                                  // this group's normaliser parts
    const float* rs_other = reinterpret_cast<const float*>(smem + Ly::kOffRed) + (1 - grp) * 12 * NH + 8 * NH;
    // hand-over of an item's state between the groups: o[NH][128], m[NH],
    // then one last-split word per group
    float* xo = reinterpret_cast<float*>(smem + Ly::kOffX);
    float* xm = xo + NH * 128;
    volatile int* my_last = reinterpret_cast<volatile int*>(xm + NH) + grp;
    auto load_q = [&](int item, uint4 (&v)[2]) {
      const int pair = item_pair<W>(a, item), b = pair / a.hkv, kvh = pair - b * a.hkv;
      const int n = t >> 3, ch = t & 7;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        v[h] = make_uint4(0, 0, 0, 0);
        if (n < g)
          v[h] = *reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(b) * a.hq + kvh * g + n) * kD + h * 64 +
                                                 ch * 8);
      }
    };
    // Q operand: 16 rows (heads, zero past g) x 128 channels, 128-byte swizzle
    auto write_q = [&](const uint4 (&v)[2]) {
      const int n = t >> 3, ch = t & 7;
#pragma unroll
      for (int h = 0; h < 2; ++h)
        *reinterpret_cast<uint4*>(smem + Ly::kOffQ + h * kQHalfBytes + n * 128 + ((ch ^ (n & 7)) << 4)) = v[h];
      fence_async_smem();
      mbar_arrive(q_full);
    };
    // An item ends with a hand-over instead of a CTA-wide barrier: the group
    // that takes the next item's first chunk (the starter) writes that item's
    // query once every S product of this one is complete (q_free), publishes
    // its state (o, m and its normaliser parts) and goes on; the other group
    // combines both states and writes the result meanwhile.  Waits across the
    // groups are bounded mbarrier waits; inside a group, every wait's outcome
    // is made uniform (warp vote, then bar.red.or at the group's named
    // barriers) so that the group's threads leave their loops together.
    int c = 0;
    int e = 0;  // items with chunks so far: the phase of q_free, x_full and x_free
    int item = w.first;
    Item it{};
    uint4 qv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (item < w.end) {
      it = item_geom(a, item, bpc, w);
      if (grp == 0) load_q(item, qv);  // the first item starts with chunk 0, group 0's
    }
    bool q_ready = false;  // this item's query was written at the end of the previous one
    bool fail = false;     // this thread saw a wait run out (uniform per warp)
    while (item < w.end) {
      // the next item's geometry reads and query rows are issued while this one runs
      const int next = item + w.stride;
      const int c0 = c;
      const bool starter = grp == ((c0 + it.nch) & 1);
      ItemPre npre{0, 0};
      uint4 nqv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
      if (next < w.end) {
        npre = item_pre(a, next, w);
        if (starter) load_q(next, nqv);
      }
      if (tid == 0) {
        prog[6] = item;
        prog[7] = it.nch;
      }
      Item nit{};  // the next item, computed once this item's chunks are done
      bool q_next = false;
      if (it.nch > 0) {
        if (grp == (c0 & 1) && !q_ready) {
          if (e == 0 || __all_sync(0xffffffffu, mbar_wait(q_free, (e - 1) & 1, abort_flag, a.wait_ns)))
            write_q(qv);
          else
            fail = true;
        }
        float m[NH], lsum[NH], oacc[NH], alpha_prev[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          m[h] = -INFINITY;
          lsum[h] = 0.0f;
          oacc[h] = 0.0f;
          alpha_prev[h] = 1.0f;
        }
        // O of an own chunk once its P.V product is complete; false (for the
        // whole warp) when the wait ran out
        auto take_o = [&](int cc) -> bool {
          if (!__all_sync(0xffffffffu, mbar_wait(o_full(grp), (cc >> 1) & 1, abort_flag, a.wait_ns))) return false;
          tc_fence_after();
          float ov[2 * NH];
          if constexpr (NH == 8) {
            tmem_ld16(tmem + lane_base + Ly::kColO + grp * 16, *reinterpret_cast<float(*)[16]>(ov));
          } else {
            tmem_ld16(tmem + lane_base + Ly::kColO + grp * 32, *reinterpret_cast<float(*)[16]>(ov));
            tmem_ld16(tmem + lane_base + Ly::kColO + grp * 32 + 16, *reinterpret_cast<float(*)[16]>(ov + 16));
          }
          tc_fence_before();
          mbar_arrive(o_free(grp));
#pragma unroll
          for (int h = 0; h < NH; ++h) oacc[h] = fmaf(oacc[h], alpha_prev[h], ov[h] + ov[NH + h]);
          return true;
        };
        int last_own = -1;
        for (int cc = c0 + ((grp - c0) & 1); cc < c0 + it.nch; cc += 2) {
          const int s = cc % kStages;
          const int bi = t / B, tok = t - bi * B;
          bool ready = !fail && mbar_wait(full_bar(s), (cc / kStages) & 1, abort_flag, a.wait_ns);
          const int2 md = ready ? meta[s * 8 + bi] : make_int2(-1, 0);
          const bool valid = md.x >= 0 && tok < md.y;
          ready = __all_sync(0xffffffffu, ready && mbar_wait(s_full(grp), (cc >> 1) & 1, abort_flag, a.wait_ns));
          float sv[16];
          if (ready) {
            tc_fence_after();
            tmem_ld16(tmem + lane_base + grp * 16, sv);
            tc_fence_before();
            mbar_arrive(s_free(grp));
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) sv[i] = 0.0f;
          }
          float x[NH], r[NH];
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            x[h] = (valid && h < g) ? sv[h] * a.scale_log2 : -INFINITY;
            r[h] = x[h];
          }
          // the group's running max moves only when some row exceeds it by
          // more than kLazyMax (one vote)
          bool over = false;
#pragma unroll
          for (int h = 0; h < NH; ++h) over |= x[h] > m[h] + kLazyMax;
          float alpha[NH], p[NH];
          if (named_barrier_or(bar, 128, over || fail || !ready)) {
            // chunk max per head over the 128 rows: warp reduce-scatter, then the 4 warps
            float* rb = red + ((cc >> 1) & 1) * 4 * NH;  // alternate buffers: a barrier per chunk at least
            const float wmax = warp_reduce_scatter<NH, true>(r);
            if ((lane % (32 / NH)) == 0) rb[wq * NH + lane / (32 / NH)] = wmax;
            if (named_barrier_or(bar, 128, fail || !ready)) {
              fail = true;
              break;
            }
#pragma unroll
            for (int h = 0; h < NH; ++h) {
              const float cm = fmaxf(fmaxf(rb[h], rb[NH + h]), fmaxf(rb[2 * NH + h], rb[3 * NH + h]));
              const float mn = fmaxf(m[h], cm);
              alpha[h] = (mn == -INFINITY) ? 1.0f : exp2f(m[h] - mn);
              m[h] = mn;
              p[h] = x[h] == -INFINITY ? 0.0f : exp2f(x[h] - mn);
              lsum[h] = fmaf(lsum[h], alpha[h], p[h]);
            }
          } else {
#pragma unroll
            for (int h = 0; h < NH; ++h) {
              alpha[h] = 1.0f;
              p[h] = x[h] == -INFINITY ? 0.0f : exp2f(x[h] - m[h]);
              lsum[h] += p[h];
            }
          }
          // with one P buffer per group, the P.V product of this group's
          // previous chunk reads it: that product must be complete (and its O
          // taken) before P is rewritten
          if (Ly::kPBufs == 2 && last_own >= 0 && !take_o(last_own)) fail = true;
          if (!fail) {
            // probabilities, split into bf16 high part + bf16 remainder
            uint32_t hi2[NH / 2], lo2[NH / 2];
#pragma unroll
            for (int h = 0; h < NH; h += 2) {
              const __nv_bfloat162 hi = __floats2bfloat162_rn(p[h], p[h + 1]);
              const float2 hf = __bfloat1622float2(hi);
              const __nv_bfloat162 lo = __floats2bfloat162_rn(p[h] - hf.x, p[h + 1] - hf.y);
              hi2[h / 2] = *reinterpret_cast<const uint32_t*>(&hi);
              lo2[h / 2] = *reinterpret_cast<const uint32_t*>(&lo);
            }
            {
              constexpr int kPLbo = 8 * 2 * NH * 2;
              uint8_t* prow = smem + Ly::kOffP + (cc % Ly::kPBufs) * Ly::kPBytes + (t >> 3) * kPLbo + (t & 7) * 16;
#pragma unroll
              for (int gi = 0; gi < NH / 8; ++gi) {
                *reinterpret_cast<uint4*>(prow + gi * 128) =
                    make_uint4(hi2[gi * 4], hi2[gi * 4 + 1], hi2[gi * 4 + 2], hi2[gi * 4 + 3]);
                *reinterpret_cast<uint4*>(prow + (NH / 8 + gi) * 128) =
                    make_uint4(lo2[gi * 4], lo2[gi * 4 + 1], lo2[gi * 4 + 2], lo2[gi * 4 + 3]);
              }
            }
            if (!valid) {
              // rows of no token (past the request's end inside its last page, or of
              // no loaded block): zero V so they contribute exactly nothing - P is 0
              // there but the bytes in shared memory need not be finite
              uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint4* row = reinterpret_cast<uint4*>(smem + s * kStageBytes + kTileBytes + h * kHalfBytes + t * 128);
#pragma unroll
                for (int i = 0; i < 8; ++i) row[i] = z;
              }
            }
            fence_async_smem();
            mbar_arrive(p_full(cc % Ly::kPBufs));
            if (t == 0) prog[3 + grp] = cc + 1;
            // two P buffers per group: the product two own chunks back is done
            // before its buffer is written again (next own chunk)
            if (Ly::kPBufs == 4 && last_own >= 0 && !take_o(last_own)) fail = true;
          }
#pragma unroll
          for (int h = 0; h < NH; ++h) alpha_prev[h] = alpha[h];
          last_own = cc;
        }
        c = c0 + it.nch;
        if (next < w.end) nit = item_geom_from(a, next, bpc, w, npre);
        // the normaliser parts (one per warp and head)
        float wsum;
        {
          float r[NH];
#pragma unroll
          for (int h = 0; h < NH; ++h) r[h] = lsum[h];
          wsum = warp_reduce_scatter<NH, false>(r);
        }
        // (the hand-over buffers - xo, xm and both groups' normaliser
        // parts - are free once the previous item's combination has read them)
        if (starter) {
          // the next item's query first, once this item's S products are
          // complete, so that its first products overlap the rest
          q_next = next < w.end && nit.nch > 0;
          if (q_next) {
            if (!fail && __all_sync(0xffffffffu, mbar_wait(q_free, e & 1, abort_flag, a.wait_ns)))
              write_q(nqv);
            else
              fail = true;
          }
          // then publish and go on (a warp whose wait ran out leaves at the
          // group's next named barrier, with the others)
          if (!fail && last_own >= 0 && !take_o(last_own)) fail = true;
          if (!fail && e > 0 && !__all_sync(0xffffffffu, mbar_wait(x_free, (e - 1) & 1, abort_flag, a.wait_ns)))
            fail = true;
          if (!fail) {
            if ((lane % (32 / NH)) == 0) rs[wq * NH + lane / (32 / NH)] = wsum;
#pragma unroll
            for (int h = 0; h < NH; ++h) xo[h * 128 + t] = oacc[h];
#pragma unroll
            for (int h = 0; h < NH; ++h)  // compile-time indices keep m[] in registers
              if (t == h) xm[h] = m[h];
            mbar_arrive(x_full);
          }
        } else {
          if (!fail && last_own >= 0 && !take_o(last_own)) fail = true;
          if (!fail && e > 0 && !__all_sync(0xffffffffu, mbar_wait(x_free, (e - 1) & 1, abort_flag, a.wait_ns)))
            fail = true;
          if (!fail && (lane % (32 / NH)) == 0) rs[wq * NH + lane / (32 / NH)] = wsum;
          // x_full: the other group's state is in; the barrier also orders
          // this group's normaliser parts
          fail = named_barrier_or(bar, 128, fail || !mbar_wait(x_full, e & 1, abort_flag, a.wait_ns));
          if (fail) break;
          // per head, once (thread h): the weights of the two states, 1 / l
          // and the lse, into this group's chunk-max buffer (no thread of the
          // group writes it again before the group's next vote barrier, which
          // every thread reaches only after the output below)
          float* fac = red;  // [NH][4]
          {
            const int h = t;
            float m0 = -INFINITY;
#pragma unroll
            for (int i = 0; i < NH; ++i) m0 = (i == h) ? m[i] : m0;  // compile-time indices keep m[] in registers
            if (h < g && h < NH) {
              const float l0 = rs[h] + rs[NH + h] + rs[2 * NH + h] + rs[3 * NH + h];
              const float m1 = xm[h];
              const float l1 = rs_other[h] + rs_other[NH + h] + rs_other[2 * NH + h] + rs_other[3 * NH + h];
              const float mx = fmaxf(m0, m1);
              const float e0 = m0 == -INFINITY ? 0.0f : exp2f(m0 - mx);
              const float e1 = m1 == -INFINITY ? 0.0f : exp2f(m1 - mx);
              const float lt = l0 * e0 + l1 * e1;
              const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
              fac[4 * h] = e0 * inv;
              fac[4 * h + 1] = e1 * inv;
              fac[4 * h + 3] = lt > 0.0f ? (mx + log2f(lt)) * kLn2 : -INFINITY;
            }
          }
          fail = named_barrier_or(bar, 128, fail);
          if (fail) break;
          // per channel two products; one copy of the code for all heads
          // (head h's accumulator picked out of oacc[] with compile-time indices)
#pragma unroll 1
          for (int h = 0; h < g && h < NH; ++h) {
            float oh = oacc[0];
#pragma unroll
            for (int i = 1; i < NH; ++i) oh = (i == h) ? oacc[i] : oh;
            const float o = fmaf(oh, fac[4 * h], xo[h * 128 + t] * fac[4 * h + 1]);
            const float lse = fac[4 * h + 3];
            if constexpr (PART_SMEM) {
              emit(h, t, o, lse);
            } else {
              put_partial(a, it, h, t, o, lse);
            }
          }
          mbar_arrive(x_free);
          if (!PART_SMEM && it.nseg > 1 && a.counters) merge_if_last(a, it, t, bar, my_last);
        }
        ++e;
      } else if (grp == 0) {
        if constexpr (PART_SMEM) {
          for (int h = 0; h < g; ++h) emit(h, t, 0.0f, -INFINITY);
        } else {
          for (int h = 0; h < g; ++h) put_partial(a, it, h, t, 0.0f, -INFINITY);
          if (it.nseg > 1 && a.counters) merge_if_last(a, it, t, bar, my_last);
        }
      }
      item = next;
      it = (it.nch > 0 || next >= w.end) ? nit : item_geom_from(a, next, bpc, w, npre);
      q_ready = q_next;
      qv[0] = nqv[0];
      qv[1] = nqv[1];
    }
  }

  // ---- tear-down ----
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0)
    report_timeout(err, PART_SMEM ? kTimeoutStepFused : kTimeoutAttnBf16, static_cast<unsigned>(abort_flag[2]), prog);
  if (warp == kMma1B) {
    tc_fence_after();
    tmem_dealloc(tmem, Ly::kTmemCols);
  }
}

template <int NH, class W>
__global__ void __launch_bounds__(kThreadsB, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   TcArgs a, unsigned* err) {
  attn_bf16_cta<NH, true, NoEmit, W>(&tm_k, &tm_v, a, persistent_work<W>(a), err);
}


// ============================================================================
// Bound scoring + selection + attention of one decode step in one launch
// ("KV 稀疏化" wiki §5 Quest and §2 sink/window, then the attention above),
// bf16 K/V and summaries, head_dim 128, g <= 8, when every (request, kv head)
// fits one wave: one cluster of F CTAs per (request, kv head), F = max(tiles
// of 128 blocks, attention splits) <= 8.
//   phase 1  CTA r scores tile r of the pair (TMA of its summary rows, 16
//            MMAs, max over the group) and stores the scores (and the range
//            of their keys) into the shared memory of every CTA of the
//            cluster, and into scores_opt; meanwhile every CTA stages the
//            pair's page-table row (and score history), and rank 0 asks L2
//            for the K/V pages of the forced blocks.
//   phase 2  after one cluster barrier every CTA smooths and selects on its
//            own copy - the same selection as the selection kernels; rank 0
//            stores it (and the history) - and resolves the blocks of its
//            own split, whole 128-token chunks spread evenly over the splits,
//            to (page, valid tokens).
//   phase 3  CTA r is the attention CTA of split r (a one-item Work); each
//            head's result is pushed into the push buffer (kOffPush, used by
//            nothing else) of the CTA of the cluster that merges that head.
//   phase 4  after a second cluster barrier, which orders those pushes and
//            keeps every CTA resident until they have landed, each CTA
//            merges its heads from its own push buffer.
// Nothing waits on another cluster.  Between the two cluster barriers a CTA
// touches another's shared memory only through the phase-3 pushes.
constexpr int kFuseMaxCluster = 8;
constexpr int kFuseList = 256;   // selected blocks of one split held in shared memory
constexpr int kPushSlots = 13;   // (split, head) results one CTA merges
constexpr int kFuseMaxBlocks = kFuseMaxCluster * bound::kTile;
// scratch of phases 1-2 inside the K/V ring, which is unused until phase 3
constexpr int kFTile = 0;                                       // summary tile
constexpr int kFQ = kFTile + bound::kTileBytes;                 // [Q+ | Q-]
constexpr int kFScores = kFQ + bound::kQBytes;                  // the pair's scores
constexpr int kFPrev = kFScores + kFuseMaxBlocks * 4;           // the pair's score history
constexpr int kFHist = kFPrev + kFuseMaxBlocks * 4;             // radix histograms
constexpr int kFWarp = kFHist + 3 * sel::kHistWords * 4;        // per-warp counts
constexpr int kFRange = kFWarp + 128;                           // key range per scoring warp
constexpr int kFPt = kFRange + 2 * 4 * kFuseMaxCluster * 4;     // the pair's page-table row
constexpr int kFSel = kFPt + kFuseMaxBlocks * 4;                // the selection
static_assert(kFSel + kFuseMaxBlocks * 4 <= kStages * kStageBytes, "scratch exceeds the ring");

template <int NH>
struct FuseLayout {
  static constexpr int kOffF = (Layout<NH>::kBytes + 15) / 16 * 16;
  static constexpr int kOffBar = kOffF;       // tile full, q full, accumulator full
  static constexpr int kOffList = kOffF + 48;  // int2[kFuseList]: (page, valid tokens) of this CTA's split
  static constexpr int kOffPush = kOffList + kFuseList * 8;  // [kPushSlots][128] o, then [kPushSlots] lse
  static constexpr int kBytes = kOffPush + (kPushSlots * 129 * 4 + 15) / 16 * 16;
  static constexpr int kAlloc = (kBytes + 1024 + 127) / 128 * 128;
  static_assert(kAlloc <= 232448, "fused shared memory layout too large");
};

struct FuseArgs {
  float* scores;  // nullable: the bound scores also go to global memory
  const uint8_t* k_pages;  // for the L2 prefetch of the forced blocks
  const uint8_t* v_pages;
  int tiles;    // 128-block tiles per (request, kv head)
  int cluster;  // CTAs per (request, kv head)
  int early;    // the summary tile may be copied before the previous kernel completes
  // reuse: no scoring and no selection; the step attends over the selection
  // given in sa.sel / sa.sel_count (another layer's), read after the
  // dependency wait (the append still runs)
  int reuse;
  // append (nullable new_k): the newest token of every pair, [batch][Hkv][128]
  // bf16, is written at position seq_lens - 1 of the cache and widens its
  // block's summary before the block is scored
  const __nv_bfloat16* new_k;
  const __nv_bfloat16* new_v;
  __nv_bfloat16* k_pages_w;
  __nv_bfloat16* v_pages_w;
  __nv_bfloat16* smin_w;
  __nv_bfloat16* smax_w;
};

// Sends a split's result for head h to the CTA that merges it: CTA h / hp,
// slot (split, h % hp) of its push buffer.
struct ClusterPush {
  float* buf;  // the push buffer (same offset in every CTA of the cluster)
  int hp, split;
  __device__ __forceinline__ void operator()(int h, int c, float o, float lse) const {
    float* dst = cg::this_cluster().map_shared_rank(buf, static_cast<unsigned>(h / hp));
    const int slot = split * hp + h % hp;
    dst[slot * 128 + c] = o;
    if (c == 0) dst[kPushSlots * 128 + slot] = lse;
  }
};

__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

template <int NH>
__global__ void __launch_bounds__(kThreadsB, 1)
    score_select_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                             const __grid_constant__ CUtensorMap tm_smax, const __grid_constant__ CUtensorMap tm_smin,
                             TcArgs a, SelectArgs sa, FuseArgs f, unsigned* err) {
  using FL = FuseLayout<NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t tile_full = sbase + FL::kOffBar, q_full = tile_full + 8, acc_full = tile_full + 16;
  // one abort flag for all phases (the attention's), so that a wait that ran
  // out in phase 1 also stops the attention of phase 3
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Layout<NH>::kOffMisc + 4);
  int2* s_list = reinterpret_cast<int2*>(smem + FL::kOffList);
  float* s_scores = reinterpret_cast<float*>(smem + kFScores);
  float* s_prev = reinterpret_cast<float*>(smem + kFPrev);
  auto s_hist = reinterpret_cast<uint32_t(*)[sel::kHistWords]>(smem + kFHist);
  int* s_warp = reinterpret_cast<int*>(smem + kFWarp);
  uint32_t* s_range = reinterpret_cast<uint32_t*>(smem + kFRange);
  int* s_pt = reinterpret_cast<int*>(smem + kFPt);
  int* s_sel = reinterpret_cast<int*>(smem + kFSel);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int pair = blockIdx.x / f.cluster;
  const int b = pair / a.hkv, kvh = pair - b * a.hkv;
  const int g = a.group;
  const bool smoothed = sa.history_weight != 0.0f && sa.history != nullptr;

  pdl_trigger();
  // barriers of phase 1, and the attention's barriers and TMEM (its S
  // columns hold the bound accumulator in phase 1); the four tensor maps
  if (warp == kProdB && lane == 0) {
    prefetch_tmap(&tm_smax);
    prefetch_tmap(&tm_smin);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (tid == 0) {
    mbar_init(tile_full, 1);
    mbar_init(q_full, 128);
    mbar_init(acc_full, 1);
    abort_flag[0] = 0;
    abort_flag[2] = 0;
  }
  attn_bf16_setup<NH>(smem);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<uint32_t*>(smem + Layout<NH>::kOffMisc);
  cluster_arrive_relaxed();  // completes once every CTA of the cluster runs
  // the summary tile is requested before the request's length is known (rows
  // past its blocks are never used); with f.early before the previous kernel
  // has completed (the caller guarantees that it does not write them)
  auto load_tile = [&]() {
    mbar_arrive_tx(tile_full, bound::kTileBytes);
    const int y = pair * a.max_blocks + rank * bound::kTile;
    const uint32_t st = sbase + kFTile;
    tma_load_2d(st, &tm_smax, 0, y, tile_full);
    tma_load_2d(st + bound::kHalf, &tm_smax, 64, y, tile_full);
    tma_load_2d(st + 2 * bound::kHalf, &tm_smin, 0, y, tile_full);
    tma_load_2d(st + 3 * bound::kHalf, &tm_smin, 64, y, tile_full);
  };
  const bool tile_loaded = !f.reuse && rank < f.tiles;
  if (f.early && warp == kProdB && lane == 0 && tile_loaded) load_tile();
  pdl_wait();  // q, the summaries, seq_lens, the page table and the history of this step are complete
  if (!f.early && warp == kProdB && lane == 0 && tile_loaded) load_tile();
  const int L = max(a.seq_lens[b], 0);
  int nb = (L + a.block - 1) / a.block;
  if (nb > a.max_blocks) {
    if (tid == 0 && rank == 0) set_error(err, HS_EBIT_BLOCK_RANGE);
    nb = a.max_blocks;
  }
  const bool has_tile = tile_loaded && rank * bound::kTile < nb;
  const int32_t* pt = a.page_table + static_cast<int64_t>(pair) * a.max_blocks;

  // ---- phase 1: bound scores of tile `rank` ----
  bool bound_issued = false;
  if (warp == kMma1B) {
    if (lane == 0 && has_tile && mbar_wait(q_full, 0, abort_flag, a.wait_ns) &&
        mbar_wait(tile_full, 0, abort_flag, a.wait_ns)) {
      tc_fence_after();
      bound::issue_mmas(tmem, sbase + kFTile, sbase + kFQ);
      mma_commit(acc_full);
      bound_issued = true;
    }
  } else if (warp < 4) {
    if (has_tile) bound::write_q(smem + kFQ, a.q, static_cast<int64_t>(b) * a.hq + kvh * g, g, tid);
    if (f.new_k && L > 0 && rank == (f.reuse ? 0 : (nb - 1) / bound::kTile)) {
      // append ("KV 稀疏化" wiki §5: the summary of the newest token's block
      // covers it): thread t writes channel t of the token's K and V rows into
      // its page and widens the block's min/max row, in the staged tile the
      // MMAs read and in global memory (a token in row 0 starts the box)
      const int jl = nb - 1, tok = (L - 1) - jl * a.block;
      const int page = pt[jl];
      const bool page_ok = page >= 0 && page < a.num_pages;
      if (!page_ok && tid == 0) set_error(err, HS_EBIT_PAGE_RANGE);
      const int64_t src = static_cast<int64_t>(pair) * kD + tid;
      const __nv_bfloat16 kx = f.new_k[src], vx = f.new_v[src];
      if (page_ok) {
        const int64_t row = (static_cast<int64_t>(page) * a.block + tok) * kD + tid;
        f.k_pages_w[row] = kx;
        f.v_pages_w[row] = vx;
      }
      const int64_t so = (static_cast<int64_t>(pair) * a.max_blocks + jl) * kD + tid;
      if (f.reuse) {  // no staged tile: the block's row of smin/smax in global memory
        const float kf = __bfloat162float(kx);
        f.smin_w[so] = tok == 0 ? kx : __float2bfloat16_rn(fminf(__bfloat162float(f.smin_w[so]), kf));
        f.smax_w[so] = tok == 0 ? kx : __float2bfloat16_rn(fmaxf(__bfloat162float(f.smax_w[so]), kf));
      } else if (mbar_wait(tile_full, 0, abort_flag, a.wait_ns)) {
        const int r = jl - rank * bound::kTile, h = tid >> 6, cc = tid & 63;
        const uint32_t off = r * 128 + ((((cc >> 3) ^ (r & 7))) << 4) + (cc & 7) * 2;
        __nv_bfloat16* mx = reinterpret_cast<__nv_bfloat16*>(smem + kFTile + h * bound::kHalf + off);
        __nv_bfloat16* mn = reinterpret_cast<__nv_bfloat16*>(smem + kFTile + (2 + h) * bound::kHalf + off);
        const float kf = __bfloat162float(kx);
        *mn = tok == 0 ? kx : __float2bfloat16_rn(fminf(__bfloat162float(*mn), kf));  // exact: bf16 values
        *mx = tok == 0 ? kx : __float2bfloat16_rn(fmaxf(__bfloat162float(*mx), kf));
        f.smin_w[so] = *mn;
        f.smax_w[so] = *mx;
      }
      // the rows written here are read by the copies (async proxy) of phase 3
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    if (has_tile) {
      fence_async_smem();
      mbar_arrive(q_full);
    }
  } else if (warp < 8) {
    // the pair's page-table row and score history, cleared histograms; with
    // reuse the given selection and its count
    const int t = tid - 128;
    for (int j = t; j < nb; j += 128) s_pt[j] = pt[j];
    if (f.reuse) {
      const int cnt = max(0, min(sa.sel_count[pair], sa.capacity));
      const int32_t* src = sa.sel + static_cast<int64_t>(pair) * sa.capacity;
      for (int j = t; j < cnt; j += 128) s_sel[j] = src[j];
      if (t == 0) s_warp[0] = cnt;
    }
    if (smoothed && !f.reuse) {
      const float* h = sa.history + static_cast<int64_t>(pair) * a.max_blocks;
      for (int j = t; j < nb; j += 128) s_prev[j] = h[j];
    }
    for (int i = t; i < sel::kHistWords; i += 128) s_hist[0][i] = 0u;
  } else if (warp == kMma2B && rank == 0) {
    // K/V pages of the forced blocks (sink, window) into L2 ahead of phase 3
    const int B = a.block;
    const int n_sink = min(nb, ceil_div(sa.sink_tokens, B));
    int w_first = nb;
    if (sa.window_tokens > 0) w_first = (L - sa.window_tokens <= 0) ? 0 : min(nb, (L - sa.window_tokens) / B);
    w_first = max(w_first, n_sink);
    const int nf = n_sink + (nb - w_first);
    const uint32_t page_bytes = static_cast<uint32_t>(B) * kD * 2;
    for (int i = lane; i < nf; i += 32) {
      const int j = i < n_sink ? i : w_first + (i - n_sink);
      const int page = pt[j];
      if (page >= 0 && page < a.num_pages) {
        prefetch_l2(f.k_pages + static_cast<int64_t>(page) * page_bytes, page_bytes);
        prefetch_l2(f.v_pages + static_cast<int64_t>(page) * page_bytes, page_bytes);
      }
    }
  }
  cluster_wait();  // every CTA of the cluster runs: its shared memory is addressable
  if (warp < 4 && has_tile) {
    float best = -INFINITY;
    if (__all_sync(0xffffffffu, mbar_wait(acc_full, 0, abort_flag, a.wait_ns))) {  // warp-wide TMEM load
      tc_fence_after();
      float u[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16), u);
      tc_fence_before();
#pragma unroll
      for (int h = 0; h < 16; ++h)
        if (h < g) best = fmaxf(best, u[h]);
    }
    const int j = rank * bound::kTile + tid;
    if (j < nb && f.scores) f.scores[static_cast<int64_t>(pair) * a.max_blocks + j] = best;
    for (int r = 0; r < f.cluster; ++r) {  // every CTA of the cluster gets the tile's scores
      if (j < nb) cluster.map_shared_rank(s_scores, r)[j] = best;
      sel::warp_key_range(best, j < nb && !sel::is_forced(j, L, a.block, sa.sink_tokens, sa.window_tokens),
                          cluster.map_shared_rank(s_range, r), rank * 4 + warp);
    }
  }
  if (warp == kProdB && lane == 0 && tile_loaded)  // the tile has landed before the ring is reused
    mbar_drain(tile_full, 0);
  if (bound_issued) mbar_drain(acc_full, 0);  // the bound product is done before TMEM is reused
  if (!f.reuse)
    cluster.sync();  // every CTA holds all scores; from here only phase 3's pushes reach another CTA's shared memory
  else
    __syncthreads();  // the reused selection and the page-table row are staged

  // ---- phase 2: every CTA selects (rank 0 stores the selection), or takes the reused one ----
  int n;
  if (f.reuse) {
    n = s_warp[0];
  } else {
    if (smoothed) sel::smooth_staged(s_scores, s_prev, nb, a.max_blocks, sa, pair, rank == 0);
    static_assert(kThreadsB * 3 >= kFuseMaxBlocks, "three blocks per thread cover the pair");
    n = sel::select_pair_regs<kThreadsB, 3>(s_scores, nb, L, a.block, sa, pair, s_hist, s_warp, err, s_sel,
                                            smoothed ? nullptr : s_range, 4 * ceil_div(nb, bound::kTile), rank == 0);
  }
  __syncthreads();  // the shared copy of the selection is complete (s_warp is free again)
  const int bpc = kChunk / a.block;
  const int per = split_len(n, bpc, a.splits, a.bps);
  const int s0 = min(n, rank * per), s1 = min(n, s0 + per);
  unsigned bad = 0;
  for (int p = s0 + tid; p < s1 && rank < a.splits; p += kThreadsB) {
    const int j = s_sel[p];
    int2 e = make_int2(-1, 0);
    if (j < 0 || j >= nb) {
      bad |= HS_EBIT_BLOCK_RANGE;
    } else {
      const int page = s_pt[j];
      if (page < 0 || page >= a.num_pages)
        bad |= HS_EBIT_PAGE_RANGE;
      else
        e = make_int2(page, min(a.block, L - j * a.block));
    }
    s_list[p - s0] = e;
  }
  if (bad) set_error(err, bad);
  if (*abort_flag && tid == 0) report_timeout(err, kTimeoutStepFused, static_cast<unsigned>(abort_flag[2]));
  fence_async_smem();  // the scratch's generic writes before the ring's TMA writes
  __syncthreads();

  // ---- phase 3: attention over split `rank`; its result per head goes to
  // the push buffer of the CTA that merges that head ----
  const int hp = (g + f.cluster - 1) / f.cluster;  // heads merged per CTA
  float* push = reinterpret_cast<float*>(smem + FL::kOffPush);
  const Work w{rank < a.splits ? pair * a.splits + rank : a.items, a.items, s_list, s0, s1, L, a.items};
  attn_bf16_cta<NH, false, ClusterPush>(&tm_k, &tm_v, a, w, err, ClusterPush{push, hp, rank});

  // ---- phase 4: the splits' log-sum-exp merge inside the cluster
  // ("分块稀疏注意力与KV Cache量化" §2.2), the same arithmetic in the same
  // order as the merge kernel; CTA r merges heads r*hp .. r*hp+hp-1 from its
  // own push buffer ----
  cluster.sync();  // every split's results are in the merging CTAs' push buffers
  {
    const int S = a.splits;
    for (int idx = tid; idx < hp * 128; idx += kThreadsB) {
      const int hl = idx / 128, c = idx % 128, h = rank * hp + hl;
      if (h >= g) break;
      float M = -INFINITY;
      for (int sp = 0; sp < S; ++sp) M = fmaxf(M, push[kPushSlots * 128 + sp * hp + hl]);
      float acc = 0.0f, lse = -INFINITY;
      if (M != -INFINITY) {
        float tot = 0.0f;
        for (int sp = 0; sp < S; ++sp) {
          const float wgt = expf(push[kPushSlots * 128 + sp * hp + hl] - M);
          tot += wgt;
          acc = wgt > 0.0f ? fmaf(wgt, push[(sp * hp + hl) * 128 + c], acc) : acc;
        }
        acc = acc / tot;
        lse = M + logf(tot);
      }
      const int64_t orow = static_cast<int64_t>(b) * a.hq + static_cast<int64_t>(kvh) * g + h;
      if (a.out_f32)
        static_cast<float*>(a.out)[orow * kD + c] = acc;
      else
        static_cast<__nv_bfloat16*>(a.out)[orow * kD + c] = __float2bfloat16_rn(acc);
      if (a.lse_out && c == 0) a.lse_out[orow] = lse;
    }
  }
}

// ============================================================================
// e4m3 K/V (one fp32 scale per 32 channels per token), head_dim 128, g <= 8.
//
// GEMM1 reads the K codes as TMA staged them (kind::f8f6f4, both operands
// e4m3).  The query side is e4m3 too: each head's bf16 query row, times a
// power of two 2^a_h that brings its largest entry into [128, 256), is split
// into two e4m3 terms q1 + q2 whose sum is that row exactly (a bf16 value has
// 8 significant bits, a term 4; entries below 2^-10 of 2^-a_h, where q2 is
// subnormal, keep an error under 2^-10 * 2^-a_h).  The terms are 64 rows of
// one B operand, side by side in N:
//   GEMM1  S'[tok][(term, grp, h)] = sum_{d in grp} code_k[tok][d] * q_term[h][d]
//          (N = 2 terms x 4 groups x 8 heads, four MMAs of 32 codes)
//          S[tok][h] = 2^-a_h * sum_grp kscale[tok][grp] * (S'[tok][(1, grp, h)] + S'[tok][(2, grp, h)])
//   GEMM2  O[d][(hl, h)] = sum_tok v[tok][d] * P_hl[tok][h],  N = 16, f16 operands,
//          v = code_v * vscale in f16 (scale and product each rounded once:
//          relative error <= 2^-10), P split into f16 hi + lo.
// TMA stages the codes (K with the 128-byte swizzle the MMA reads) and the
// scales, four stages.  Two converter warpgroups (two threads per row) turn
// V codes times their scales into one of two f16 V tiles once GEMM2 of the
// chunk two back is done with it (each tile has its own free barrier).  The
// ring is the deeper of the two: the loads in flight set the chunk rate, and
// a V tile is free again soon after its product is issued.  Two softmax groups of 4 warps take the
// chunks alternately (group g the chunks c with c % 2 == g, with its own S,
// O and running state, combined at the end of an item); a group releases a
// stage once GEMM1 of its chunk is complete and its K scales are read, and
// takes the O of its previous chunk before it writes P of chunk c into its
// own P buffer.
// ============================================================================
constexpr int kStages8 = 4;
constexpr int kVTiles = 2;                        // f16 V tiles: chunk c converts into tile c % 2
constexpr int kCodeBytes = kChunk * 128;          // 128 tokens x 128 codes
constexpr int kScaleBytes = kChunk * 16;          // 128 tokens x 4 scales
constexpr int kStage8Bytes = 2 * kCodeBytes + 2 * kScaleBytes;
constexpr int kConv8Warp0 = 4;                    // warps 4-11 convert V; 0-3 and 15-18 are the softmax groups
struct Layout8 {
  static constexpr int kOffVh = kStages8 * kStage8Bytes;     // kVTiles f16 V tiles
  static constexpr int kQTerm = 32 * 128;                    // one e4m3 query term: 32 rows (group x head) x 128 codes
  static constexpr int kOffQ = kOffVh + kVTiles * kTileBytes;
  static constexpr int kPLbo = 8 * 16 * 2;                   // bytes between 8-token groups of P
  static constexpr int kPBytes = kChunk * 16 * 2;            // 128 tokens x (hi, lo) x 8 heads, f16
  static constexpr int kPBufs = 2;                           // one per softmax group
  static constexpr int kOffP = kOffQ + 2 * kQTerm;
  static constexpr int kOffBar = kOffP + kPBufs * kPBytes;
  static constexpr int kNumBars = 2 * kStages8 + 9 + 2 * kVTiles + kPBufs;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kOffRed = kOffMisc + 16;             // per group: 2 x [4 warps][8] maxima, [4][8] sums
  // (group 1's o [8][128] is handed to group 0 at the end of an item in its
  // own P buffer, its m [8] and l [8] in its chunk-max buffers: both are free
  // once the group's last P.V product is taken)
  static constexpr int kOffMeta = kOffRed + 2 * 3 * 4 * 8 * 4;
  static constexpr int kOffProg = kOffMeta + kStages8 * 8 * 8;  // progress words (as in the bf16 kernel)
  static constexpr int kOffQx = (kOffProg + 32 + 15) / 16 * 16;  // per head: the exponent a_h of the item's query,
  static constexpr int kBytes = kOffQx + 64;                     // then the softmax scale times 2^-a_h (16-byte loads)
  static constexpr int kAlloc = (kBytes + 1024 + 127) / 128 * 128;  // layout + base alignment
  static_assert(kAlloc <= 232448, "shared memory layout too large");
  static_assert(kStage8Bytes % 1024 == 0 && kOffVh % 1024 == 0 && kOffQ % 1024 == 0 && kOffP % 1024 == 0,
                "swizzled tiles need 1024-byte alignment");
  static_assert(kOffQx % 16 == 0 && kOffMeta % 8 == 0 && kOffBar % 8 == 0, "vector accesses need alignment");
  static constexpr int kTmemCols = 256;
  static constexpr int kColO = 128;  // S' of group g: columns [64 g, 64 g + 64); O of group g: [128 + 16 g, +16)
};

// Half a token row of e4m3 codes (channels 64 cp .. 64 cp + 63) -> f16 in a
// 128-byte-swizzled K-major tile, each code multiplied by its 32-channel
// group's scale in f16 (the scale and the product each rounded once); zeros
// for a row of no token.  Two threads per row (r, cp = 0, 1); the 16-byte
// segments are staggered so that eight consecutive threads touch eight
// different bank groups on the loads and on the stores.  In two parts: the
// codes and scales out of the stage into registers (after which the stage
// may be refilled), then the conversion into the tile.
struct HalfRow {
  uint4 raw[4];
  float2 s2;
};
__device__ __forceinline__ HalfRow load_half_row(const uint8_t* codes_row, const float* scales, int r, int cp,
                                                 bool valid) {
  HalfRow h;
  h.s2 = valid ? *reinterpret_cast<const float2*>(scales + 2 * cp) : make_float2(0.0f, 0.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    h.raw[i] = valid ? *reinterpret_cast<const uint4*>(codes_row + (4 * cp + ((i + r + 2 * cp) & 3)) * 16)
                     : make_uint4(0, 0, 0, 0);
  return h;
}
__device__ __forceinline__ void store_half_row(const HalfRow& hr, uint8_t* tile, int r, int cp) {
  const __half2 sc[2] = {__float2half2_rn(hr.s2.x), __float2half2_rn(hr.s2.y)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ch = 4 * cp + ((i + r + 2 * cp) & 3);  // 16-code segment of the row
    const uint32_t words[4] = {hr.raw[i].x, hr.raw[i].y, hr.raw[i].z, hr.raw[i].w};
    uint32_t w[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int hw = 0; hw < 2; ++hw) {
        const __half2_raw h =
            __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>((words[j] >> (16 * hw)) & 0xffffu), __NV_E4M3);
        uint32_t bits = static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
        const __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&bits), sc[(ch & 3) >> 1]);
        w[2 * j + hw] = *reinterpret_cast<const uint32_t*>(&v);
      }
    }
    uint8_t* row = tile + (ch >> 2) * kHalfBytes + r * 128;
    const int lc = (ch & 3) * 2;
    *reinterpret_cast<uint4*>(row + (((lc) ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(row + (((lc + 1) ^ (r & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <class W>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_fp8_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       TcArgs a, unsigned* err) {
  using Ly = Layout8;
  constexpr int NH = 8;
  const W w = persistent_work<W>(a);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + Ly::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (kStages8 + s); };
  auto s_full = [&](int b) { return bar0 + 8 * (2 * kStages8 + b); };      // per group
  auto s_free = [&](int b) { return bar0 + 8 * (2 * kStages8 + 2 + b); };  // per group
  auto o_full = [&](int b) { return bar0 + 8 * (2 * kStages8 + 4 + b); };  // per group
  auto o_free = [&](int b) { return bar0 + 8 * (2 * kStages8 + 6 + b); };  // per group
  const uint32_t q_full = bar0 + 8 * (2 * kStages8 + 8);
  auto vconv_full = [&](int b) { return bar0 + 8 * (2 * kStages8 + 9 + b); };            // per V tile
  auto vfree = [&](int b) { return bar0 + 8 * (2 * kStages8 + 9 + kVTiles + b); };        // per V tile
  auto p_full = [&](int b) { return bar0 + 8 * (2 * kStages8 + 9 + 2 * kVTiles + b); };  // per P buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly::kOffMisc + 4);
  volatile int* s_last = reinterpret_cast<volatile int*>(smem + Ly::kOffMisc + 8);  // last split of an item
  volatile int* prog = reinterpret_cast<volatile int*>(smem + Ly::kOffProg);
  auto vc_stage = [&](int s) { return smem + s * kStage8Bytes + kCodeBytes; };
  auto ks_stage = [&](int s) { return smem + s * kStage8Bytes + 2 * kCodeBytes; };
  auto vs_stage = [&](int s) { return smem + s * kStage8Bytes + 2 * kCodeBytes + kScaleBytes; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.block;
  const int bpc = kChunk / B;

  pdl_trigger();
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (tid == 0) {
    for (int s = 0; s < kStages8; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 384);  // released by the converters and the chunk's softmax group
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_free(b), 128);
      mbar_init(o_full(b), 1);
      mbar_init(o_free(b), 128);
    }
    for (int b = 0; b < kVTiles; ++b) {
      mbar_init(vconv_full(b), 256);
      mbar_init(vfree(b), 1);
    }
    for (int b = 0; b < Ly::kPBufs; ++b) mbar_init(p_full(b), 128);
    mbar_init(q_full, 128);
    abort_flag[0] = 0;
    abort_flag[2] = 0;
    for (int i = 0; i < 8; ++i) prog[i] = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), Ly::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  int2* meta = reinterpret_cast<int2*>(smem + Ly::kOffMeta);
  if (warp == kProducerWarp) {
    run_producer<kStages8>(a, w, bpc, full_bar(0), empty_bar(0), meta, 2u * B * 128u + 2u * B * 16u, abort_flag, err,
                           prog, [&](int s, int bi, int page) {
                             const int y = page * B;
                             tma_load_2d(sbase + s * kStage8Bytes + bi * B * 128, &tm_k, 0, y, full_bar(s));
                             tma_load_2d(smem_u32(vc_stage(s)) + bi * B * 128, &tm_v, 0, y, full_bar(s));
                             bulk_load(smem_u32(ks_stage(s)) + bi * B * 16, a.k_scales + static_cast<int64_t>(y) * 4,
                                       B * 16, full_bar(s));
                             bulk_load(smem_u32(vs_stage(s)) + bi * B * 16, a.v_scales + static_cast<int64_t>(y) * 4,
                                       B * 16, full_bar(s));
                           });
  } else if (warp == kMmaWarp || warp == kMma2Warp || warp == kMma3Warp) {
    if (lane == 0) {
      const bool first = warp == kMmaWarp;
      const int par = warp == kMma2Warp ? 0 : 1;  // a P.V issuer's chunk parity
      constexpr uint32_t idesc1 = idesc_e4m3(128, 64);
      constexpr uint32_t idesc2 = idesc_f16(128, 2 * NH, true, true);
      const uint64_t kdesc = smem_desc(sbase, 16, 1024, 2);  // stage 0's K codes
      const uint64_t qdesc = smem_desc(sbase + Ly::kOffQ, 16, 1024, 2);
      const uint64_t vdesc = smem_desc(sbase + Ly::kOffVh, kHalfBytes, 1024, 2);
      const uint64_t pdesc = smem_desc(sbase + Ly::kOffP, Ly::kPLbo, 128, 0);
      int c = 0, qi = 0;
      int item = w.first;
      Item it = item < w.end ? item_geom(a, item, bpc, w) : Item{};
      bool ok = true;
      while (ok && item < w.end && !*abort_flag) {
        const int next = item + w.stride;
        const Item nit = next < w.end ? item_geom(a, next, bpc, w) : Item{};
        if (it.nch > 0 && first) {
          ok = mbar_wait(q_full, qi & 1, abort_flag, a.wait_ns);
          ++qi;
        }
        for (int ci = 0; ok && ci < it.nch; ++ci, ++c) {
          const int bb = c & 1;  // the chunk's softmax group
          if (first) {
            const int s = c % kStages8;
            ok = mbar_wait(full_bar(s), (c / kStages8) & 1, abort_flag, a.wait_ns) &&
                 (c < 2 || mbar_wait(s_free(bb), ((c >> 1) + 1) & 1, abort_flag, a.wait_ns));
            if (!ok) break;
            tc_fence_after();
            // four K steps of 32 codes; both query terms (64 rows) in each
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t koff = s * kStage8Bytes + k * 32;
              mma_e4m3(tmem + bb * 64, kdesc + (koff >> 4), qdesc + ((k * 32) >> 4), idesc1, k > 0 ? 1u : 0u);
            }
            mma_commit(s_full(bb));
            prog[1] = c + 1;
          } else {
            if (bb != par) continue;
            const int pb = c % Ly::kPBufs, vt = c % kVTiles;
            ok = mbar_wait(p_full(pb), (c / Ly::kPBufs) & 1, abort_flag, a.wait_ns) &&
                 mbar_wait(vconv_full(vt), (c / kVTiles) & 1, abort_flag, a.wait_ns) &&
                 (c < 2 || mbar_wait(o_free(bb), ((c >> 1) + 1) & 1, abort_flag, a.wait_ns));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < kChunk / 16; ++k) {
              const uint32_t voff = vt * kTileBytes + k * 2048;
              const uint32_t poff = pb * Ly::kPBytes + k * 2 * Ly::kPLbo;
              mma_f16(tmem + Ly::kColO + bb * 16, vdesc + (voff >> 4), pdesc + (poff >> 4), idesc2, k > 0 ? 1u : 0u);
            }
            mma_commit(o_full(bb));
            mma_commit(vfree(vt));
            prog[2] = c + 1;
          }
        }
        item = next;
        it = nit;
      }
      // every product this thread issued is complete before TMEM is released
      // (a commit arrives once all of the thread's earlier MMAs are done)
      if (first && c > 0) mbar_drain(s_full((c - 1) & 1), ((c - 1) >> 1) & 1);
      if (!first) {
        const int last = ((c - 1) & 1) == par ? c - 1 : c - 2;  // this issuer's last chunk
        if (last >= 0) mbar_drain(o_full(par), (last >> 1) & 1);
      }
    }
  } else if (warp >= kConv8Warp0 && warp < kConv8Warp0 + 8) {
    // ================= V conversion: e4m3 rows times scales -> f16 V tiles =================
    // threads (r, cp) take half cp of row r of chunk c out of the stage,
    // release their part of it, and convert it into V tile c % 2 once the
    // P.V product of chunk c-2 is done with that tile
    const int ct = tid - kConv8Warp0 * 32;  // 0..255
    const int r = ct >> 1, cp = ct & 1;
    int c = 0;
    bool ok = true;
    for (int item = w.first; ok && item < w.end && !*abort_flag; item += w.stride) {
      const Item it = item_geom(a, item, bpc, w);
      for (int ci = 0; ci < it.nch; ++ci, ++c) {
        const int s = c % kStages8;
        const int vt = c % kVTiles;  // its last reader, the P.V product of chunk c - 2
        ok = mbar_wait(full_bar(s), (c / kStages8) & 1, abort_flag, a.wait_ns);
        if (!ok) break;
        const int2 md = meta[s * 8 + r / B];
        const bool valid = md.x >= 0 && (r % B) < md.y;
        const HalfRow hr = load_half_row(vc_stage(s) + r * 128, reinterpret_cast<const float*>(vs_stage(s) + r * 16),
                                         r, cp, valid);
        mbar_arrive(empty_bar(s));  // (the arrival's release orders the reads above before the stage's refill)
        ok = c < kVTiles || mbar_wait(vfree(vt), ((c / kVTiles) - 1) & 1, abort_flag, a.wait_ns);
        if (!ok) break;
        store_half_row(hr, smem + Ly::kOffVh + vt * kTileBytes, r, cp);
        fence_async_smem();
        mbar_arrive(vconv_full(vt));
      }
    }
  } else {
    // ================= softmax / correction: two groups of 4 warps =================
    const int grp = warp < 4 ? 0 : 1;
    const int wq = warp & 3;      // TMEM lane quarter
    const int t = wq * 32 + lane;  // token row of S, channel of O
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const int bar = 1 + grp;      // the group's named barrier; 3 = both groups
    const int g = a.group;
    float* red = reinterpret_cast<float*>(smem + Ly::kOffRed) + grp * 3 * 4 * NH;
    float* xo = reinterpret_cast<float*>(smem + Ly::kOffP + Ly::kPBytes);  // group 1's P buffer
    float* xm = reinterpret_cast<float*>(smem + Ly::kOffRed) + 3 * 4 * NH;  // group 1's chunk maxima
    float* xl = xm + NH;
    int c = 0;
    // Query terms: row (cg, h) of each term holds head h's codes of channel
    // group cg, zeros elsewhere.  The zeros are written once; per item warp 0
    // (lane 4h + cg: head h, channel group cg) loads its 32 channels, takes
    // the head's largest entry over the four lanes of the head, and writes
    // the two 16-byte pieces of its row in both terms.
    int* s_qx = reinterpret_cast<int*>(smem + Ly::kOffQx);
    if (grp == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        reinterpret_cast<uint4*>(smem + Ly::kOffQ)[t * 4 + i] = make_uint4(0, 0, 0, 0);
      if (t < 8 && t >= g) {
        s_qx[t] = 0;
        reinterpret_cast<float*>(s_qx + 8)[t] = 0.0f;
      }
      named_barrier(bar, 128);  // the zeros are in place before warp 0 writes its pieces
    }
    auto write_q = [&](int item) {  // warp 0 of group 0
      const int pair = item_pair<W>(a, item), b = pair / a.hkv, kvh = pair - b * a.hkv;
      const int h = lane >> 2, cg = lane & 3;
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = make_uint4(0, 0, 0, 0);
      if (h < g) {
        const uint4* qr =
            reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(b) * a.hq + kvh * g + h) * kD + 32 * cg);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = qr[i];
      }
      uint32_t amax = 0u;  // bits of the largest |entry| (order of non-negative floats)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = max(amax, max(max(v[i].x & 0x7fff7fffu, v[i].y & 0x7fff7fffu),
                             max(v[i].z & 0x7fff7fffu, v[i].w & 0x7fff7fffu)) & 0xffff0000u);
        amax = max(amax, max(max((v[i].x << 16) & 0x7fff0000u, (v[i].y << 16) & 0x7fff0000u),
                             max((v[i].z << 16) & 0x7fff0000u, (v[i].w << 16) & 0x7fff0000u)));
      }
      amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      if (h >= g) return;
      // 2^ax brings the head's largest entry into [128, 256)
      int ex = 0;
      if (amax != 0u) frexpf(__uint_as_float(amax), &ex);
      const int ax = amax != 0u ? 8 - ex : 0;
      if (cg == 0) {
        s_qx[h] = ax;
        reinterpret_cast<float*>(s_qx + 8)[h] = ldexpf(a.scale_log2, -ax);
      }
      uint32_t w1[8], w2[8];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint4 vv = v[i >> 2];
        const uint32_t wq2 = (i & 3) == 0 ? vv.x : (i & 3) == 1 ? vv.y : (i & 3) == 2 ? vv.z : vv.w;
        const float y0 = ldexpf(__uint_as_float(wq2 << 16), ax), y1 = ldexpf(__uint_as_float(wq2 & 0xffff0000u), ax);
        const __nv_fp8x2_storage_t c1 = __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
        const __half2_raw h1 = __nv_cvt_fp8x2_to_halfraw2(c1, __NV_E4M3);
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h1));
        const __nv_fp8x2_storage_t c2 =
            __nv_cvt_float2_to_fp8x2(make_float2(y0 - f1.x, y1 - f1.y), __NV_SATFINITE, __NV_E4M3);
        if ((i & 1) == 0) {
          w1[i >> 1] = static_cast<uint32_t>(c1);
          w2[i >> 1] = static_cast<uint32_t>(c2);
        } else {
          w1[i >> 1] |= static_cast<uint32_t>(c1) << 16;
          w2[i >> 1] |= static_cast<uint32_t>(c2) << 16;
        }
      }
      // 16-byte pieces 2cg, 2cg+1 of row cg * 8 + h, 128-byte swizzle
      const int row = cg * 8 + h;
#pragma unroll
      for (int term = 0; term < 2; ++term) {
        uint8_t* rowp = smem + Ly::kOffQ + term * Ly::kQTerm + row * 128;
        const uint32_t* wv = term ? w2 : w1;
#pragma unroll
        for (int k = 0; k < 2; ++k)
          *reinterpret_cast<uint4*>(rowp + (((2 * cg + k) ^ (row & 7)) << 4)) =
              make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
      }
    };
    int item = w.first;
    Item it{};
    if (item < w.end) it = item_geom(a, item, bpc, w);
    // a wait that runs out is made uniform across the warp (warp-wide TMEM
    // loads), across a group at its named barrier and across both groups at
    // barrier 3 (bar.red.or), so that all leave the loops at the same point
    while (item < w.end) {
      const int next = item + w.stride;
      // the next item's two reads are issued now, its geometry computed at the end
      const ItemPre npre = next < w.end ? item_pre(a, next, w) : ItemPre{0, 0};
      if (it.nch == 0) {
        if (grp == 0) {
          for (int h = 0; h < g; ++h) put_partial(a, it, h, t, 0.0f, -INFINITY);
          if (it.nseg > 1 && a.counters) merge_if_last(a, it, t, bar, s_last);
        }
        item = next;
        it = next < w.end ? item_geom_from(a, next, bpc, w, npre) : Item{};
        continue;
      }
      if (grp == 0) {
        if (wq == 0) write_q(item);  // the item's query terms (every GEMM1 of the previous item is complete)
        fence_async_smem();
        mbar_arrive(q_full);
        if (t == 0) {
          prog[6] = item;
          prog[7] = it.nch;
        }
      }
      named_barrier(3, 256);  // the exponents a_h are written
      // per head log2(e) / sqrt(d) * 2^-a_h, read from shared memory at each chunk
      const float* s_sl = reinterpret_cast<const float*>(s_qx + 8);

      bool fail = false;  // this thread saw a wait run out (uniform per group)
      float m[NH], lsum[NH], oacc[NH], alpha_prev[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        m[h] = -INFINITY;
        lsum[h] = 0.0f;
        oacc[h] = 0.0f;
        alpha_prev[h] = 1.0f;
      }
      auto take_o = [&](int cc) -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait(o_full(grp), (cc >> 1) & 1, abort_flag, a.wait_ns))) return false;
        tc_fence_after();
        float ov[16];
        tmem_ld16(tmem + lane_base + Ly::kColO + grp * 16, ov);
        tc_fence_before();
        mbar_arrive(o_free(grp));
#pragma unroll
        for (int h = 0; h < NH; ++h) oacc[h] = fmaf(oacc[h], alpha_prev[h], ov[h] + ov[NH + h]);
        return true;
      };
      const int c0 = c;
      int last_own = -1;
      for (int cc = c0 + ((grp - c0) & 1); cc < c0 + it.nch; cc += 2) {
        const int s = cc % kStages8;
        // row t of the chunk: token t % B of its (t / B)-th block; its K
        // scales come from this chunk's stage
        bool ready = !fail && mbar_wait(full_bar(s), (cc / kStages8) & 1, abort_flag, a.wait_ns);
        const int2 md = ready ? meta[s * 8 + t / B] : make_int2(-1, 0);
        const bool valid_cur = md.x >= 0 && (t % B) < md.y;
        float ks_cur[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid_cur) {
          const float4 sc = *reinterpret_cast<const float4*>(ks_stage(s) + t * 16);
          ks_cur[0] = sc.x; ks_cur[1] = sc.y; ks_cur[2] = sc.z; ks_cur[3] = sc.w;
        }
        ready = __all_sync(0xffffffffu, ready && mbar_wait(s_full(grp), (cc >> 1) & 1, abort_flag, a.wait_ns));
        // S = sum over the 4 channel groups of kscale * (S' of term 1 + S' of term 2)
        float x[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) x[h] = 0.0f;
        if (ready) {
          tc_fence_after();
#pragma unroll
          for (int term = 0; term < 2; ++term) {
            float sv[32];
            tmem_ld32(tmem + lane_base + grp * 64 + term * 32, sv);
#pragma unroll
            for (int cg = 0; cg < 4; ++cg)
#pragma unroll
              for (int h = 0; h < NH; ++h) x[h] = fmaf(ks_cur[cg], sv[cg * 8 + h], x[h]);
          }
          tc_fence_before();
          mbar_arrive(s_free(grp));
          mbar_arrive(empty_bar(s));  // the stage's K codes, meta and K scales are used
        }
        {
          const float4 sa = *reinterpret_cast<const float4*>(s_sl), sb = *reinterpret_cast<const float4*>(s_sl + 4);
          const float sl[NH] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
          for (int h = 0; h < NH; ++h) x[h] = (valid_cur && h < g) ? x[h] * sl[h] : -INFINITY;
        }
        // the running max moves only when some row of the chunk exceeds it by
        // more than kLazyMax (one vote); otherwise P = 2^(x - m) <= 2^kLazyMax
        bool over = false;
#pragma unroll
        for (int h = 0; h < NH; ++h) over |= x[h] > m[h] + kLazyMax;
        float alpha[NH], p[NH];
        if (named_barrier_or(bar, 128, over || fail || !ready)) {
          // chunk max per head over the 128 rows: one warp reduction per head
          // (on order-preserving integer keys), then the 4 warps
          float* rb = red + ((cc >> 1) & 1) * 4 * NH;  // alternate buffers: a barrier per chunk at least
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const uint32_t k = __reduce_max_sync(0xffffffffu, float_order_key(x[h]));
            if (lane == h) rb[wq * NH + h] = order_key_float(k);
          }
          if (named_barrier_or(bar, 128, fail || !ready)) {
            fail = true;
            break;
          }
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            const float cm = fmaxf(fmaxf(rb[h], rb[NH + h]), fmaxf(rb[2 * NH + h], rb[3 * NH + h]));
            const float mn = fmaxf(m[h], cm);
            alpha[h] = (mn == -INFINITY) ? 1.0f : exp2f(m[h] - mn);
            m[h] = mn;
            p[h] = x[h] == -INFINITY ? 0.0f : exp2f(x[h] - mn);
            lsum[h] = fmaf(lsum[h], alpha[h], p[h]);
          }
        } else {
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            alpha[h] = 1.0f;
            p[h] = x[h] == -INFINITY ? 0.0f : exp2f(x[h] - m[h]);
            lsum[h] += p[h];
          }
        }
        // O of this group's previous chunk: its P.V product is then complete,
        // and with it the last read of this group's P buffer
        if (last_own >= 0 && !take_o(last_own)) fail = true;
        // P of chunk cc into the group's buffer, as f16 high part + remainder
        {
          uint32_t hi2[NH / 2], lo2[NH / 2];
#pragma unroll
          for (int h = 0; h < NH; h += 2) {
            const __half2 hi = __floats2half2_rn(p[h], p[h + 1]);
            const float2 hf = __half22float2(hi);
            const __half2 lo = __floats2half2_rn(p[h] - hf.x, p[h + 1] - hf.y);
            hi2[h / 2] = *reinterpret_cast<const uint32_t*>(&hi);
            lo2[h / 2] = *reinterpret_cast<const uint32_t*>(&lo);
          }
          uint8_t* prow = smem + Ly::kOffP + (cc % Ly::kPBufs) * Ly::kPBytes + (t >> 3) * Ly::kPLbo + (t & 7) * 16;
          *reinterpret_cast<uint4*>(prow) = make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
          *reinterpret_cast<uint4*>(prow + 128) = make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
        }
        fence_async_smem();
        mbar_arrive(p_full(cc % Ly::kPBufs));
        if (t == 0) prog[3 + grp] = cc + 1;
#pragma unroll
        for (int h = 0; h < NH; ++h) alpha_prev[h] = alpha[h];
        last_own = cc;
      }
      c = c0 + it.nch;
      // the normaliser reduction overlaps the last P.V product
      float* rs = red + 8 * NH;
      {
        float r[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) r[h] = lsum[h];
        const float wsum = warp_reduce_scatter<NH, false>(r);
        if ((lane % (32 / NH)) == 0) rs[wq * NH + lane / (32 / NH)] = wsum;
      }
      if (!fail && last_own >= 0 && !take_o(last_own)) fail = true;
      fail = named_barrier_or(bar, 128, fail);
      // combine the two groups' states: group 1 publishes, group 0 merges and writes
      if (grp == 1 && !fail) {
#pragma unroll
        for (int h = 0; h < NH; ++h) xo[h * 128 + t] = oacc[h];
#pragma unroll
        for (int h = 0; h < NH; ++h) {  // compile-time indices keep m[] in registers
          if (t == h) {
            xm[h] = m[h];
            xl[h] = rs[h] + rs[NH + h] + rs[2 * NH + h] + rs[3 * NH + h];
          }
        }
      }
      if (named_barrier_or(3, 256, fail)) break;  // both groups leave together after a wait ran out
      if (grp == 0) {
        float* fac = red;  // [NH][4], the chunk-max buffers are free after the chunk loop
        {
          // thread h < g takes head h: its running max picked out of m[] with
          // compile-time indices (m[] stays in registers), the arithmetic once
          const int h = t;
          float m0 = -INFINITY;
#pragma unroll
          for (int i = 0; i < NH; ++i) m0 = (i == h) ? m[i] : m0;
          if (h < g && h < NH) {
            const float l0 = rs[h] + rs[NH + h] + rs[2 * NH + h] + rs[3 * NH + h];
            const float m1 = xm[h], l1 = xl[h];
            const float mx = fmaxf(m0, m1);
            const float e0 = m0 == -INFINITY ? 0.0f : exp2f(m0 - mx);
            const float e1 = m1 == -INFINITY ? 0.0f : exp2f(m1 - mx);
            const float lt = l0 * e0 + l1 * e1;
            const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
            fac[4 * h] = e0 * inv;
            fac[4 * h + 1] = e1 * inv;
            fac[4 * h + 3] = lt > 0.0f ? (mx + log2f(lt)) * kLn2 : -INFINITY;
          }
        }
        named_barrier(bar, 128);
        // one copy of the output code for all heads: head h's accumulator
        // picked out of oacc[] with compile-time indices
#pragma unroll 1
        for (int h = 0; h < g && h < NH; ++h) {
          float oh = oacc[0];
#pragma unroll
          for (int i = 1; i < NH; ++i) oh = (i == h) ? oacc[i] : oh;
          put_partial(a, it, h, t, fmaf(oh, fac[4 * h], xo[h * 128 + t] * fac[4 * h + 1]), fac[4 * h + 3]);
        }
        if (it.nseg > 1 && a.counters) merge_if_last(a, it, t, bar, s_last);
      }
      named_barrier(3, 256);  // the exchange buffer and s_qx are free again
      item = next;
      it = next < w.end ? item_geom_from(a, next, bpc, w, npre) : Item{};
    }
  }

  tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) report_timeout(err, kTimeoutAttnE4m3, static_cast<unsigned>(abort_flag[2]), prog);
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, Ly::kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D view of a page pool [num_pages*B rows][128 channels] bf16; box = one
// page of rows x 64 channels (128 bytes), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int block) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(block)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D view of an e4m3 page pool [num_pages*B rows][128 codes]; box = one
// page; swizzled (the layout the MMA reads) or plain rows
bool make_map_codes(CUtensorMap* m, const void* base, int64_t rows, int block, bool swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD)};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(block)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

TcArgs make_args(const KvView& kv, const AttnArgs& aa) {
  TcArgs a;
  a.sel = aa.sel;
  a.sel_count = aa.sel_count;
  a.page_table = kv.page_table;
  a.seq_lens = kv.seq_lens;
  a.q = static_cast<const __nv_bfloat16*>(aa.q);
  a.k_scales = kv.k_scales;
  a.v_scales = kv.v_scales;
  a.ws_o = aa.ws_o;
  a.ws_lse = aa.ws_lse;
  a.out = aa.out;
  a.lse_out = aa.lse;
  a.counters = aa.counters;
  a.out_f32 = aa.out_is_fp32;
  a.num_pages = kv.num_pages;
  a.hkv = kv.hkv;
  a.hq = kv.hq;
  a.group = kv.group;
  a.block = kv.block;
  a.max_blocks = kv.max_blocks;
  a.capacity = aa.capacity;
  a.bps = aa.blocks_per_split;
  a.splits = aa.splits;
  a.stream_per = aa.stream_per;
  a.stream_n = aa.stream_n;
  a.items = kv.batch * kv.hkv * (aa.stream_per > 0 ? 1 : aa.splits);
  a.scale_log2 = aa.scale * kLog2e;
  a.wait_ns = aa.wait_ns > 0 ? aa.wait_ns : kWaitLimitNs;
  return a;
}


// Persistent grid: one CTA per balanced range, else min(items, CTAs allowed).
int attn_grid(const TcArgs& a, int sms) {
  if (a.stream_per > 0)
    return static_cast<int>((static_cast<int64_t>(a.items) * a.stream_n + a.stream_per - 1) / a.stream_per);
  return a.items < sms ? a.items : sms;
}

cudaError_t launch_fp8(const KvView& kv, AttnArgs& aa, unsigned* err, cudaStream_t st) {
  CUtensorMap mk, mv;
  const int64_t rows = kv.num_pages * kv.block;
  if (rows <= 0) return cudaErrorInvalidValue;
  if (!make_map_codes(&mk, kv.k_pages, rows, kv.block, true) || !make_map_codes(&mv, kv.v_pages, rows, kv.block, false))
    return cudaErrorInvalidValue;
  const TcArgs a = make_args(kv, aa);
  if (a.items == 0) return cudaSuccess;
  auto kern = a.stream_per > 0 ? attn_tc_fp8_kernel<RangeWork> : attn_tc_fp8_kernel<Work>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout8::kAlloc);
  if (e != cudaSuccess) return e;
  const int grid = attn_grid(a, aa.sms);
  TcArgs b = a;
  // CTAs with several uniform splits: the merge kernel is cheaper (balanced
  // ranges always merge in place)
  if (a.stream_per == 0 && a.items > grid) b.counters = nullptr;
  aa.merged = aa.splits == 1 || b.counters != nullptr;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), Layout8::kAlloc, st, mk, mv, b, err);
}

template <int NH>
cudaError_t launch_nh(const KvView& kv, AttnArgs& aa, unsigned* err, cudaStream_t st) {
  using Ly = Layout<NH>;
  CUtensorMap mk, mv;
  const int64_t rows = kv.num_pages * kv.block;
  if (rows <= 0) return cudaErrorInvalidValue;
  if (!make_map(&mk, kv.k_pages, rows, kv.block) || !make_map(&mv, kv.v_pages, rows, kv.block))
    return cudaErrorInvalidValue;
  const TcArgs a = make_args(kv, aa);
  if (a.items == 0) return cudaSuccess;
  auto kern = a.stream_per > 0 ? attn_tc_kernel<NH, RangeWork> : attn_tc_kernel<NH, Work>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Ly::kAlloc);
  if (e != cudaSuccess) return e;
  const int grid = attn_grid(a, aa.sms);
  TcArgs b = a;
  // CTAs with several uniform splits: the merge kernel is cheaper (balanced
  // ranges always merge in place)
  if (a.stream_per == 0 && a.items > grid) b.counters = nullptr;
  aa.merged = aa.splits == 1 || b.counters != nullptr;
  return launch_pdl(kern, dim3(grid), dim3(kThreadsB), Ly::kAlloc, st, mk, mv, b, err);
}

}  // namespace

bool score_select_attn_supported(const KvView& kv, const AttnArgs& aa, int sms) {
  if (kv.kv_dtype != HS_KV_BF16 || kv.group > 8 || aa.stream_per > 0 || !attn_tc_supported(kv)) return false;
  const int tiles = (kv.max_blocks + bound::kTile - 1) / bound::kTile;
  const int f = tiles > aa.splits ? tiles : aa.splits;
  const int64_t pairs = static_cast<int64_t>(kv.batch) * kv.hkv;
  if (f > kFuseMaxCluster || pairs * f > sms || aa.blocks_per_split > kFuseList) return false;
  if (aa.splits * ((kv.group + f - 1) / f) > kPushSlots) return false;  // the merging CTAs' push buffers
  return pairs * kv.max_blocks < (int64_t(1) << 31);
}

cudaError_t launch_score_select_attn(const KvView& kv, const void* smin, const void* smax, const SelectArgs& sa,
                                     AttnArgs& aa, unsigned* err, cudaStream_t st, const void* new_k,
                                     const void* new_v, bool reuse) {
  using FL = FuseLayout<8>;
  const int64_t pairs = static_cast<int64_t>(kv.batch) * kv.hkv;
  if (pairs == 0) return cudaSuccess;
  CUtensorMap mk, mv, mmax, mmin;
  const int64_t rows = kv.num_pages * kv.block;
  if (rows <= 0) return cudaErrorInvalidValue;
  if (!make_map(&mk, kv.k_pages, rows, kv.block) || !make_map(&mv, kv.v_pages, rows, kv.block) ||
      !make_map(&mmax, smax, pairs * kv.max_blocks, bound::kTile) ||
      !make_map(&mmin, smin, pairs * kv.max_blocks, bound::kTile))
    return cudaErrorInvalidValue;
  const TcArgs a = make_args(kv, aa);
  FuseArgs f;
  f.early = aa.early_summaries ? 1 : 0;
  f.reuse = reuse ? 1 : 0;
  f.scores = sa.scores;
  f.k_pages = static_cast<const uint8_t*>(kv.k_pages);
  f.v_pages = static_cast<const uint8_t*>(kv.v_pages);
  f.tiles = (kv.max_blocks + bound::kTile - 1) / bound::kTile;
  f.cluster = f.tiles > aa.splits ? f.tiles : aa.splits;
  f.new_k = static_cast<const __nv_bfloat16*>(new_k);
  f.new_v = static_cast<const __nv_bfloat16*>(new_v);
  f.k_pages_w = static_cast<__nv_bfloat16*>(const_cast<void*>(kv.k_pages));
  f.v_pages_w = static_cast<__nv_bfloat16*>(const_cast<void*>(kv.v_pages));
  f.smin_w = static_cast<__nv_bfloat16*>(const_cast<void*>(smin));
  f.smax_w = static_cast<__nv_bfloat16*>(const_cast<void*>(smax));
  auto kern = score_select_attn_kernel<8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, FL::kAlloc);
  if (e != cudaSuccess) return e;
  aa.merged = 1;  // the cluster merges its splits
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pairs * f.cluster));
  cfg.blockDim = dim3(kThreadsB);
  cfg.dynamicSmemBytes = FL::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = f.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, mk, mv, mmax, mmin, a, sa, f, err);
}

bool attn_tc_supported(const KvView& kv) {
  if (kv.head_dim != kD) return false;
  if (kv.kv_dtype == HS_KV_BF16) {
    if (kv.group > 16) return false;
  } else if (kv.kv_dtype == HS_KV_FP8E4M3_G32) {
    if (kv.group > 8 || !kv.k_scales || !kv.v_scales) return false;
  } else {
    return false;
  }
  if (kv.block != 16 && kv.block != 32 && kv.block != 64 && kv.block != 128) return false;
  if (kv.num_pages * kv.block >= (int64_t(1) << 31)) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_attn_tc(const KvView& kv, AttnArgs& a, unsigned* err, cudaStream_t st) {
  if (kv.kv_dtype == HS_KV_FP8E4M3_G32) return launch_fp8(kv, a, err, st);
  return kv.group <= 8 ? launch_nh<8>(kv, a, err, st) : launch_nh<16>(kv, a, err, st);
}

}  // namespace hs
