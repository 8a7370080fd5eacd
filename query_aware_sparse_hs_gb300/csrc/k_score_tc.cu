// Bound scoring on the tensor cores ("KV 稀疏化" wiki §5 Quest: coarse filter
// of the query against the per-block summaries), for bf16 summaries and
// head_dim 128.
//
//   U[j][h] = sum_d max(q_hd * smax_jd, q_hd * smin_jd)
//           = sum_d smax_jd * q+_hd + smin_jd * q-_hd,   q+ = max(q, 0), q- = min(q, 0)
//
// is one small GEMM per tile of 128 blocks: A = [Smax | Smin] (128 blocks x 256,
// K-major, straight from the summary array by TMA), B = [Q+ | Q-] (16 padded
// heads x 256).  Every product is exact (bf16 x bf16) and accumulates in fp32
// TMEM, so the result matches the CUDA-core bound up to summation order.  The
// block score is the max of U over the kv head's query heads; scores go to
// global memory and the selection kernel takes over.
//
// Persistent, warp-specialised CTA (one per SM): warp 4 streams summary tiles
// with TMA into a 3-stage ring, warp 5 issues the 16 MMAs of a tile into one of
// two TMEM accumulators, warps 0-3 write the [Q+ | Q-] operand of each tile's
// (request, kv head) and turn accumulator rows into block scores.
#include <cooperative_groups.h>
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
constexpr int kTile = bound::kTile;           // blocks per tile (MMA M)
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr int kHalf = bound::kHalf;
constexpr int kStageBytes = bound::kTileBytes;
constexpr int kQBytes = bound::kQBytes;
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffBar = kOffQ + 2 * kQBytes;
constexpr int kNumBars = 2 * kStages + 8;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kAlloc = 232448;
static_assert(kOffMisc + 32 + 1024 <= kAlloc, "shared memory layout too large");
constexpr int kTmemCols = 32;

struct ScoreArgs {
  const __nv_bfloat16* q;
  const int32_t* seq_lens;
  float* scores;
  int batch, hkv, hq, group, block, max_blocks, tiles, items;
};

// Blocks of request b (every kv head of it has as many).
__device__ __forceinline__ int request_blocks(const ScoreArgs& a, int b) {
  const int L = max(a.seq_lens[b], 0);
  return min((L + a.block - 1) / a.block, a.max_blocks);
}

// Position in the sequence of valid tiles (tile t of (request, kv head) pair
// holds blocks [t*128, t*128+128); it is valid when one of them is < N_b),
// taken pair by pair and tile by tile.
struct TileCursor {
  int pair, tile, nb;  // nb = blocks of the pair
};

__device__ __forceinline__ int tiles_of(int nb) { return (nb + kTile - 1) / kTile; }

// The next valid tile (pairs without blocks are skipped; past the last pair
// the cursor stays on a sentinel pair).
__device__ __forceinline__ void next_tile(const ScoreArgs& a, TileCursor& c) {
  if (++c.tile < tiles_of(c.nb)) return;
  c.tile = 0;
  const int pairs = a.batch * a.hkv;
  do {
    ++c.pair;
    c.nb = c.pair < pairs ? request_blocks(a, c.pair / a.hkv) : kTile;
  } while (c.nb == 0);
}

// The CTA's tiles: `count` consecutive valid tiles from `first`.
struct TileRun {
  TileCursor first;
  int count;
};

// Without FUSE the valid tiles of all pairs are cut into gridDim.x contiguous
// runs of (nearly) equal length, so that a CTA's tiles mostly share a pair
// and its query operand.  Run by one warp; the result is in every lane.
__device__ TileRun contiguous_run(const ScoreArgs& a) {
  const int lane = threadIdx.x & 31;
  int64_t total = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int b = b0 + lane;
    total += warp_sum(static_cast<int64_t>(b < a.batch ? tiles_of(request_blocks(a, b)) : 0));
  }
  total *= a.hkv;
  const int64_t start = total * blockIdx.x / gridDim.x, end = total * (blockIdx.x + 1) / gridDim.x;
  TileRun r{{0, 0, 0}, static_cast<int>(end - start)};
  if (r.count == 0) return r;
  int64_t acc = 0;  // valid tiles of the requests before this round of 32
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int b = b0 + lane;
    const int nb = b < a.batch ? request_blocks(a, b) : 0;
    const int64_t tb = static_cast<int64_t>(tiles_of(nb)) * a.hkv;
    int64_t incl = tb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const int64_t lo = acc + incl - tb;
    const unsigned hit = __ballot_sync(0xffffffffu, tb > 0 && start >= lo && start < lo + tb);
    if (hit) {
      const int src = __ffs(hit) - 1;
      int pair = 0, tile = 0;
      if (lane == src) {
        const int t = tiles_of(nb);
        const int64_t off = start - lo;
        const int kvh = static_cast<int>(off / t);
        tile = static_cast<int>(off - static_cast<int64_t>(kvh) * t);
        pair = b * a.hkv + kvh;
      }
      r.first.pair = __shfl_sync(0xffffffffu, pair, src);
      r.first.tile = __shfl_sync(0xffffffffu, tile, src);
      r.first.nb = __shfl_sync(0xffffffffu, nb, src);
      return r;
    }
    acc += __shfl_sync(0xffffffffu, incl, 31);
  }
  r.count = 0;
  return r;
}

// Moves a segment cursor (the first tile of a run of tiles of one pair, with
// `left` tiles of the CTA's run from there on) to the next segment; false
// when the run ends first.
__device__ __forceinline__ bool next_segment(const ScoreArgs& a, TileCursor& c, int& left) {
  left -= tiles_of(c.nb) - c.tile;
  if (left <= 0) return false;
  c.tile = tiles_of(c.nb) - 1;
  next_tile(a, c);
  return true;
}

// FUSE: launched as one cluster per (request, kv head) with one CTA per tile
// (every CTA takes exactly one item); once all tiles' scores are stored, rank
// 0 of the cluster reads them back and runs the selection itself.
template <bool FUSE>
__global__ void __launch_bounds__(kThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tm_max, const __grid_constant__ CUtensorMap tm_min,
                    ScoreArgs a, SelectArgs sa, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8 * s; };
  auto empty_bar = [&](int s) { return bar0 + 8 * (kStages + s); };
  auto acc_full = [&](int b) { return bar0 + 8 * (2 * kStages + b); };
  auto acc_free = [&](int b) { return bar0 + 8 * (2 * kStages + 2 + b); };
  auto q_full = [&](int b) { return bar0 + 8 * (2 * kStages + 4 + b); };
  auto q_free = [&](int b) { return bar0 + 8 * (2 * kStages + 6 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  pdl_trigger();
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tm_max);
    prefetch_tmap(&tm_min);
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_free(b), 128);
      mbar_init(q_full(b), 128);
      mbar_init(q_free(b), 1);
    }
    abort_flag[0] = 0;
    abort_flag[2] = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // q, the summaries and seq_lens of this step are complete

  // the CTA's tiles: one per CTA with FUSE, else a contiguous run of valid tiles
  int* s_run = reinterpret_cast<int*>(smem + kOffMisc + 16);
  if (warp == 0) {
    TileRun r;
    if constexpr (FUSE) {
      r.first.pair = blockIdx.x / a.tiles;
      r.first.tile = blockIdx.x - r.first.pair * a.tiles;
      r.first.nb = request_blocks(a, r.first.pair / a.hkv);
      r.count = r.first.tile * kTile < r.first.nb ? 1 : 0;
    } else {
      r = contiguous_run(a);
    }
    if (lane == 0) {
      s_run[0] = r.first.pair;
      s_run[1] = r.first.tile;
      s_run[2] = r.first.nb;
      s_run[3] = r.count;
    }
  }
  __syncthreads();
  const TileCursor first{s_run[0], s_run[1], s_run[2]};
  const int count = s_run[3];

  // A segment is a run of the CTA's tiles of one pair; segment s's [Q+ | Q-]
  // operand is in buffer s & 1, written by the epilogue warps a segment ahead.
  if (warp == kProducerWarp) {
    if (lane == 0) {
      TileCursor cur = first;
      int n = 0;
      for (; n < count && !*abort_flag; ++n) {
        const int s = n % kStages;
        if (n >= kStages && !mbar_wait(empty_bar(s), ((n / kStages) + 1) & 1, abort_flag)) break;
        mbar_arrive_tx(full_bar(s), 4u * kHalf);
        const int y = cur.pair * a.max_blocks + cur.tile * kTile;
        const uint32_t st = sbase + s * kStageBytes;
        tma_load_2d(st, &tm_max, 0, y, full_bar(s));
        tma_load_2d(st + kHalf, &tm_max, 64, y, full_bar(s));
        tma_load_2d(st + 2 * kHalf, &tm_min, 0, y, full_bar(s));
        tma_load_2d(st + 3 * kHalf, &tm_min, 64, y, full_bar(s));
        next_tile(a, cur);
      }
      for (int s = 0; s < kStages && s < n; ++s) {  // every copy lands before exit
        const int last = n - 1 - ((n - 1 - s) % kStages);
        mbar_drain(full_bar(s), (last / kStages) & 1);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      TileCursor cur = first;
      int n = 0, seg = 0;
      for (; n < count && !*abort_flag; ++n) {
        const int s = n % kStages, b = n & 1, qb = seg & 1;
        if ((n == 0 || cur.tile == 0) && !mbar_wait(q_full(qb), (seg >> 1) & 1, abort_flag)) break;
        if (!mbar_wait(full_bar(s), (n / kStages) & 1, abort_flag)) break;
        if (n >= 2 && !mbar_wait(acc_free(b), ((n >> 1) + 1) & 1, abort_flag)) break;
        tc_fence_after();
        bound::issue_mmas(tmem + b * 16, sbase + s * kStageBytes, sbase + kOffQ + qb * kQBytes);
        mma_commit(acc_full(b));
        mma_commit(empty_bar(s));
        next_tile(a, cur);
        if (n + 1 == count || cur.tile == 0) {  // the segment's last tile: its operand buffer is free after it
          mma_commit(q_free(qb));
          ++seg;
        }
      }
      if (n > 0) mbar_drain(acc_full((n - 1) & 1), ((n - 1) >> 1) & 1);
    }
  } else {
    // epilogue warps: Q operands and scores; a warp leaves the loop as a
    // whole (its TMEM loads are warp-wide) once a wait has run out or the CTA
    // is stopping
    const int t = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int g = a.group;
    // [Q+ | Q-] of a (request, kv head)
    auto write_q = [&](int pair, int b) {
      const int bq = pair / a.hkv, kvh = pair - bq * a.hkv;
      bound::write_q(smem + kOffQ + b * kQBytes, a.q, static_cast<int64_t>(bq) * a.hq + kvh * g, g, t);
    };
    TileCursor cur = first, qc = first;  // qc: first tile of the next segment whose operand is to be written
    int qleft = count, q_done = 0, seg = 0;
    bool more_q = count > 0;
    if (more_q) {
      write_q(qc.pair, 0);
      fence_async_smem();
      mbar_arrive(q_full(0));
      q_done = 1;
      more_q = next_segment(a, qc, qleft);
    }
    for (int n = 0; n < count; ++n) {
      bool ok = !*abort_flag;
      // the next segment's operand, once the MMAs of the segment before this one are done with its buffer
      if (more_q && q_done == seg + 1) {
        const int b1 = q_done & 1;
        ok = __all_sync(0xffffffffu, ok && (q_done < 2 || mbar_wait(q_free(b1), ((q_done - 2) >> 1) & 1, abort_flag)));
        if (ok) {
          write_q(qc.pair, b1);
          fence_async_smem();
          mbar_arrive(q_full(b1));
          ++q_done;
          more_q = next_segment(a, qc, qleft);
        }
      }
      const int b = n & 1;
      if (!__all_sync(0xffffffffu, ok && mbar_wait(acc_full(b), (n >> 1) & 1, abort_flag))) break;
      tc_fence_after();
      float u[16];
      tmem_ld16(tmem + lane_base + b * 16, u);
      tc_fence_before();
      mbar_arrive(acc_free(b));
      float best = -INFINITY;
#pragma unroll
      for (int h = 0; h < 16; ++h)
        if (h < g) best = fmaxf(best, u[h]);
      const int j = cur.tile * kTile + t;
      if (j < cur.nb) a.scores[static_cast<int64_t>(cur.pair) * a.max_blocks + j] = best;
      next_tile(a, cur);
      if (cur.tile == 0) ++seg;
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (FUSE) {
    // every CTA of the cluster has stored its tile's scores (the cluster
    // barrier orders those global stores before rank 0's loads); the ring's
    // shared memory is free again and holds the selection's work arrays
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    if (cluster.block_rank() == 0) {
      float* s_scores = reinterpret_cast<float*>(smem);  // <= 16 tiles x 128
      auto s_hist = reinterpret_cast<uint32_t(*)[sel::kHistWords]>(smem + 65536);  // 3 buffers
      int* s_warp = reinterpret_cast<int*>(smem + 65536 + 4096);                    // kThreads / 32
      uint32_t* s_range = reinterpret_cast<uint32_t*>(smem + 65536 + 4096 + 128);   // 2 per warp
      const int pair = blockIdx.x / a.tiles;
      const int b = pair / a.hkv;
      const int L = max(a.seq_lens[b], 0);
      int nb = (L + a.block - 1) / a.block;
      if (nb > a.max_blocks) {
        if (tid == 0) set_error(err, HS_EBIT_BLOCK_RANGE);
        nb = a.max_blocks;
      }
      const float* src = a.scores + static_cast<int64_t>(pair) * a.max_blocks;
      uint32_t lo = 0xffffffffu, hi = 0u;  // per warp: the range of the scored blocks' keys
      for (int j0 = 0; j0 < nb; j0 += kThreads) {
        const int j = j0 + tid;
        if (j < nb) {
          const float v = __ldcg(src + j);
          s_scores[j] = v;
          if (!sel::is_forced(j, L, a.block, sa.sink_tokens, sa.window_tokens)) {
            lo = min(lo, score_key(v));
            hi = max(hi, score_key(v));
          }
        }
      }
      lo = __reduce_min_sync(0xffffffffu, lo);
      hi = __reduce_max_sync(0xffffffffu, hi);
      if (lane == 0) {
        s_range[2 * warp] = lo;
        s_range[2 * warp + 1] = hi;
      }
      for (int i = tid; i < sel::kHistWords; i += kThreads) s_hist[0][i] = 0u;
      __syncthreads();
      const bool smoothed = sa.history_weight != 0.0f && sa.history != nullptr;  // the range no longer holds
      sel::smooth_scores(s_scores, nb, a.max_blocks, sa, pair);
      static_assert(kThreads * 6 >= 8 * kTile, "six blocks per thread cover up to 8 tiles");
      sel::select_pair_regs<kThreads, 6>(s_scores, nb, L, a.block, sa, pair, s_hist, s_warp, err, nullptr,
                                         smoothed ? nullptr : s_range, kThreads / 32, true);
    }
  }
  if (*abort_flag && tid == 0) report_timeout(err, kTimeoutScore, static_cast<unsigned>(abort_flag[2]));
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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

// summaries as [rows = pairs * max_blocks][128] bf16; box = 128 rows x 64 channels, 128-byte swizzle
bool make_map(CUtensorMap* m, const void* base, int64_t rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kTile)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool score_tc_supported(const KvView& kv) {
  if (kv.kv_dtype == HS_KV_F32 || kv.head_dim != kD || kv.group > 16) return false;
  const int64_t rows = static_cast<int64_t>(kv.batch) * kv.hkv * kv.max_blocks;
  if (rows >= (int64_t(1) << 31)) return false;
  return encode_fn() != nullptr;
}

bool score_select_fused_supported(const KvView& kv, int sms) {
  const int tiles = (kv.max_blocks + kTile - 1) / kTile;
  return score_tc_supported(kv) && tiles <= 8 && static_cast<int64_t>(kv.batch) * kv.hkv * tiles <= sms;
}

cudaError_t launch_score_tc(const KvView& kv, const void* q, const void* smin, const void* smax, float* scores,
                            int sms, unsigned* err, cudaStream_t st, const SelectArgs* fuse) {
  const int64_t rows = static_cast<int64_t>(kv.batch) * kv.hkv * kv.max_blocks;
  if (rows == 0) return cudaSuccess;
  CUtensorMap mmax, mmin;
  if (!make_map(&mmax, smax, rows) || !make_map(&mmin, smin, rows)) return cudaErrorInvalidValue;
  ScoreArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.seq_lens = kv.seq_lens;
  a.scores = scores;
  a.hkv = kv.hkv;
  a.hq = kv.hq;
  a.group = kv.group;
  a.block = kv.block;
  a.max_blocks = kv.max_blocks;
  a.batch = kv.batch;
  a.tiles = (kv.max_blocks + kTile - 1) / kTile;
  a.items = kv.batch * kv.hkv * a.tiles;
  if (!fuse) {
    cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
    if (e != cudaSuccess) return e;
    const int grid = a.items < sms ? a.items : sms;
    return launch_pdl(score_tc_kernel<false>, dim3(grid), dim3(kThreads), kAlloc, st, mmax, mmin, a, SelectArgs{},
                      err);
  }
  // one cluster of a.tiles CTAs per (request, kv head), one CTA per tile
  cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.items);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.tiles;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, score_tc_kernel<true>, mmax, mmin, a, *fuse, err);
}

}  // namespace hs
