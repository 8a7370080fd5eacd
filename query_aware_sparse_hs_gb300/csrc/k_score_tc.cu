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
static_assert(kOffMisc + 16 + 1024 <= kAlloc, "shared memory layout too large");
constexpr int kTmemCols = 32;

struct ScoreArgs {
  const __nv_bfloat16* q;
  const int32_t* seq_lens;
  float* scores;
  int hkv, hq, group, block, max_blocks, tiles, items;
};

// tile `tile` of (request, kv head) `pair` holds blocks [tile*128, tile*128+128): valid if any is < N_b
__device__ __forceinline__ bool tile_valid(const ScoreArgs& a, int item, int* pair, int* tile, int* nb) {
  *pair = item / a.tiles;
  *tile = item - *pair * a.tiles;
  const int b = *pair / a.hkv;
  const int L = max(a.seq_lens[b], 0);
  *nb = min((L + a.block - 1) / a.block, a.max_blocks);
  return *tile * kTile < *nb;
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
    *abort_flag = 0;
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

  if (warp == kProducerWarp) {
    if (lane == 0) {
      int n = 0;
      for (int item = blockIdx.x; item < a.items && !*abort_flag; item += gridDim.x) {
        int pair, tile, nb;
        if (!tile_valid(a, item, &pair, &tile, &nb)) continue;
        const int s = n % kStages;
        if (n >= kStages && !mbar_wait(empty_bar(s), ((n / kStages) + 1) & 1, abort_flag)) break;
        mbar_arrive_tx(full_bar(s), 4u * kHalf);
        const int y = pair * a.max_blocks + tile * kTile;
        const uint32_t st = sbase + s * kStageBytes;
        tma_load_2d(st, &tm_max, 0, y, full_bar(s));
        tma_load_2d(st + kHalf, &tm_max, 64, y, full_bar(s));
        tma_load_2d(st + 2 * kHalf, &tm_min, 0, y, full_bar(s));
        tma_load_2d(st + 3 * kHalf, &tm_min, 64, y, full_bar(s));
        ++n;
      }
      for (int s = 0; s < kStages && s < n; ++s) {  // every copy lands before exit
        const int last = n - 1 - ((n - 1 - s) % kStages);
        mbar_wait(full_bar(s), (last / kStages) & 1, abort_flag, 500000000ull);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      int n = 0;
      for (int item = blockIdx.x; item < a.items && !*abort_flag; item += gridDim.x) {
        int pair, tile, nb;
        if (!tile_valid(a, item, &pair, &tile, &nb)) continue;
        const int s = n % kStages, b = n & 1;
        if (!mbar_wait(q_full(b), (n >> 1) & 1, abort_flag)) break;
        if (!mbar_wait(full_bar(s), (n / kStages) & 1, abort_flag)) break;
        if (n >= 2 && !mbar_wait(acc_free(b), ((n >> 1) + 1) & 1, abort_flag)) break;
        tc_fence_after();
        bound::issue_mmas(tmem + b * 16, sbase + s * kStageBytes, sbase + kOffQ + b * kQBytes);
        mma_commit(acc_full(b));
        mma_commit(empty_bar(s));
        mma_commit(q_free(b));
        ++n;
      }
      if (n > 0) mbar_wait(acc_full((n - 1) & 1), ((n - 1) >> 1) & 1, abort_flag, 500000000ull);
    }
  } else {
    // epilogue warps: Q operands and scores
    const int t = tid;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int g = a.group;
    // [Q+ | Q-] of a (request, kv head)
    auto write_q = [&](int pair, int b) {
      const int bq = pair / a.hkv, kvh = pair - bq * a.hkv;
      bound::write_q(smem + kOffQ + b * kQBytes, a.q, static_cast<int64_t>(bq) * a.hq + kvh * g, g, t);
    };
    int n = 0;
    int item = blockIdx.x;
    int pair = 0, tile = 0, nb = 0;
    while (item < a.items && !tile_valid(a, item, &pair, &tile, &nb)) item += gridDim.x;
    if (item < a.items) {
      write_q(pair, 0);
      fence_async_smem();
      mbar_arrive(q_full(0));
    }
    while (item < a.items && !*abort_flag) {
      // the next tile's operand is written while this tile is in flight
      int nitem = item + gridDim.x, npair = 0, ntile = 0, nnb = 0;
      while (nitem < a.items && !tile_valid(a, nitem, &npair, &ntile, &nnb)) nitem += gridDim.x;
      if (nitem < a.items) {
        const int b1 = (n + 1) & 1;
        if (n + 1 >= 2 && !mbar_wait(q_free(b1), (((n + 1) >> 1) + 1) & 1, abort_flag)) break;
        write_q(npair, b1);
        fence_async_smem();
        mbar_arrive(q_full(b1));
      }
      const int b = n & 1;
      if (!mbar_wait(acc_full(b), (n >> 1) & 1, abort_flag)) break;
      tc_fence_after();
      float u[16];
      tmem_ld16(tmem + lane_base + b * 16, u);
      tc_fence_before();
      mbar_arrive(acc_free(b));
      float best = -INFINITY;
#pragma unroll
      for (int h = 0; h < 16; ++h)
        if (h < g) best = fmaxf(best, u[h]);
      const int j = tile * kTile + t;
      if (j < nb) a.scores[static_cast<int64_t>(pair) * a.max_blocks + j] = best;
      item = nitem;
      pair = npair;
      tile = ntile;
      nb = nnb;
      ++n;
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
      uint32_t lo = 0xffffffffu, hi = 0u;  // per warp: the range of the keys
      for (int j0 = 0; j0 < nb; j0 += kThreads) {
        const int j = j0 + tid;
        if (j < nb) {
          const float v = __ldcg(src + j);
          s_scores[j] = v;
          lo = min(lo, score_key(v));
          hi = max(hi, score_key(v));
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
  if (*abort_flag && tid == 0) set_error(err, HS_EBIT_TIMEOUT);
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
