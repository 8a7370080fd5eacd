// Per-block key summaries (Quest, "KV 稀疏化" wiki §5): channel-wise min and
// max of K over each block's valid tokens.  Each lane owns D/32 consecutive
// channels, so every token row is one coalesced warp load.  HBM-bound: one pass
// over the K pages of the blocks asked for.
#include "hs_internal.h"

namespace hs {
namespace {

template <int C, int KIND>
struct RowLoad;

// fp32 K
template <int C>
struct RowLoad<C, HS_KV_F32> {
  static __device__ __forceinline__ void get(const KvView& kv, int64_t row, int d0, float (&x)[C]) {
    const float* p = static_cast<const float*>(kv.k_pages) + row * kv.head_dim + d0;
    if constexpr (C == 4) {
      float4 v = __ldg(reinterpret_cast<const float4*>(p));
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
      float2 v = __ldg(reinterpret_cast<const float2*>(p));
      x[0] = v.x; x[1] = v.y;
    }
  }
};

// bf16 K
template <int C>
struct RowLoad<C, HS_KV_BF16> {
  static __device__ __forceinline__ void get(const KvView& kv, int64_t row, int d0, float (&x)[C]) {
    const uint16_t* p = static_cast<const uint16_t*>(kv.k_pages) + row * kv.head_dim + d0;
    if constexpr (C == 4) {
      uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
      x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xffff0000u);
      x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xffff0000u);
    } else {
      uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(p));
      x[0] = __uint_as_float(v << 16); x[1] = __uint_as_float(v & 0xffff0000u);
    }
  }
};

// e4m3 K: code value times the token's 32-channel group scale, in fp32
template <int C>
struct RowLoad<C, HS_KV_FP8E4M3_G32> {
  static __device__ __forceinline__ void get(const KvView& kv, int64_t row, int d0, float (&x)[C]) {
    const uint8_t* p = static_cast<const uint8_t*>(kv.k_pages) + row * kv.head_dim + d0;
    const float s = __ldg(kv.k_scales + row * (kv.head_dim / kQuantGroup) + d0 / kQuantGroup);
    if constexpr (C == 4) {
      uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(p));
      float2 a = e4m3x2_to_float2(static_cast<uint16_t>(v & 0xffffu));
      float2 b = e4m3x2_to_float2(static_cast<uint16_t>(v >> 16));
      x[0] = a.x * s; x[1] = a.y * s; x[2] = b.x * s; x[3] = b.y * s;
    } else {
      uint16_t v = __ldg(reinterpret_cast<const unsigned short*>(p));
      float2 a = e4m3x2_to_float2(v);
      x[0] = a.x * s; x[1] = a.y * s;
    }
  }
};

constexpr int kWarps = 8;
constexpr int kRowsPerRound = 8;  // rows a warp has in flight

// Warps per block: enough that each warp reads about 8 rows (B/8, from 1 to
// 8); a CTA of 8 warps therefore covers 8 / wpb blocks.  Each warp loads all
// the rows of a round before using any, so a block costs about one memory
// latency; the warps' partial boxes are combined in shared memory.
__host__ __device__ __forceinline__ int warps_per_block(int B) { return B >= 64 ? 8 : (B >= 8 ? B / 8 : 1); }

template <int C, int KIND>
__global__ __launch_bounds__(kWarps * 32) void summaries_kernel(KvView kv, int first_block,
                                                               void* smin, void* smax,
                                                               unsigned* err) {
  constexpr int D = C * 32;
  __shared__ float s_mn[kWarps][D], s_mx[kWarps][D];
  __shared__ int s_ok[kWarps];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int B = kv.block;
  const int wpb = warps_per_block(B), per_cta = kWarps / wpb;
  const int j = first_block + blockIdx.x * per_cta + warp / wpb;
  const int sub = warp % wpb;
  const int L = kv.seq_lens[b];
  const int nb = min(ceil_div(max(L, 0), B), kv.max_blocks);
  const int64_t pair = static_cast<int64_t>(b) * kv.hkv + kvh;
  const int d0 = lane * C;
  float mn[C], mx[C];
#pragma unroll
  for (int c = 0; c < C; ++c) { mn[c] = INFINITY; mx[c] = -INFINITY; }
  bool ok = j < nb;
  if (ok) {
    const int page = kv.page_table[pair * kv.max_blocks + j];
    if (page < 0 || page >= kv.num_pages) {
      if (lane == 0 && sub == 0) set_error(err, HS_EBIT_PAGE_RANGE);
      ok = false;
    } else {
      const int valid = min(B, L - j * B);
      const int64_t row0 = static_cast<int64_t>(page) * B;
      for (int t0 = sub; t0 < valid; t0 += wpb * kRowsPerRound) {
        float x[kRowsPerRound][C];
#pragma unroll
        for (int u = 0; u < kRowsPerRound; ++u) {
          const int t = min(t0 + u * wpb, valid - 1);  // clamp: a repeated valid row changes nothing
          RowLoad<C, KIND>::get(kv, row0 + t, d0, x[u]);
        }
#pragma unroll
        for (int u = 0; u < kRowsPerRound; ++u)
#pragma unroll
          for (int c = 0; c < C; ++c) { mn[c] = fminf(mn[c], x[u][c]); mx[c] = fmaxf(mx[c], x[u][c]); }
      }
    }
  }
#pragma unroll
  for (int c = 0; c < C; ++c) { s_mn[warp][d0 + c] = mn[c]; s_mx[warp][d0 + c] = mx[c]; }
  if (lane == 0) s_ok[warp] = ok ? 1 : 0;
  __syncthreads();
  for (int idx = threadIdx.x; idx < per_cta * D; idx += kWarps * 32) {
    const int bl = idx / D, d = idx - bl * D;
    const int w0 = bl * wpb;
    if (!s_ok[w0]) continue;
    float lo = s_mn[w0][d], hi = s_mx[w0][d];
    for (int w = 1; w < wpb; ++w) { lo = fminf(lo, s_mn[w0 + w][d]); hi = fmaxf(hi, s_mx[w0 + w][d]); }
    const int64_t o = (pair * kv.max_blocks + first_block + blockIdx.x * per_cta + bl) * D + d;
    if constexpr (KIND == HS_KV_F32) {
      static_cast<float*>(smin)[o] = lo;
      static_cast<float*>(smax)[o] = hi;
    } else {
      // bf16 K: min/max are bf16 values, the conversion is exact.  e4m3 K:
      // round outward so the stored box still contains every dequantised key.
      static_cast<__nv_bfloat16*>(smin)[o] = (KIND == HS_KV_BF16) ? __float2bfloat16_rn(lo) : __float2bfloat16_rd(lo);
      static_cast<__nv_bfloat16*>(smax)[o] = (KIND == HS_KV_BF16) ? __float2bfloat16_rn(hi) : __float2bfloat16_ru(hi);
    }
  }
}

template <int C>
cudaError_t launch_c(const KvView& kv, int first_block, int nblocks, void* smin, void* smax,
                     unsigned* err, cudaStream_t st) {
  const int per_cta = kWarps / warps_per_block(kv.block);
  dim3 grid(ceil_div(nblocks, per_cta), kv.hkv, kv.batch);
  switch (kv.kv_dtype) {
    case HS_KV_F32:
      return launch_pdl(summaries_kernel<C, HS_KV_F32>, grid, dim3(kWarps * 32), 0, st, kv, first_block, smin, smax, err);
    case HS_KV_BF16:
      return launch_pdl(summaries_kernel<C, HS_KV_BF16>, grid, dim3(kWarps * 32), 0, st, kv, first_block, smin, smax, err);
    default:
      return launch_pdl(summaries_kernel<C, HS_KV_FP8E4M3_G32>, grid, dim3(kWarps * 32), 0, st, kv, first_block, smin, smax, err);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_summaries(const KvView& kv, int first_block, void* smin, void* smax,
                             unsigned* err, cudaStream_t st) {
  const int nblocks = kv.max_blocks - first_block;
  if (nblocks <= 0 || kv.batch == 0) return cudaSuccess;
  return kv.head_dim == 128 ? launch_c<4>(kv, first_block, nblocks, smin, smax, err, st)
                            : launch_c<2>(kv, first_block, nblocks, smin, smax, err, st);
}

}  // namespace hs
