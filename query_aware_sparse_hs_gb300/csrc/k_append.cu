// Append step of a decode loop: the newest token of every (request, kv head)
// stream, at position seq_lens[b] - 1, is written into its page, and the
// min/max summary of its block ("KV 稀疏化" wiki §5, Quest) is widened to
// cover it.  An e4m3 cache stores the token with the grouped quantisation of
// "分块稀疏注意力与KV Cache量化" §2.4/§3.2 and widens the summary by the
// dequantised values (code * scale in fp32), rounded outward to bf16.
// Rounding down (up) is monotone, so min(round_down(old box), round_down(x))
// equals round_down of the minimum over the block: the widened box is the box
// a full rebuild over the block gives.  A token in row 0 of its block starts
// the box afresh.
// One warp per stream; lane owns D/32 consecutive channels.  Latency-bound:
// 2 rows of D values in, 2 rows (+ scales) and 2 summary rows out per stream.
#include "hs_internal.h"

namespace hs {
namespace {

constexpr int kWarps = 4;

// C source values of this lane: f32 for an f32 cache, bf16 otherwise.
template <int C, bool F32>
__device__ __forceinline__ void load_src(const void* src, int64_t off, float (&x)[C]) {
  if constexpr (F32) {
    const float* p = static_cast<const float*>(src) + off;
#pragma unroll
    for (int c = 0; c < C; ++c) x[c] = p[c];
  } else {
    const uint16_t* p = static_cast<const uint16_t*>(src) + off;
#pragma unroll
    for (int c = 0; c < C; ++c) x[c] = bf16_bits_to_float(p[c]);
  }
}

// Stores the lane's channels of one token row into the cache and returns the
// values the cache now holds (e4m3: decoded code times the group scale).
template <int C, int KIND>
__device__ __forceinline__ void store_row(const void* pages, const float* scales, int64_t row, int lane,
                                          const float (&x)[C], float (&held)[C]) {
  constexpr int D = C * 32;
  if constexpr (KIND == HS_KV_F32) {
    float* p = static_cast<float*>(const_cast<void*>(pages)) + row * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      p[c] = x[c];
      held[c] = x[c];
    }
  } else if constexpr (KIND == HS_KV_BF16) {
    uint16_t* p = static_cast<uint16_t*>(const_cast<void*>(pages)) + row * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      p[c] = static_cast<uint16_t>(__float_as_uint(x[c]) >> 16);  // x is a bf16 value
      held[c] = x[c];
    }
  } else {
    constexpr int kLanesPerGroup = kQuantGroup / C;
    uint8_t code[C];
    const float s = quantize_e4m3_lane<C>(x, code);
    uint8_t* p = static_cast<uint8_t*>(const_cast<void*>(pages)) + row * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; c += 2) {
      p[c] = code[c];
      p[c + 1] = code[c + 1];
      const float2 v = e4m3x2_to_float2(static_cast<uint16_t>(code[c] | (code[c + 1] << 8)));
      held[c] = v.x * s;
      held[c + 1] = v.y * s;
    }
    if ((lane % kLanesPerGroup) == 0)
      const_cast<float*>(scales)[row * (D / kQuantGroup) + lane / kLanesPerGroup] = s;
  }
}

template <int C, int KIND>
__global__ __launch_bounds__(kWarps * 32) void append_kernel(KvView kv, const void* __restrict__ new_k,
                                                             const void* __restrict__ new_v, void* smin,
                                                             void* smax, unsigned* err) {
  constexpr int D = C * 32;
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (pair >= kv.batch * kv.hkv) return;
  const int b = pair / kv.hkv;
  const int L = kv.seq_lens[b];
  if (L <= 0) return;
  const int t = L - 1;
  const int j = t / kv.block;
  const int r = t - j * kv.block;
  if (j >= kv.max_blocks) {
    if (lane == 0) set_error(err, HS_EBIT_BLOCK_RANGE);
    return;
  }
  const int64_t page = kv.page_table[static_cast<int64_t>(pair) * kv.max_blocks + j];
  if (page < 0 || page >= kv.num_pages) {
    if (lane == 0) set_error(err, HS_EBIT_PAGE_RANGE);
    return;
  }
  const int64_t row = page * kv.block + r;
  const int64_t src = static_cast<int64_t>(pair) * D + lane * C;
  float x[C], held[C], unused[C];
  load_src<C, KIND == HS_KV_F32>(new_v, src, x);
  store_row<C, KIND>(kv.v_pages, kv.v_scales, row, lane, x, unused);
  load_src<C, KIND == HS_KV_F32>(new_k, src, x);
  store_row<C, KIND>(kv.k_pages, kv.k_scales, row, lane, x, held);

  const int64_t o = (static_cast<int64_t>(pair) * kv.max_blocks + j) * D + lane * C;
  if constexpr (KIND == HS_KV_F32) {
    float* mn = static_cast<float*>(smin) + o;
    float* mx = static_cast<float*>(smax) + o;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      mn[c] = r == 0 ? held[c] : fminf(mn[c], held[c]);
      mx[c] = r == 0 ? held[c] : fmaxf(mx[c], held[c]);
    }
  } else {
    __nv_bfloat16* mn = static_cast<__nv_bfloat16*>(smin) + o;
    __nv_bfloat16* mx = static_cast<__nv_bfloat16*>(smax) + o;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      // bf16 K: the value is a bf16 already; e4m3 K: round outward
      const float lo = KIND == HS_KV_BF16 ? held[c] : __bfloat162float(__float2bfloat16_rd(held[c]));
      const float hi = KIND == HS_KV_BF16 ? held[c] : __bfloat162float(__float2bfloat16_ru(held[c]));
      const float a = r == 0 ? lo : fminf(__bfloat162float(mn[c]), lo);
      const float z = r == 0 ? hi : fmaxf(__bfloat162float(mx[c]), hi);
      mn[c] = __float2bfloat16_rn(a);  // exact: a and z are bf16 values
      mx[c] = __float2bfloat16_rn(z);
    }
  }
}

template <int C>
cudaError_t launch_c(const KvView& kv, const void* new_k, const void* new_v, void* smin, void* smax,
                     unsigned* err, cudaStream_t st) {
  const dim3 grid(ceil_div(kv.batch * kv.hkv, kWarps));
  switch (kv.kv_dtype) {
    case HS_KV_F32:
      return launch_pdl(append_kernel<C, HS_KV_F32>, grid, dim3(kWarps * 32), 0, st, kv, new_k, new_v, smin, smax, err);
    case HS_KV_BF16:
      return launch_pdl(append_kernel<C, HS_KV_BF16>, grid, dim3(kWarps * 32), 0, st, kv, new_k, new_v, smin, smax, err);
    default:
      return launch_pdl(append_kernel<C, HS_KV_FP8E4M3_G32>, grid, dim3(kWarps * 32), 0, st, kv, new_k, new_v, smin,
                        smax, err);
  }
}

}  // namespace

cudaError_t launch_append(const KvView& kv, const void* new_k, const void* new_v, void* smin, void* smax,
                          unsigned* err, cudaStream_t st) {
  if (kv.batch == 0) return cudaSuccess;
  return kv.head_dim == 128 ? launch_c<4>(kv, new_k, new_v, smin, smax, err, st)
                            : launch_c<2>(kv, new_k, new_v, smin, smax, err, st);
}

}  // namespace hs
