// Grouped e4m3 quantisation of K/V rows ("分块稀疏注意力与KV Cache量化" §2.4:
// channels split into groups with one scale each; §3.2: group size 32).
// One warp per row; lane owns C = D/32 consecutive channels, so a 32-channel
// group spans 32/C lanes and its amax is a shuffle reduction inside them.
#include "hs_internal.h"

namespace hs {
namespace {

constexpr int kWarps = 8;

template <int C, bool F32>
__global__ __launch_bounds__(kWarps * 32) void quant_kernel(const void* __restrict__ src, int64_t rows,
                                                           uint8_t* __restrict__ codes,
                                                           float* __restrict__ scales) {
  constexpr int D = C * 32;
  constexpr int kLanesPerGroup = kQuantGroup / C;
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  float x[C];
  if constexpr (F32) {
    const float* p = static_cast<const float*>(src) + row * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; ++c) x[c] = p[c];
  } else {
    const uint16_t* p = static_cast<const uint16_t*>(src) + row * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; ++c) x[c] = bf16_bits_to_float(p[c]);
  }
  uint8_t out[C];
  const float scale = quantize_e4m3_lane<C>(x, out);
  uint8_t* q = codes + row * D + lane * C;
#pragma unroll
  for (int c = 0; c < C; ++c) q[c] = out[c];
  if ((lane % kLanesPerGroup) == 0) scales[row * (D / kQuantGroup) + lane / kLanesPerGroup] = scale;
}

template <int C>
cudaError_t launch_c(const void* src, bool f32, int64_t rows, uint8_t* codes, float* scales,
                     cudaStream_t st) {
  const int64_t grid = (rows + kWarps - 1) / kWarps;
  if (f32)
    quant_kernel<C, true><<<static_cast<unsigned>(grid), kWarps * 32, 0, st>>>(src, rows, codes, scales);
  else
    quant_kernel<C, false><<<static_cast<unsigned>(grid), kWarps * 32, 0, st>>>(src, rows, codes, scales);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const void* src, bool src_f32, int64_t rows, int head_dim,
                            uint8_t* codes, float* scales, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  switch (head_dim) {
    case 64: return launch_c<2>(src, src_f32, rows, codes, scales, st);
    case 128: return launch_c<4>(src, src_f32, rows, codes, scales, st);
    case 256: return launch_c<8>(src, src_f32, rows, codes, scales, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hs
