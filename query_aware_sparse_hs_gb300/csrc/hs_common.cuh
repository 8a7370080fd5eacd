// Shared device helpers and the launch descriptors passed from the C-ABI layer
// to the kernels.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/hs.h"

namespace hs {

constexpr int kQuantGroup = 32;          // channels per e4m3 scale
constexpr int kMaxSelectBlocks = 16384;  // blocks per request the selector holds in smem
constexpr int kSelectCluster = 8;        // CTAs scoring one (request, kv head)

// Everything a kernel needs to address the paged cache of one call.
struct KvView {
  const void* k_pages;
  const void* v_pages;
  const float* k_scales;
  const float* v_scales;
  const int32_t* page_table;
  const int32_t* seq_lens;
  int64_t num_pages;
  int32_t batch;
  int32_t max_blocks;
  int32_t hq, hkv, group, head_dim, block;
  int32_t kv_dtype;
};

__device__ __forceinline__ void set_error(unsigned* err, unsigned bit) {
  if (err) atomicOr(err, bit);
}

// Kernels that can report a wait that ran out, for the record below.
enum TimeoutKernel : unsigned {
  kTimeoutAttnBf16 = 1,
  kTimeoutStepFused = 2,
  kTimeoutAttnE4m3 = 3,
  kTimeoutScore = 4,
};

// HS_EBIT_TIMEOUT plus, for the first CTA that reports one, a record of
// where: err[1] = kernel, err[2] = CTA index, err[3] = the wait (the word a
// bounded wait leaves next to the abort flag: barrier address, parity, warp),
// err[4..11] = the CTA's progress words (nullable: zeros).
constexpr int kErrorWords = 12;
__device__ __forceinline__ void report_timeout(unsigned* err, unsigned kernel, unsigned wait_info,
                                               const volatile int* progress = nullptr) {
  if (!err) return;
  atomicOr(err, HS_EBIT_TIMEOUT);
  if (atomicCAS(err + 1, 0u, kernel) == 0u) {
    err[2] = blockIdx.x;
    err[3] = wait_info;
    for (int i = 0; i < 8; ++i) err[4 + i] = progress ? static_cast<unsigned>(progress[i]) : 0u;
  }
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two e4m3 codes (low byte first) to two floats: the conversion is exact.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// fp32 score -> unsigned key whose integer order is the float order (-0 and +0
// are one key); NaN is mapped below every number (key 0).
__device__ __forceinline__ uint32_t score_key(float s) {
  if (isnan(s)) return 0u;
  uint32_t u = (s == 0.0f) ? 0u : __float_as_uint(s);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Grouped e4m3 quantisation of one row held C consecutive channels per lane
// ("分块稀疏注意力与KV Cache量化" §2.4 grouped scales, §3.2 group size 32):
// scale = amax of the 32-channel group / 448 (1 when the group is all zero),
// code = e4m3(x / scale), nearest-even, saturating.  All 32 lanes must call
// it.  Returns the lane's group scale.
template <int C>
__device__ __forceinline__ float quantize_e4m3_lane(const float (&x)[C], uint8_t (&out)[C]) {
  constexpr int kLanesPerGroup = kQuantGroup / C;
  float amax = 0.0f;
#pragma unroll
  for (int c = 0; c < C; ++c) amax = fmaxf(amax, fabsf(x[c]));
#pragma unroll
  for (int o = kLanesPerGroup / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;  // IEEE division
#pragma unroll
  for (int c = 0; c < C; c += 2) {
    float2 y = make_float2(x[c] / scale, x[c + 1] / scale);
    __nv_fp8x2_storage_t two = __nv_cvt_float2_to_fp8x2(y, __NV_SATFINITE, __NV_E4M3);
    out[c] = static_cast<uint8_t>(two & 0xff);
    out[c + 1] = static_cast<uint8_t>(two >> 8);
  }
  return scale;
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Programmatic dependent launch: every kernel of a step lets its successor be
// scheduled at once (trigger) and waits for its predecessor's results before it
// reads any input (wait).  Both are no-ops without a dependent launch.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets `kern` take `dynamic` bytes of dynamic shared memory where that plus
// its static shared memory passes the 48 KB a launch gets by default.
template <typename... KArgs>
cudaError_t allow_dynamic_smem(void (*kern)(KArgs...), size_t dynamic) {
  if (dynamic <= 16 * 1024) return cudaSuccess;  // no kernel here has 32 KB of static shared memory
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (dynamic + fa.sharedSizeBytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(dynamic));
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace hs
