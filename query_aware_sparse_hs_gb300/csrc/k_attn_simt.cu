// CUDA-core gather-attention over the selected blocks, split-K, plus the
// log-sum-exp merge of the splits ("KV 稀疏化" wiki §5: full attention on the
// chosen blocks only; "分块稀疏注意力与KV Cache量化" §2.2: running max and
// normaliser carried across tiles).
//
// This path serves every K/V dtype (it is the fp32 path; bf16 and e4m3 normally
// run on the tensor-core kernel).  CTA = (split, kv head, request), 4 warps;
// each warp walks tokens of the CTA's blocks, each lane owning D/32 channels,
// and keeps an online softmax per query head of the group.  The 4 warps' states
// are combined in shared memory and written as one normalised partial
// (o, lse) per query head and split.
#include "hs_internal.h"

namespace hs {
namespace {

constexpr int kWarps = 4;

template <int C, int KIND>
__device__ __forceinline__ void load_row(const void* pages, const float* scales, int64_t row,
                                         int D, int d0, float (&x)[C]) {
  if constexpr (KIND == HS_KV_F32) {
    const float* p = static_cast<const float*>(pages) + row * D + d0;
#pragma unroll
    for (int c = 0; c < C; ++c) x[c] = __ldg(p + c);
  } else if constexpr (KIND == HS_KV_BF16) {
    const uint16_t* p = static_cast<const uint16_t*>(pages) + row * D + d0;
#pragma unroll
    for (int c = 0; c < C; ++c) x[c] = bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(p + c)));
  } else {
    const uint8_t* p = static_cast<const uint8_t*>(pages) + row * D + d0;
    const float s = __ldg(scales + row * (D / kQuantGroup) + d0 / kQuantGroup);
#pragma unroll
    for (int c = 0; c < C; c += 2) {
      const uint16_t two = static_cast<uint16_t>(__ldg(p + c)) | (static_cast<uint16_t>(__ldg(p + c + 1)) << 8);
      float2 f = e4m3x2_to_float2(two);
      x[c] = f.x * s;
      x[c + 1] = f.y * s;
    }
  }
}

template <int C, int G, int KIND>
__global__ __launch_bounds__(kWarps * 32) void attn_simt_kernel(KvView kv, AttnArgs a,
                                                                unsigned* err) {
  constexpr int D = C * 32;
  pdl_trigger();
  pdl_wait();
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = kv.block;
  const int64_t pair = static_cast<int64_t>(b) * kv.hkv + kvh;
  int cnt = a.sel_count[pair];
  if (cnt > a.capacity) {
    if (threadIdx.x == 0 && split == 0) set_error(err, HS_EBIT_CAPACITY);
    cnt = a.capacity;
  }
  const int s0 = split * a.blocks_per_split;
  const int s1 = min(cnt, s0 + a.blocks_per_split);
  const int L = kv.seq_lens[b];
  const int nb = min(ceil_div(max(L, 0), B), kv.max_blocks);

  float qf[G][C];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int64_t qo = (static_cast<int64_t>(b) * kv.hq + kvh * G + h) * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; ++c)
      qf[h][c] = (KIND == HS_KV_F32) ? static_cast<const float*>(a.q)[qo + c]
                                     : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[qo + c]);
  }
  float m[G], l[G], o[G][C];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int c = 0; c < C; ++c) o[h][c] = 0.0f;
  }

  for (int i = s0; i < s1; ++i) {
    const int j = a.sel[pair * a.capacity + i];
    if (j < 0 || j >= nb) {
      if (threadIdx.x == 0) set_error(err, HS_EBIT_BLOCK_RANGE);
      continue;
    }
    const int page = kv.page_table[pair * kv.max_blocks + j];
    if (page < 0 || page >= kv.num_pages) {
      if (threadIdx.x == 0) set_error(err, HS_EBIT_PAGE_RANGE);
      continue;
    }
    const int valid = min(B, L - j * B);
    const int64_t row0 = static_cast<int64_t>(page) * B;
    for (int t = warp; t < valid; t += kWarps) {
      float kx[C], vx[C];
      load_row<C, KIND>(kv.k_pages, kv.k_scales, row0 + t, D, lane * C, kx);
      load_row<C, KIND>(kv.v_pages, kv.v_scales, row0 + t, D, lane * C, vx);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float dot = 0.0f;
#pragma unroll
        for (int c = 0; c < C; ++c) dot = fmaf(qf[h][c], kx[c], dot);
        const float s = warp_sum(dot) * a.scale;
        const float mn = fmaxf(m[h], s);
        const float alpha = expf(m[h] - mn);
        const float p = expf(s - mn);
        l[h] = fmaf(l[h], alpha, p);
#pragma unroll
        for (int c = 0; c < C; ++c) o[h][c] = fmaf(p, vx[c], o[h][c] * alpha);
        m[h] = mn;
      }
    }
  }

  __shared__ float sm_m[kWarps][G], sm_l[kWarps][G];
  __shared__ float sm_o[kWarps][G][D];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (lane == 0) {
      sm_m[warp][h] = m[h];
      sm_l[warp][h] = l[h];
    }
#pragma unroll
    for (int c = 0; c < C; ++c) sm_o[warp][h][lane * C + c] = o[h][c];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += kWarps * 32) {
    const int h = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][h]);
    float ov = 0.0f, lse = -INFINITY;
    if (M != -INFINITY) {
      float lsum = 0.0f, osum = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float e = expf(sm_m[w][h] - M);
        lsum = fmaf(sm_l[w][h], e, lsum);
        osum = fmaf(sm_o[w][h][d], e, osum);
      }
      ov = osum / lsum;
      lse = M + logf(lsum);
    }
    const int64_t row = (static_cast<int64_t>(b) * kv.hq + kvh * G + h) * a.splits + split;
    a.ws_o[row * D + d] = ov;
    if (d == 0) a.ws_lse[row] = lse;
  }
}

template <int C, int KIND>
cudaError_t launch_g(const KvView& kv, const AttnArgs& a, unsigned* err, cudaStream_t st) {
  dim3 grid(a.splits, kv.hkv, kv.batch);
  dim3 block(kWarps * 32);
  switch (kv.group) {
    case 1: return launch_pdl(attn_simt_kernel<C, 1, KIND>, grid, block, 0, st, kv, a, err);
    case 2: return launch_pdl(attn_simt_kernel<C, 2, KIND>, grid, block, 0, st, kv, a, err);
    case 4: return launch_pdl(attn_simt_kernel<C, 4, KIND>, grid, block, 0, st, kv, a, err);
    case 8: return launch_pdl(attn_simt_kernel<C, 8, KIND>, grid, block, 0, st, kv, a, err);
    default: return launch_pdl(attn_simt_kernel<C, 16, KIND>, grid, block, 0, st, kv, a, err);
  }
  return cudaGetLastError();
}

template <int C>
cudaError_t launch_c(const KvView& kv, const AttnArgs& a, unsigned* err, cudaStream_t st) {
  switch (kv.kv_dtype) {
    case HS_KV_F32: return launch_g<C, HS_KV_F32>(kv, a, err, st);
    case HS_KV_BF16: return launch_g<C, HS_KV_BF16>(kv, a, err, st);
    default: return launch_g<C, HS_KV_FP8E4M3_G32>(kv, a, err, st);
  }
}

// Log-sum-exp merge of attention partials over disjoint token sets ("分块稀疏
// 注意力与KV Cache量化" §2.2: running max and normaliser): with m = max_i lse_i,
// out = sum_i e^(lse_i - m) o_i / sum_i e^(lse_i - m), lse = m + log of the sum.
// Partial i of row r sits at o[r * o_row + i * o_part], lse[r * l_row + i * l_part].
// One warp per (request, query head) row; lane owns C = D/32 consecutive channels.
constexpr int kMergeWarps = 8;

template <int C>
__global__ __launch_bounds__(kMergeWarps * 32) void merge_kernel(int rows, int parts, const float* __restrict__ o,
                                                                 const float* __restrict__ lse, int64_t o_row,
                                                                 int64_t o_part, int64_t l_row, int64_t l_part,
                                                                 void* out, int out_f32, float* lse_out) {
  constexpr int D = C * 32;
  pdl_trigger();
  pdl_wait();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  float M = -INFINITY;
  for (int i = 0; i < parts; ++i) M = fmaxf(M, lse[row * l_row + i * l_part]);
  float acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.0f;
  float lse_v = -INFINITY;
  if (M != -INFINITY) {
    float tot = 0.0f;
    for (int i = 0; i < parts; ++i) {
      const float w = expf(lse[row * l_row + i * l_part] - M);
      tot += w;
      if (w > 0.0f) {
        const float* src = o + row * o_row + i * o_part + lane * C;
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] = fmaf(w, src[c], acc[c]);
      }
    }
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = acc[c] / tot;
    lse_v = M + logf(tot);
  }
  if (out_f32) {
    float* dst = static_cast<float*>(out) + row * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; ++c) dst[c] = acc[c];
  } else {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(out) + row * D + lane * C;
#pragma unroll
    for (int c = 0; c < C; ++c) dst[c] = __float2bfloat16_rn(acc[c]);
  }
  if (lse_out && lane == 0) lse_out[row] = lse_v;
}

cudaError_t launch_merge_rows(int rows, int head_dim, int parts, const float* o, const float* lse, int64_t o_row,
                              int64_t o_part, int64_t l_row, int64_t l_part, void* out, int out_f32,
                              float* lse_out, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const dim3 grid((rows + kMergeWarps - 1) / kMergeWarps);
  if (head_dim == 128)
    return launch_pdl(merge_kernel<4>, grid, dim3(kMergeWarps * 32), 0, st, rows, parts, o, lse, o_row, o_part,
                      l_row, l_part, out, out_f32, lse_out);
  return launch_pdl(merge_kernel<2>, grid, dim3(kMergeWarps * 32), 0, st, rows, parts, o, lse, o_row, o_part, l_row,
                    l_part, out, out_f32, lse_out);
}

}  // namespace

cudaError_t launch_attn_simt(const KvView& kv, const AttnArgs& a, unsigned* err, cudaStream_t st) {
  if (kv.batch == 0 || kv.hkv == 0) return cudaSuccess;
  return kv.head_dim == 128 ? launch_c<4>(kv, a, err, st) : launch_c<2>(kv, a, err, st);
}

cudaError_t launch_merge(const KvView& kv, const AttnArgs& a, cudaStream_t st) {
  const int64_t D = kv.head_dim, S = a.splits;
  return launch_merge_rows(kv.batch * kv.hq, kv.head_dim, a.splits, static_cast<const float*>(a.ws_o),
                           static_cast<const float*>(a.ws_lse), S * D, D, S, int64_t(1), a.out, a.out_is_fp32,
                           a.lse, st);
}

cudaError_t launch_merge_parts(int rows, int head_dim, int parts, const float* outs, const float* lses, void* out,
                               int out_f32, float* lse_out, cudaStream_t st) {
  // A plain launch: the parts usually come from kernels on two streams, and the
  // merge must wait for all of them, not only for the last kernel of its own
  // stream.
  if (rows == 0) return cudaSuccess;
  const int64_t D = head_dim, R = rows;
  const dim3 grid((rows + kMergeWarps - 1) / kMergeWarps);
  if (head_dim == 128)
    merge_kernel<4><<<grid, kMergeWarps * 32, 0, st>>>(rows, parts, outs, lses, D, R * D, int64_t(1), R, out, out_f32,
                                                         lse_out);
  else
    merge_kernel<2><<<grid, kMergeWarps * 32, 0, st>>>(rows, parts, outs, lses, D, R * D, int64_t(1), R, out, out_f32,
                                                         lse_out);
  return cudaGetLastError();
}

}  // namespace hs
