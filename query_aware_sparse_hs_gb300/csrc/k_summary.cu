// Per-block key summaries (Quest, "KV 稀疏化" wiki §5): channel-wise min and
// max of K over each block's valid tokens.  Each lane owns 16 bytes of
// consecutive channels of a row, so one warp load reads whole consecutive
// rows.  HBM-bound: one pass over the K pages of the blocks asked for.
#include "hs_internal.h"

namespace hs {
namespace {

// Each lane loads 16 bytes of a row (V channels), so a warp load covers RPL
// consecutive rows of the page - one contiguous 512-byte span - and a lane
// keeps U loads in flight before it uses any.
template <int KIND>
struct Elem;
template <>
struct Elem<HS_KV_F32> { static constexpr int kBytes = 4; };
template <>
struct Elem<HS_KV_BF16> { static constexpr int kBytes = 2; };
template <>
struct Elem<HS_KV_FP8E4M3_G32> { static constexpr int kBytes = 1; };

// 16 bytes of one row -> min/max of its V channels into mn/mx
template <int KIND, int V>
__device__ __forceinline__ void fold(const uint4& raw, float s, float (&mn)[V], float (&mx)[V]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  if constexpr (KIND == HS_KV_F32) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float x = __uint_as_float(w[c]);
      mn[c] = fminf(mn[c], x); mx[c] = fmaxf(mx[c], x);
    }
  } else if constexpr (KIND == HS_KV_BF16) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float lo = __uint_as_float(w[c] << 16), hi = __uint_as_float(w[c] & 0xffff0000u);
      mn[2 * c] = fminf(mn[2 * c], lo); mx[2 * c] = fmaxf(mx[2 * c], lo);
      mn[2 * c + 1] = fminf(mn[2 * c + 1], hi); mx[2 * c + 1] = fmaxf(mx[2 * c + 1], hi);
    }
  } else {
    // e4m3 K: code value times the token's 32-channel group scale, in fp32
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float2 x = e4m3x2_to_float2(static_cast<uint16_t>(w[c >> 1] >> (16 * (c & 1))));
      const float a = x.x * s, b = x.y * s;
      mn[2 * c] = fminf(mn[2 * c], a); mx[2 * c] = fmaxf(mx[2 * c], a);
      mn[2 * c + 1] = fminf(mn[2 * c + 1], b); mx[2 * c + 1] = fmaxf(mx[2 * c + 1], b);
    }
  }
}

constexpr int kWarps = 8;

// Warps per block: enough that each warp reads about one round of R rows per
// block (from 1 to 8); a CTA of 8 warps covers 8 / wpb blocks, and the warps'
// partial boxes are combined in shared memory.
__host__ __device__ __forceinline__ int warps_per_block(int B, int R) { return B >= 8 * R ? 8 : (B >= R ? B / R : 1); }

// rows in flight per lane: up to 8, no more than a block holds per warp load
__host__ __forceinline__ int rounds_for(int B, int rpl) {
  const int r = ceil_div(B, rpl);
  return r >= 8 ? 8 : (r >= 4 ? 4 : (r >= 2 ? 2 : 1));
}

// Persistent: CTA x takes block groups x, x + gridDim.x, ... of the flattened
// (request, kv head, group of per_cta blocks) space; groups past a request's
// blocks are skipped without work (requests of very different lengths would
// otherwise launch most CTAs for nothing).
template <int D, int KIND, int U>
__global__ __launch_bounds__(kWarps * 32) void summaries_kernel(KvView kv, int first_block, int groups_per_pair,
                                                               int64_t total_groups, void* smin, void* smax,
                                                               unsigned* err) {
  constexpr int E = Elem<KIND>::kBytes, V = 16 / E, LPR = D / V, RPL = 32 / LPR, R = RPL * U;
  static_assert(D % V == 0 && 32 % LPR == 0, "a row is a whole number of 16-byte lanes");
  __shared__ float s_mn[kWarps][D], s_mx[kWarps][D];
  __shared__ int s_ok[kWarps];
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rs = lane / LPR, d0 = (lane % LPR) * V;
  const int B = kv.block;
  const int wpb = warps_per_block(B, R), per_cta = kWarps / wpb;
  const int bl = warp / wpb, sub = warp % wpb;
  for (int64_t gi = blockIdx.x; gi < total_groups; gi += gridDim.x) {
    const int64_t pair = gi / groups_per_pair;
    const int grp = static_cast<int>(gi - pair * groups_per_pair);
    const int b = static_cast<int>(pair / kv.hkv);
    const int L = kv.seq_lens[b];
    const int nb = min(ceil_div(max(L, 0), B), kv.max_blocks);
    const int jg = first_block + grp * per_cta;  // the group's first block
    if (jg >= nb) continue;  // the same for every thread of the CTA
    const int j = jg + bl;
    float mn[V], mx[V];
#pragma unroll
    for (int c = 0; c < V; ++c) { mn[c] = INFINITY; mx[c] = -INFINITY; }
    bool ok = bl < per_cta && j < nb;
    if (ok) {
      const int page = kv.page_table[pair * kv.max_blocks + j];
      if (page < 0 || page >= kv.num_pages) {
        if (lane == 0 && sub == 0) set_error(err, HS_EBIT_PAGE_RANGE);
        ok = false;
      } else {
        const int valid = min(B, L - j * B);
        const int64_t row0 = static_cast<int64_t>(page) * B;
        const uint8_t* base = static_cast<const uint8_t*>(kv.k_pages) + d0 * E;
        for (int t0 = sub * RPL; t0 < valid; t0 += wpb * R) {
          uint4 raw[U];
          float sc[U];
#pragma unroll
          for (int u = 0; u < U; ++u) {
            // clamp: a repeated valid row changes nothing
            const int64_t row = row0 + min(t0 + u * wpb * RPL + rs, valid - 1);
            raw[u] = __ldg(reinterpret_cast<const uint4*>(base + row * (D * E)));
            if constexpr (KIND == HS_KV_FP8E4M3_G32)
              sc[u] = __ldg(kv.k_scales + row * (D / kQuantGroup) + d0 / kQuantGroup);
            else
              sc[u] = 1.0f;
          }
#pragma unroll
          for (int u = 0; u < U; ++u) fold<KIND, V>(raw[u], sc[u], mn, mx);
        }
      }
    }
    // the RPL row slots of the warp hold the same channels: combine them
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1)
#pragma unroll
      for (int c = 0; c < V; ++c) {
        mn[c] = fminf(mn[c], __shfl_xor_sync(0xffffffffu, mn[c], off));
        mx[c] = fmaxf(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], off));
      }
    if (rs == 0)
#pragma unroll
      for (int c = 0; c < V; ++c) { s_mn[warp][d0 + c] = mn[c]; s_mx[warp][d0 + c] = mx[c]; }
    if (lane == 0) s_ok[warp] = ok ? 1 : 0;
    __syncthreads();
    for (int idx = threadIdx.x; idx < per_cta * D; idx += kWarps * 32) {
      const int cb = idx / D, d = idx - cb * D;
      const int w0 = cb * wpb;
      if (!s_ok[w0]) continue;
      float lo = s_mn[w0][d], hi = s_mx[w0][d];
      for (int w = 1; w < wpb; ++w) { lo = fminf(lo, s_mn[w0 + w][d]); hi = fmaxf(hi, s_mx[w0 + w][d]); }
      const int64_t o = (pair * kv.max_blocks + jg + cb) * D + d;
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
    __syncthreads();  // the shared buffers are reused by the next group
  }
}

template <int D, int KIND, int U>
cudaError_t launch_u(const KvView& kv, int first_block, int nblocks, void* smin, void* smax,
                     unsigned* err, int sms, cudaStream_t st) {
  constexpr int RPL = 32 / (D * Elem<KIND>::kBytes / 16);
  const int per_cta = kWarps / warps_per_block(kv.block, RPL * U);
  const int gpp = ceil_div(nblocks, per_cta);
  const int64_t total = static_cast<int64_t>(gpp) * kv.hkv * kv.batch;
  static int per_sm = 0;  // resident CTAs of this kernel per SM
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, summaries_kernel<D, KIND, U>, kWarps * 32, 0) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
  }
  const int64_t resident = static_cast<int64_t>(sms > 0 ? sms : 148) * per_sm;
  const unsigned grid = static_cast<unsigned>(total < resident ? total : resident);
  return launch_pdl(summaries_kernel<D, KIND, U>, dim3(grid), dim3(kWarps * 32), 0, st, kv, first_block, gpp, total,
                    smin, smax, err);
}

template <int D, int KIND>
cudaError_t launch_k(const KvView& kv, int first_block, int nblocks, void* smin, void* smax,
                     unsigned* err, int sms, cudaStream_t st) {
  constexpr int RPL = 32 / (D * Elem<KIND>::kBytes / 16);
  switch (rounds_for(kv.block, RPL)) {
    case 8: return launch_u<D, KIND, 8>(kv, first_block, nblocks, smin, smax, err, sms, st);
    case 4: return launch_u<D, KIND, 4>(kv, first_block, nblocks, smin, smax, err, sms, st);
    case 2: return launch_u<D, KIND, 2>(kv, first_block, nblocks, smin, smax, err, sms, st);
    default: return launch_u<D, KIND, 1>(kv, first_block, nblocks, smin, smax, err, sms, st);
  }
}

template <int D>
cudaError_t launch_d(const KvView& kv, int first_block, int nblocks, void* smin, void* smax,
                     unsigned* err, int sms, cudaStream_t st) {
  switch (kv.kv_dtype) {
    case HS_KV_F32: return launch_k<D, HS_KV_F32>(kv, first_block, nblocks, smin, smax, err, sms, st);
    case HS_KV_BF16: return launch_k<D, HS_KV_BF16>(kv, first_block, nblocks, smin, smax, err, sms, st);
    default: return launch_k<D, HS_KV_FP8E4M3_G32>(kv, first_block, nblocks, smin, smax, err, sms, st);
  }
}

}  // namespace

cudaError_t launch_summaries(const KvView& kv, int first_block, void* smin, void* smax,
                             unsigned* err, int sms, cudaStream_t st) {
  const int nblocks = kv.max_blocks - first_block;
  if (nblocks <= 0 || kv.batch == 0) return cudaSuccess;
  return kv.head_dim == 128 ? launch_d<128>(kv, first_block, nblocks, smin, smax, err, sms, st)
                            : launch_d<64>(kv, first_block, nblocks, smin, smax, err, sms, st);
}

}  // namespace hs
