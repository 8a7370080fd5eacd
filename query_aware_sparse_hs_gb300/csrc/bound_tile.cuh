// One 128-block tile of the tensor-core bound score ("KV 稀疏化" wiki §5 Quest),
// bf16 summaries, head_dim 128, shared by the scoring kernel and the fused
// scoring + selection + attention kernel:
//
//   U[j][h] = sum_d smax_jd * q+_hd + smin_jd * q-_hd,   q+ = max(q, 0), q- = min(q, 0)
//
// A = [Smax | Smin] (128 blocks x 256, K-major, four 128-row x 64-channel
// halves with the 128-byte swizzle of the TMA copies), B = [Q+ | Q-] (16
// padded heads x 256, same layout), one M128 N16 accumulator in TMEM.
#pragma once

#include <cuda_bf16.h>

#include "tc_ptx.cuh"

namespace hs {
namespace bound {

constexpr int kTile = 128;             // blocks per tile (MMA M)
constexpr int kHalf = kTile * 128;     // 128 rows x 64 bf16
constexpr int kTileBytes = 4 * kHalf;  // smax halves, smin halves
constexpr int kQHalf = 16 * 128;       // 16 heads x 64 bf16
constexpr int kQBytes = 4 * kQHalf;    // Q+ halves, Q- halves

// [Q+ | Q-] operand of the g query heads whose first row is q_row0 (rows of
// 128 bf16 channels): thread t (0..127) writes 16-byte pieces of head row t/8,
// zero rows past g.  dst is 1024-byte aligned shared memory of kQBytes.
__device__ __forceinline__ void write_q(uint8_t* dst, const __nv_bfloat16* q, int64_t q_row0, int g, int t) {
  const int n = t >> 3, ch = t & 7;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 v = make_uint4(0, 0, 0, 0);
    if (n < g) v = *reinterpret_cast<const uint4*>(q + (q_row0 + n) * 128 + h * 64 + ch * 8);
    uint32_t w[4] = {v.x, v.y, v.z, v.w}, pos[4], neg[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // bf16 pair: keep the positive (negative) halves, zero the others
      const uint32_t lo = w[i] & 0xffffu, hi = w[i] >> 16;
      const bool lneg = (lo & 0x8000u) != 0, hneg = (hi & 0x8000u) != 0;
      pos[i] = (lneg ? 0u : lo) | ((hneg ? 0u : hi) << 16);
      neg[i] = (lneg ? lo : 0u) | ((hneg ? hi : 0u) << 16);
    }
    const int off = n * 128 + ((ch ^ (n & 7)) << 4);
    *reinterpret_cast<uint4*>(dst + h * kQHalf + off) = make_uint4(pos[0], pos[1], pos[2], pos[3]);
    *reinterpret_cast<uint4*>(dst + (2 + h) * kQHalf + off) = make_uint4(neg[0], neg[1], neg[2], neg[3]);
  }
}

// The 16 MMAs of one tile (issued by one thread): k < 8 Smax . Q+, k >= 8 Smin . Q-.
// tile / qop: shared-memory addresses of the A tile and the B operand.
__device__ __forceinline__ void issue_mmas(uint32_t d_tmem, uint32_t tile, uint32_t qop) {
  constexpr uint32_t idesc = tc::idesc_bf16(128, 16, false, false);
  const uint64_t adesc = tc::smem_desc(tile, 16, 1024, 2);
  const uint64_t bdesc = tc::smem_desc(qop, 16, 1024, 2);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int part = k >> 3, h = (k >> 2) & 1, kk = k & 3;
    const uint32_t aoff = (2 * part + h) * kHalf + kk * 32;
    const uint32_t boff = (2 * part + h) * kQHalf + kk * 32;
    tc::mma_f16(d_tmem, adesc + (aoff >> 4), bdesc + (boff >> 4), idesc, k > 0 ? 1u : 0u);
  }
}

}  // namespace bound
}  // namespace hs
