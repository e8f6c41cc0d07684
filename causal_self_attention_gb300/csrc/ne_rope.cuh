// ne_rope.cuh -- RoPE applied in place to a 128 x 64 bf16 tile held in shared
// memory with the 128-byte swizzle, right after its TMA load.
//
// Rotate-half arrangement (RoFormer, Su et al. 2021): element i < 32 is paired
// with element i + 32 and turned by p * theta_i,
//     x'_i      = x_i c - x_{i+32} s,      x'_{i+32} = x_{i+32} c + x_i s,
// where (c, s) come from the fp32 table built on the host from double values.
// The fp32 evaluation order is fixed: lo = fma(x_i, c, -(x_{i+32} * s)),
// hi = fma(x_{i+32}, c, x_i * s), then round to nearest even bf16.  ("Tiny
// Hackable CUDA", section 3: RoPE encodes relative position in the attention
// projections.)
//
// The table row of a position (32 (cos, sin) pairs = 256 bytes) is loaded into
// registers by rope_load_row ahead of time, from the warp-interleaved copy of
// the table (a warp's 32 consecutive positions come in 16 fully used
// 512-byte pieces instead of 512 scattered 16-byte pieces), so that the table
// is off the critical path; rope_rotate_row then only touches shared memory.
#pragma once

#include "ne_sm100.cuh"

namespace ne {

struct RopeRow {
  float4 t[16];  // t[4c + w] = (cos_i, sin_i, cos_{i+1}, sin_{i+1}), i = 8c + 2w
};

__device__ __forceinline__ void rope_load_row(const RopeTable& rt, int pos, RopeRow& r) {
  if (pos >= rt.capacity) pos = rt.capacity - 1;  // only rows past the sequence end
  const float4* cs = rt.csw + static_cast<long long>(pos >> 5) * (16 * 32) + (pos & 31);
#pragma unroll
  for (int i = 0; i < 16; ++i) r.t[i] = __ldg(cs + 32 * i);
}

// The same registers from the row layout of the table (cs: one 256-byte row
// per position; for a thread that loads its rows rarely, off the critical
// path, where the warp-interleaved copy buys nothing).
__device__ __forceinline__ void rope_load_row_flat(const RopeTable& rt, int pos, RopeRow& r) {
  if (pos >= rt.capacity) pos = rt.capacity - 1;  // only rows past the sequence end
  const float4* cs = reinterpret_cast<const float4*>(rt.cs + static_cast<long long>(pos) * 32);
#pragma unroll
  for (int i = 0; i < 16; ++i) r.t[i] = __ldg(cs + i);
}

// Rotate one row (64 elements = 8 swizzled 16-byte chunks) of `tile` with the
// table row `cs` of its position.
__device__ __forceinline__ void rope_rotate_row(uint8_t* tile, int row, const RopeRow& cs) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4* plo = reinterpret_cast<uint4*>(tile + sw128_offset(row, c));
    uint4* phi = reinterpret_cast<uint4*>(tile + sw128_offset(row, c + 4));
    const uint4 lo = *plo, hi = *phi;
    uint32_t wl[4] = {lo.x, lo.y, lo.z, lo.w};
    uint32_t wh[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      // Elements i = 8c + 2w and i + 1 (low and high half of the word).
      const float4 t = cs.t[4 * c + w];
      const float a0 = bf16lo_to_f32(wl[w]), a1 = bf16hi_to_f32(wl[w]);
      const float b0 = bf16lo_to_f32(wh[w]), b1 = bf16hi_to_f32(wh[w]);
      const float lo0 = __fmaf_rn(a0, t.x, -__fmul_rn(b0, t.y));
      const float hi0 = __fmaf_rn(b0, t.x, __fmul_rn(a0, t.y));
      const float lo1 = __fmaf_rn(a1, t.z, -__fmul_rn(b1, t.w));
      const float hi1 = __fmaf_rn(b1, t.z, __fmul_rn(a1, t.w));
      wl[w] = pack_bf16x2(lo0, lo1);
      wh[w] = pack_bf16x2(hi0, hi1);
    }
    *plo = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    *phi = make_uint4(wh[0], wh[1], wh[2], wh[3]);
  }
}

}  // namespace ne
