// One warp's sum of squares of a token's hidden row, for the RMSNorm folded
// into the column-parallel GEMM after it: 1 / sqrt(sum / width + eps).  The
// same arithmetic (and so the same bits) wherever the factor is computed.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace tpk {

// From the bf16 row itself: lane l takes 16-byte chunks l, l + 32, ... (eight
// loads in flight at a time), squares in fp32 with fused multiply-adds, then
// a butterfly over the warp.  Every lane returns the sum.
__device__ __forceinline__ float warp_row_sumsq(const uint16_t* row, int width) {
  const int lane = threadIdx.x & 31;
  const uint4* xr = reinterpret_cast<const uint4*>(row);
  const int nv = width >> 3;
  float ss = 0.f;
  auto add_sq = [&](const uint4& p) {
    const uint32_t w4[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float lo = __uint_as_float(w4[q] << 16), hi = __uint_as_float(w4[q] & 0xFFFF0000u);
      ss = fmaf(lo, lo, ss);
      ss = fmaf(hi, hi, ss);
    }
  };
  int v = lane;
  for (; v + 7 * 32 < nv; v += 8 * 32) {
    uint4 p[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) p[q] = __ldcg(xr + v + q * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) add_sq(p[q]);
  }
  for (; v < nv; v += 32) add_sq(__ldcg(xr + v));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return ss;
}

// From per-32-feature partial sums left by the kernel that wrote the row
// (n_slots floats, a multiple of 4, 16-byte aligned): lane l adds the float4
// chunks l, l + 32, ..., then a butterfly over the warp.
__device__ __forceinline__ float warp_partials_sumsq(const float* slots, int n_slots) {
  const int lane = threadIdx.x & 31;
  float ss = 0.f;
  for (int i4 = lane; i4 < (n_slots >> 2); i4 += 32) {
    const float4 p = __ldcg(reinterpret_cast<const float4*>(slots) + i4);
    ss += (p.x + p.y) + (p.z + p.w);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return ss;
}

}  // namespace tpk
