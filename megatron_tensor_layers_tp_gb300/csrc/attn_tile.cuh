// Attention building blocks shared by the decode / prefill attention kernels
// and the persistent decode-layer kernel: one warp's scores of 16 query rows
// against a K/V tile in shared memory (mma.sync m16n8k16 on ldmatrix
// fragments) and the fp32 online-softmax update of its running (m, l, O).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ptx.cuh"

namespace tpk {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 8-element chunk `ch` of row `row` in a K/V tile made of
// D/64 TMA boxes of [64 rows][128 B] with 128-byte swizzle.
__device__ __forceinline__ uint32_t kv_off(int row, int ch) {
  return (ch >> 3) * 8192 + row * 128 + (((ch & 7) ^ (row & 7)) << 4);
}

constexpr int kKeyTile = 64;

// One warp: scores of 16 query rows against NKT*8 keys (rows krow0.. of the
// smem tile), then the online-softmax update of (m, l, O).  qa: Q
// A-fragments; sK/sV: smem tiles.  key0: position of the first of those keys;
// lim[2]: last visible key position (inclusive) of the thread's two rows.
template <int D, int NKT>
__device__ __forceinline__ void attn_tile(const uint32_t (&qa)[D / 16][4], uint32_t sK,
                                          uint32_t sV, int krow0, int key0, const int (&lim)[2],
                                          float scale_log2, float (&m)[2], float (&l)[2],
                                          float (&o)[D / 8][4]) {
  const int lane = threadIdx.x & 31;
  float s[NKT][4];
#pragma unroll
  for (int nt = 0; nt < NKT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) s[nt][i] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
    for (int np = 0; np < NKT / 2; ++np) {  // pairs of 8-key n-tiles
      const int j = lane >> 3, r = lane & 7;
      const int key = krow0 + (np * 2 + (j >> 1)) * 8 + r;
      const int ch = kk * 2 + (j & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(sK + kv_off(key, ch), b0, b1, b2, b3);
      mma_16816(s[np * 2], qa[kk], b0, b1);
      mma_16816(s[np * 2 + 1], qa[kk], b2, b3);
    }
  }
  // mask + tile row max
  float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < NKT; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int key = key0 + nt * 8 + (lane & 3) * 2 + (i & 1);
      const int h = i >> 1;
      float v = s[nt][i] * scale_log2;
      v = key <= lim[h] ? v : -INFINITY;
      s[nt][i] = v;
      tmax[h] = fmaxf(tmax[h], v);
    }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
    tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
  }
  float alpha[2], mnew[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    mnew[h] = fmaxf(m[h], tmax[h]);
    alpha[h] = (mnew[h] == -INFINITY) ? 1.f : exp2f(m[h] - mnew[h]);
    m[h] = mnew[h];
    l[h] *= alpha[h];
  }
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt) {
    o[nt][0] *= alpha[0]; o[nt][1] *= alpha[0];
    o[nt][2] *= alpha[1]; o[nt][3] *= alpha[1];
  }
  uint32_t pa[NKT / 2][4];
#pragma unroll
  for (int nt = 0; nt < NKT; ++nt) {
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int h = i >> 1;
      p[i] = (mnew[h] == -INFINITY) ? 0.f : exp2f(s[nt][i] - mnew[h]);
      l[h] += p[i];
    }
    pa[nt >> 1][(nt & 1) * 2 + 0] = pack2(p[0], p[1]);
    pa[nt >> 1][(nt & 1) * 2 + 1] = pack2(p[2], p[3]);
  }
  // O += P V
#pragma unroll
  for (int kk = 0; kk < NKT / 2; ++kk) {
#pragma unroll
    for (int np = 0; np < D / 16; ++np) {
      const int j = lane >> 3, r = lane & 7;
      const int key = krow0 + kk * 16 + (j & 1) * 8 + r;
      const int ch = np * 2 + (j >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(sV + kv_off(key, ch), b0, b1, b2, b3);
      mma_16816(o[np * 2], pa[kk], b0, b1);
      mma_16816(o[np * 2 + 1], pa[kk], b2, b3);
    }
  }
}

// Decode with at most 8 query rows per KV head (one token per sequence): the
// keys go on the MMA M side and the query rows on N (S^T = K Q^T, then
// O^T += V^T P^T), so a 16-key step needs half the MMAs and exponentials of a
// 16-row query tile.

// Transposes the 8x8 b16 matrix held in the usual fragment layout (thread t:
// row t/4, columns 2(t%4) and 2(t%4)+1).
__device__ __forceinline__ uint32_t movm_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// B fragments of Q^T (16 d x 8 query rows) for every 16-wide d step, from 8
// padded query rows in shared memory (rows past the KV head's group are zero).
template <int D>
__device__ __forceinline__ void load_qt_frags(uint32_t sQ, int row_bytes, uint32_t (&qb)[D / 16][2]) {
  const int lane = threadIdx.x & 31;
  const int j = lane >> 3, r = lane & 7;
#pragma unroll
  for (int k2 = 0; k2 < D / 32; ++k2)  // matrix j: d columns (4 k2 + j) * 8 ..
    ldsm_x4(sQ + r * row_bytes + (k2 * 4 + j) * 16, qb[2 * k2][0], qb[2 * k2][1],
            qb[2 * k2 + 1][0], qb[2 * k2 + 1][1]);
}

// One warp: scores of 16 keys (rows krow0.. of the smem tile) against the 8
// query columns, then the online-softmax update of each column's (m, l) and
// of O^T.  key0: position of the first key; lim: last visible key position.
// m[c], l[c]: query columns 2 (lane % 4) + c; l holds this thread's share
// (its two keys per step), summed over the 8 lanes of a column at the end.
// o[dt]: O^T rows 16 dt + lane / 4 (+ 8), the same two columns.
template <int D>
__device__ __forceinline__ void attn_tile_t(const uint32_t (&qb)[D / 16][2], uint32_t sK,
                                            uint32_t sV, int krow0, int key0, int lim,
                                            float scale_log2, float (&m)[2], float (&l)[2],
                                            float (&o)[D / 16][4]) {
  const int lane = threadIdx.x & 31;
  const int j = lane >> 3, r = lane & 7;
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    // A = K[16 keys][16 d]: matrices (keys 0-7 | 8-15) x (d 0-7 | 8-15)
    uint32_t a[4];
    ldsm_x4(sK + kv_off(krow0 + (j & 1) * 8 + r, kk * 2 + (j >> 1)), a[0], a[1], a[2], a[3]);
    mma_16816(s, a, qb[kk][0], qb[kk][1]);
  }
  // s: keys lane/4 (s[0], s[1]) and lane/4 + 8 (s[2], s[3]); columns 2 (lane%4) + 0/1
  const int k_lo = key0 + (lane >> 2), k_hi = k_lo + 8;
  float v[4];
  v[0] = k_lo <= lim ? s[0] * scale_log2 : -INFINITY;
  v[1] = k_lo <= lim ? s[1] * scale_log2 : -INFINITY;
  v[2] = k_hi <= lim ? s[2] * scale_log2 : -INFINITY;
  v[3] = k_hi <= lim ? s[3] * scale_log2 : -INFINITY;
  float t[2] = {fmaxf(v[0], v[2]), fmaxf(v[1], v[3])};
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    t[c] = fmaxf(t[c], __shfl_xor_sync(0xffffffffu, t[c], 4));
    t[c] = fmaxf(t[c], __shfl_xor_sync(0xffffffffu, t[c], 8));
    t[c] = fmaxf(t[c], __shfl_xor_sync(0xffffffffu, t[c], 16));
  }
  float alpha[2], mnew[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    mnew[c] = fmaxf(m[c], t[c]);
    alpha[c] = (mnew[c] == -INFINITY) ? 1.f : exp2f(m[c] - mnew[c]);
    m[c] = mnew[c];
    l[c] *= alpha[c];
  }
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c = i & 1;
    p[i] = (mnew[c] == -INFINITY) ? 0.f : exp2f(v[i] - mnew[c]);
  }
  l[0] += p[0] + p[2];
  l[1] += p[1] + p[3];
#pragma unroll
  for (int dt = 0; dt < D / 16; ++dt) {
    o[dt][0] *= alpha[0]; o[dt][1] *= alpha[1];
    o[dt][2] *= alpha[0]; o[dt][3] *= alpha[1];
  }
  // P^T (16 keys x 8 columns) as the B operand: transpose each 8x8 block
  const uint32_t b0 = movm_trans(pack2(p[0], p[1]));
  const uint32_t b1 = movm_trans(pack2(p[2], p[3]));
#pragma unroll
  for (int dt = 0; dt < D / 16; ++dt) {
    // A = V^T[16 d][16 keys]: transposed loads of V (keys 0-7 | 8-15) x (d 0-7 | 8-15)
    uint32_t a[4];
    ldsm_x4_t(sV + kv_off(krow0 + (j >> 1) * 8 + r, dt * 2 + (j & 1)), a[0], a[1], a[2], a[3]);
    mma_16816(o[dt], a, b0, b1);
  }
}

// Loads the A fragments of 16 query rows from a padded smem block.
template <int D>
__device__ __forceinline__ void load_q_frags(uint32_t sQ, int row_bytes, uint32_t (&qa)[D / 16][4]) {
  const int lane = threadIdx.x & 31;
  const int j = lane >> 3, r = lane & 7;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int row = r + (j & 1) * 8;
    const int col = kk * 16 + (j >> 1) * 8;
    ldsm_x4(sQ + row * row_bytes + col * 2, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  }
}

}  // namespace tpk
