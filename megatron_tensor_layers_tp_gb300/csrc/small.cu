// Memory-bound kernels of the layer: vocab-parallel embedding, replicated
// RMSNorm, the separate rank-ordered reduction of the unfused row-parallel
// variant, the RoPE table and the shard builder's row copies.  All move
// 16-byte vectors with consecutive threads on consecutive addresses.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include <algorithm>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace tpk {

// ---------------------------------------------------------------------------
// Vocab-parallel embedding ("第 9 章 多进程与张量并行", §3.2 Vocab Parallel;
// "张量、流水线与数据并行", 线性层怎么切: 词嵌入).  Rank r holds vocab rows
// [r Vp/t, (r+1) Vp/t); a token contributes its row on the owner rank and -0.0
// on every other rank, and the all-reduce sums the t contributions in rank
// order.  Because x + (-0.0) == x for every x, that sum is the owner's row bit
// for bit, so the kernel copies the owner's row: the masked lookups of the
// other ranks and the reduction are exact no-ops it does not need to execute.
// One warp per token; the t shards are stored back to back, so rank r's local
// row l sits at padded row r*Vp/t + l.
// ---------------------------------------------------------------------------
__global__ void embed_kernel(const uint16_t* __restrict__ table, int vocab, int vocab_per_rank,
                             int t, const int32_t* __restrict__ ids, int M, int H,
                             uint16_t* __restrict__ h, float* __restrict__ sq, int* status) {
  pdl_launch_dependents();
  pdl_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= M) return;
  const int id = ids[warp];
  uint4* dst = reinterpret_cast<uint4*>(h + (int64_t)warp * H);
  const int nvec = H / 8;
  float ss = 0.f;
  if (id < 0 || id >= vocab) {
    if (lane == 0) record_status(status, kStatusTokenRange);
    for (int i = lane; i < nvec; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
  } else {
    const int owner = id / vocab_per_rank;          // the one rank whose lookup hits
    const int local = id - owner * vocab_per_rank;  // row inside that rank's shard
    const uint4* src = reinterpret_cast<const uint4*>(
        table + ((int64_t)owner * vocab_per_rank + local) * H);
    // kEmbedBatch 16-byte loads of a lane in flight together, then their stores
    constexpr int kEmbedBatch = 8;
    for (int i0 = lane; i0 < nvec; i0 += 32 * kEmbedBatch) {
      uint4 v[kEmbedBatch];
#pragma unroll
      for (int k = 0; k < kEmbedBatch; ++k) {
        const int i = i0 + 32 * k;
        v[k] = i < nvec ? __ldg(&src[i]) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kEmbedBatch; ++k) {
        const int i = i0 + 32 * k;
        if (i < nvec) dst[i] = v[k];
        const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = __uint_as_float(w4[q] << 16), hi = __uint_as_float(w4[q] & 0xFFFF0000u);
          ss = fmaf(lo, lo, fmaf(hi, hi, ss));
        }
      }
    }
  }
  if (sq) {
    // the row's sum of squares for the RMSNorm of the first layer, in the
    // [token][4 slots] form the GEMMs read (slot 0, the rest zero)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane < 4) sq[(int64_t)warp * 4 + lane] = lane == 0 ? ss : 0.f;
  }
}

cudaError_t launch_embed(const uint16_t* table, int vocab, int vocab_per_rank, int t,
                         const int32_t* ids, int M, int H, uint16_t* h, float* sq, int* status,
                         cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const int warps_per_block = 8;
  const int blocks = (M + warps_per_block - 1) / warps_per_block;
  return launch_k(embed_kernel, dim3(blocks), dim3(warps_per_block * 32), 0, st, table, vocab,
                  vocab_per_rank, t, ids, M, H, h, sq, status);
}

// ---------------------------------------------------------------------------
// RMSNorm, replicated on every rank ("第 9 章", §3.2: small layers such as
// RMSNorm are copied whole to each rank): one copy serves all emulated ranks.
// y = x / sqrt(mean(x^2) + eps) * w in fp32; one CTA per row.  With `rows`,
// row i of y normalises row rows[i] of x (the sampled rows before the head).
// ---------------------------------------------------------------------------
constexpr int kNormThreads = 256;
constexpr int kNormVec = 4;  // 16-byte vectors a thread keeps in registers (H <= 8192)

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(
    const uint16_t* __restrict__ x, int64_t ldx, const int32_t* __restrict__ rows,
    const uint16_t* __restrict__ w, int H, float eps, uint16_t* __restrict__ y, int64_t ldy,
    bool w_loaded) {
  __shared__ float red[kNormThreads / 32];
  pdl_launch_dependents();
  const int i = blockIdx.x;
  const uint4* wr = reinterpret_cast<const uint4*>(w);
  const int nvec = H / 8;
  const bool cached = nvec <= kNormVec * kNormThreads;
  // a model's norm weight is written once, when the model is loaded
  // (w_loaded): then it is fetched before waiting for the kernel that wrote x
  uint4 wv[kNormVec], xv[kNormVec];
  auto load_w = [&]() {
#pragma unroll
    for (int k = 0; k < kNormVec; ++k) {
      const int v = threadIdx.x + k * kNormThreads;
      if (v < nvec) wv[k] = wr[v];
    }
  };
  if (cached && w_loaded) load_w();
  pdl_wait();
  if (cached && !w_loaded) load_w();
  const int src_row = rows ? rows[i] : i;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)src_row * ldx);
  uint4* yr = reinterpret_cast<uint4*>(y + (int64_t)i * ldy);
  auto sumsq = [](const uint4& p, float ss) {
    const uint16_t* e = reinterpret_cast<const uint16_t*>(&p);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float f = bf16_to_f(e[j]);
      ss = fmaf(f, f, ss);
    }
    return ss;
  };
  auto scaled = [](const uint4& p, const uint4& q, float inv) {
    const uint16_t* e = reinterpret_cast<const uint16_t*>(&p);
    const uint16_t* g = reinterpret_cast<const uint16_t*>(&q);
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      op[j] = pack_bf16x2(bf16_to_f(e[2 * j]) * inv * bf16_to_f(g[2 * j]),
                          bf16_to_f(e[2 * j + 1]) * inv * bf16_to_f(g[2 * j + 1]));
    return o;
  };
  float ss = 0.f;
  if (cached) {  // one pass over x: its vectors stay in registers
#pragma unroll
    for (int k = 0; k < kNormVec; ++k) {
      const int v = threadIdx.x + k * kNormThreads;
      if (v < nvec) xv[k] = xr[v];
    }
#pragma unroll
    for (int k = 0; k < kNormVec; ++k)
      if (threadIdx.x + k * kNormThreads < nvec) ss = sumsq(xv[k], ss);
  } else {
    for (int v = threadIdx.x; v < nvec; v += kNormThreads) ss = sumsq(xr[v], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int k = 0; k < kNormThreads / 32; ++k) tot += red[k];
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  if (cached) {
#pragma unroll
    for (int k = 0; k < kNormVec; ++k) {
      const int v = threadIdx.x + k * kNormThreads;
      if (v < nvec) yr[v] = scaled(xv[k], wv[k], inv);
    }
  } else {
    for (int v = threadIdx.x; v < nvec; v += kNormThreads) yr[v] = scaled(xr[v], wr[v], inv);
  }
}

cudaError_t launch_rmsnorm(const uint16_t* x, int64_t ldx, const int32_t* rows, const uint16_t* w,
                           int M, int H, float eps, uint16_t* y, int64_t ldy, cudaStream_t st,
                           bool w_loaded) {
  if (M == 0) return cudaSuccess;
  return launch_k(rmsnorm_kernel, dim3(M), dim3(kNormThreads), 0, st, x, ldx, rows, w, H, eps, y,
                  ldy, w_loaded);
}

// ---------------------------------------------------------------------------
// Unfused row-parallel reduction: y = (P_0 + P_1 + ... + P_{t-1}) + residual,
// summed in fp32 in rank order and rounded once to bf16 ("第 9 章", §3.1: the
// all-reduce of a row-parallel layer is a sum).  P_r: [M, H] fp32 partials.
// ---------------------------------------------------------------------------
__global__ void reduce_ranks_kernel(const float4* __restrict__ P, int64_t rank_stride4, int t,
                                    int64_t n4, int H4, const uint2* __restrict__ bias,
                                    const uint2* __restrict__ residual, uint2* __restrict__ y) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 acc = P[i];
    for (int r = 1; r < t; ++r) {
      const float4 p = P[r * rank_stride4 + i];
      acc.x += p.x; acc.y += p.y; acc.z += p.z; acc.w += p.w;
    }
    if (bias) {  // the output's bias, once, after the rank sum
      const uint2 bv = bias[i % H4];
      acc.x += __uint_as_float(bv.x << 16);
      acc.y += __uint_as_float(bv.x & 0xFFFF0000u);
      acc.z += __uint_as_float(bv.y << 16);
      acc.w += __uint_as_float(bv.y & 0xFFFF0000u);
    }
    if (residual) {
      const uint2 rv = residual[i];
      acc.x += __uint_as_float(rv.x << 16);
      acc.y += __uint_as_float(rv.x & 0xFFFF0000u);
      acc.z += __uint_as_float(rv.y << 16);
      acc.w += __uint_as_float(rv.y & 0xFFFF0000u);
    }
    y[i] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
}

cudaError_t launch_reduce_ranks(const float* partials, int64_t rank_stride, int t, int M, int H,
                                const uint16_t* bias, const uint16_t* residual, uint16_t* y,
                                cudaStream_t st) {
  const int64_t n4 = (int64_t)M * H / 4;
  if (n4 == 0) return cudaSuccess;
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  return launch_k(reduce_ranks_kernel, dim3(blocks), dim3(256), 0, st,
                  reinterpret_cast<const float4*>(partials), rank_stride / 4, t, n4, H / 4,
                  reinterpret_cast<const uint2*>(bias), reinterpret_cast<const uint2*>(residual),
                  reinterpret_cast<uint2*>(y));
}

// ---------------------------------------------------------------------------
// RoPE table: (cos, sin) of p * theta^(-2j/d), evaluated in double, stored as
// float, for p < max_pos and j < d/2 (rotate-half pairing of j and j + d/2).
// ---------------------------------------------------------------------------
__global__ void rope_table_kernel(float2* table, int max_pos, int half, int head_dim,
                                  double theta) {
  const int64_t n = (int64_t)max_pos * half;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int p = (int)(i / half), j = (int)(i % half);
    const double inv_freq = pow(theta, -(2.0 * j) / head_dim);
    double s, c;
    sincos((double)p * inv_freq, &s, &c);
    table[i] = make_float2((float)c, (float)s);
  }
}

cudaError_t launch_rope_table(float2* table, int max_pos, int head_dim, double theta,
                              cudaStream_t st) {
  const int half = head_dim / 2;
  const int64_t n = (int64_t)max_pos * half;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  rope_table_kernel<<<blocks, 256, 0, st>>>(table, max_pos, half, head_dim, theta);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Shard builder: dst row i <- src row row_map[i] (n_cols elements), or zeros
// when row_map[i] < 0.  Used once at load time.
// ---------------------------------------------------------------------------
__global__ void copy_rows_kernel(uint16_t* __restrict__ dst, int64_t dst_ld,
                                 const uint16_t* __restrict__ src, int64_t src_ld,
                                 const int32_t* __restrict__ row_map, int n_cols, bool vec) {
  const int i = blockIdx.x;
  const int sr = row_map[i];
  uint16_t* d = dst + (int64_t)i * dst_ld;
  if (vec) {
    uint4* d4 = reinterpret_cast<uint4*>(d);
    const uint4* s4 = sr >= 0 ? reinterpret_cast<const uint4*>(src + (int64_t)sr * src_ld) : nullptr;
    for (int c = threadIdx.x; c < n_cols / 8; c += blockDim.x)
      d4[c] = s4 ? s4[c] : make_uint4(0, 0, 0, 0);
  } else {
    const uint16_t* s = sr >= 0 ? src + (int64_t)sr * src_ld : nullptr;
    for (int c = threadIdx.x; c < n_cols; c += blockDim.x) d[c] = s ? s[c] : 0;
  }
}

// ---------------------------------------------------------------------------
// Pipeline-stage hand-off ("张量、流水线与数据并行", 流水线并行): CTA (row i,
// rank r) moves rank r's slice of columns [r H/t, (r+1) H/t) of hidden row i
// into the next stage's buffer, where the t slices land side by side (the
// receiving stage's all-gather inside its TP group).  16-byte vectors;
// (H/t) % 8 == 0 is checked by the host.
// ---------------------------------------------------------------------------
__global__ void stage_send_kernel(const uint16_t* __restrict__ src, uint16_t* __restrict__ dst,
                                  int H, int slice) {
  pdl_launch_dependents();
  pdl_wait();  // the sending stage's last kernel wrote src
  const int64_t off = (int64_t)blockIdx.x * H + (int64_t)blockIdx.y * slice;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + off);
  uint4* d4 = reinterpret_cast<uint4*>(dst + off);
  for (int c = threadIdx.x; c < slice / 8; c += blockDim.x) d4[c] = s4[c];
}

cudaError_t launch_stage_send(const uint16_t* src, uint16_t* dst, int M, int H, int t,
                              cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  return launch_k(stage_send_kernel, dim3(M, t), dim3(128), 0, st, src, dst, H, H / t);
}

// ---------------------------------------------------------------------------
// Failure-detection self-test: one warp waits on an mbarrier phase that no
// arrival ever completes.  The bounded wait gives up after `limit` SM cycles,
// records the timeout in *status and the kernel returns normally.
// ---------------------------------------------------------------------------
__global__ void wait_timeout_kernel(int* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, status, limit);  // phase 0 never completes
}

cudaError_t launch_wait_timeout(int* status, long long limit, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(status, limit);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// RMSNorm weight folded into the rows of the GEMM that consumes the norm's
// output (load time): (x / rms(x) * w) . W[n] = (x . (W[n] * w)) / rms(x), so
// W[n][k] * w[k] is stored once and the per-token 1/rms is applied to the
// GEMM's output.  One thread per element; fp32 product (exact for two bf16
// values), rounded to nearest even.
// ---------------------------------------------------------------------------
__global__ void fold_cols_kernel(uint16_t* __restrict__ dst, const uint16_t* __restrict__ src,
                                 const uint16_t* __restrict__ w, int64_t n, int cols) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = f_to_bf16(bf16_to_f(src[i]) * bf16_to_f(w[i % cols]));
}

cudaError_t launch_fold_cols(uint16_t* dst, const uint16_t* src, const uint16_t* w, int64_t n_rows,
                             int cols, cudaStream_t st) {
  const int64_t n = n_rows * cols;
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, 1 << 20);
  fold_cols_kernel<<<(unsigned)blocks, 256, 0, st>>>(dst, src, w, n, cols);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Host <-> device transfers of the host-buffer entry point, as kernels: on a
// GPU that reaches host memory coherently (NVLink-C2C) a kernel can read and
// write pinned host memory directly, so the step's chain of programmatically
// dependent launches is not broken by copy-engine operations.  Both wait for
// their predecessor before touching memory (the host buffers may be reused
// from one call to the next).  Host loads are volatile (ld.cv: fetched from
// host memory every time, never from a cached line) and host stores write
// through.  16-byte vectors, grid-stride.
// ---------------------------------------------------------------------------
__global__ void host_in_kernel(const uint4* __restrict__ src_host, uint4* __restrict__ dst,
                               int64_t n16) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += stride)
    dst[i] = __ldcv(src_host + i);
}

__global__ void host_out_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst_host,
                                int64_t n16) {
  pdl_launch_dependents();
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16; i += stride)
    __stwt(dst_host + i, src[i]);
}

cudaError_t launch_host_copy(const void* src, void* dst, size_t bytes, bool to_host,
                             cudaStream_t st) {
  const int64_t n16 = (int64_t)(bytes / 16);
  if (n16 == 0) return cudaSuccess;
  const int blocks = (int)std::min<int64_t>((n16 + 255) / 256, 1024);
  if (to_host)
    return launch_k(host_out_kernel, dim3(blocks), dim3(256), 0, st,
                    static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16);
  return launch_k(host_in_kernel, dim3(blocks), dim3(256), 0, st, static_cast<const uint4*>(src),
                  static_cast<uint4*>(dst), n16);
}

// ---------------------------------------------------------------------------
// Weight shards in K blocks: src [ranks][rows][cols] (row-major, cols % 64 ==
// 0) -> dst [ranks][cols / 64][rows][64], so that the 128-byte row pieces of
// one 64-wide K step are contiguous (a 128-row TMA box is then one 16 KB
// run of memory instead of 128 pieces 2*cols bytes apart).  Block (row,
// rank) moves its row; 8 threads per 128-byte piece.  Used once at load time.
// ---------------------------------------------------------------------------
__global__ void reblock_k64_kernel(uint16_t* __restrict__ dst, const uint16_t* __restrict__ src,
                                   int rows, int cols) {
  const int row = blockIdx.x, rank = blockIdx.y;
  const int64_t slice = (int64_t)rows * cols;
  const uint4* s4 = reinterpret_cast<const uint4*>(src + rank * slice + (int64_t)row * cols);
  uint16_t* d = dst + rank * slice + (int64_t)row * 64;
  for (int v = threadIdx.x; v < cols / 8; v += blockDim.x) {
    const int kb = v >> 3, part = v & 7;  // 64-wide block, 16-byte part of its 128 bytes
    reinterpret_cast<uint4*>(d + (int64_t)kb * rows * 64)[part] = s4[v];
  }
}

cudaError_t launch_reblock_k64(uint16_t* dst, const uint16_t* src, int ranks, int rows, int cols,
                               cudaStream_t st) {
  if (ranks == 0 || rows == 0 || cols == 0) return cudaSuccess;
  if (cols % 64 || (reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) % 16)
    return cudaErrorInvalidValue;
  reblock_k64_kernel<<<dim3(rows, ranks), 128, 0, st>>>(dst, src, rows, cols);
  return cudaGetLastError();
}

cudaError_t launch_copy_rows(uint16_t* dst, int64_t dst_ld, const uint16_t* src, int64_t src_ld,
                             const int32_t* row_map, int n_rows, int n_cols, cudaStream_t st) {
  if (n_rows == 0) return cudaSuccess;
  const bool vec = (n_cols % 8 == 0) && (dst_ld % 8 == 0) && (src_ld % 8 == 0) &&
                   (reinterpret_cast<uintptr_t>(dst) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(src) % 16 == 0);
  copy_rows_kernel<<<n_rows, 256, 0, st>>>(dst, dst_ld, src, src_ld, row_map, n_cols, vec);
  return cudaGetLastError();
}

}  // namespace tpk
