// Head-sharded GQA attention over the per-rank KV caches ("Tensor Parallelism
// 执行路径", KV Cache 在 TP 下怎样分布: rank i stores and reads only the K/V of
// its own heads; "张量、流水线与数据并行", 线性层怎么切: attention on each rank's own
// heads with its own KV).
//
// All t ranks run in one launch.  Rank r owns Q heads [r n_h/t, (r+1) n_h/t),
// which in the concatenated q/o buffers is simply the global head order, and
// Q head j reads KV head g = j / (n_h/n_kv).  KV head g lives in rank copy
// g / kv_r at local index g % kv_r; replica ranks (n_kv < t) share that copy,
// so one CTA serves every Q head of KV head g and reads its K/V once.
//
// K/V tiles of 64 positions arrive by TMA (128-byte swizzle) and feed
// mma.sync tiles from ldmatrix; scores and the online softmax stay in fp32.
//   decode : one query token per sequence; the (sequence, KV head, key tile)
//            space is split evenly over the grid: whole (sequence, KV head)
//            pairs per CTA when the host finds such a grid that fills the
//            GPU with short enough streams, otherwise a flat split over all
//            SMs whose pieces of one pair are combined in key order by the
//            last CTA to finish one (atomic ticket, no waiting).
//   prefill: causal; one CTA per (sequence, Q head, 64-token query block).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn_tile.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace tpk {

// ============================================================================
// decode
// ============================================================================
// Two groups of four compute warps take alternate 64-key tiles (each warp 16
// keys of its group's tile), so two tiles are in the mma/softmax chain at once.
constexpr int kDecGroupWarps = 4;
constexpr int kDecGroups = 2;
constexpr int kDecWarps = kDecGroups * kDecGroupWarps;  // compute warps
constexpr int kDecThreads = (kDecWarps + 1) * 32;        // + producer warp

template <int D>
struct DecSmem {
  static constexpr int kTileBytes = (D / 64) * 8192;       // one K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kQRow = D * 2 + 16;                 // padded bf16 row
  // An even stage count pins every stage to one warp group inside a segment
  // (stage n % S, group n % 2 relative to the segment's first unit), so a
  // group never waits on a stage whose previous fill, owned by the other
  // group, is still in flight (an mbarrier parity wait cannot tell that fill
  // from the one it wants).
  static constexpr int kStages = D == 128 ? 4 : 8;
  static_assert(kStages % kDecGroups == 0, "stages must split evenly between the warp groups");
  // combine rows: O, m, l per warp/row; the pitch keeps the two rows a warp
  // reads at once 18 banks apart (16 lanes per row, columns lane + 16 j)
  static constexpr int kCombLd = D + 18;
  static constexpr int kComb = kDecWarps * 16 * kCombLd;  // floats
  static constexpr size_t bytes(int) {
    return 1024 + (size_t)kStages * kStageBytes + 16 * kQRow + (size_t)kComb * 4 + 256;
  }
};

// N fp32 values of one output row scaled by inv, stored as bf16 at columns
// dst[0], dst[16], dst[32], ... (a row's 16 threads write 32 contiguous bytes
// per store)
template <int N>
__device__ __forceinline__ void store_out_row(uint16_t* dst, const float (&v)[N], float inv) {
#pragma unroll
  for (int j = 0; j < N; ++j) dst[16 * j] = f_to_bf16(v[j] * inv);
}

template <int D>
__global__ void __launch_bounds__(kDecThreads, 1) attn_decode_kernel(const __grid_constant__ AttnArgs a) {
  using L = DecSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem;
  uint8_t* sQ = tiles + L::kStages * L::kStageBytes;
  float* comb = reinterpret_cast<float*>(sQ + 16 * L::kQRow);
  uint64_t* full = reinterpret_cast<uint64_t*>(comb + L::kComb);
  uint64_t* empty = full + L::kStages;
  int* last_flag = reinterpret_cast<int*>(empty + L::kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = L::kStages;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], kDecGroupWarps); }
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  uint64_t pol = 0;
  if (threadIdx.x == kDecWarps * 32) {  // producer: descriptors are parameters, fetch early
    tma_prefetch_desc(&a.tmK);
    tma_prefetch_desc(&a.tmV);
    pol = policy_evict_first();
  }
  __syncthreads();
  pdl_launch_dependents();

  const int G = a.grid, c = blockIdx.x;
  const int64_t T = a.total_units;
  const int TB = a.tiles_per_bg;
  const int64_t beg = range_begin(c, T, G), end = range_begin(c + 1, T, G);

  if (warp == kDecWarps) {
    // producer
    if (lane == 0) {
      uint32_t n = 0;
      // (sequence, KV head, tile) of unit u, walked incrementally
      const int64_t bg0 = beg / TB;
      int tile = static_cast<int>(beg - bg0 * TB);
      int b = static_cast<int>(bg0 / a.n_kv), g = static_cast<int>(bg0 % a.n_kv);
      auto issue = [&](uint32_t s) {
        const int slice = ((g / a.kv_r) * a.n_seqs + b) * a.kv_r + (g % a.kv_r);
        mbar_arrive_expect_tx(&full[s], L::kStageBytes);
        uint8_t* kt = tiles + s * L::kStageBytes;
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_load_3d(kt + bx * 8192, &a.tmK, &full[s], bx * 64, tile * kKeyTile, slice, pol);
          tma_load_3d(kt + L::kTileBytes + bx * 8192, &a.tmV, &full[s], bx * 64, tile * kKeyTile,
                      slice, pol);
        }
      };
      auto advance = [&]() {
        if (++tile == TB) {
          tile = 0;
          if (++g == a.n_kv) { g = 0; ++b; }
        }
      };
      // Cache rows below a sequence's position were written before this
      // launch chain: the qkv projection that writes this step's rows signals
      // its dependents only after its own wait, so every kernel older than it
      // has completed.  Tiles wholly below the position therefore fill the
      // first stages before the wait for q and the new rows.
      int64_t u = beg;
      while (u < end && n < (uint32_t)S && (tile + 1) * kKeyTile <= a.positions[b]) {
        issue(n);
        ++n;
        if (++u < end) advance();
      }
      pdl_wait();
      for (; u < end; ++u) {
        const uint32_t s = n % S, ph = (n / S) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, a.status)) break;
        issue(s);
        ++n;
        if (u + 1 < end) advance();
      }
      for (uint32_t i = (n > (uint32_t)S ? n - S : 0); i < n; ++i)
        mbar_wait(&full[i % S], (i / S) & 1, a.status);
    } else {
      pdl_wait();
    }
  } else {
    pdl_wait();  // q and the newest cache rows were written by the preceding kernels
    const int ctid = threadIdx.x;  // 0..255
    uint32_t n_base = 0;           // CTA-local index of the segment's first unit
    bool alive = true;
    for (int64_t u0 = beg; u0 < end;) {
      const int64_t bg = u0 / TB;
      const int64_t seg_end = min(end, (bg + 1) * TB);
      const int len = static_cast<int>(seg_end - u0);
      const int tile0 = static_cast<int>(u0 - bg * TB);
      const int b = static_cast<int>(bg / a.n_kv), g = static_cast<int>(bg % a.n_kv);
      const int pos = a.positions[b];
      // stage the group's query rows (16 rows, zero beyond the group)
      for (int i = ctid; i < 16 * (D / 8); i += kDecWarps * 32) {
        const int row = i / (D / 8), ch = i % (D / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < a.group)
          v = *reinterpret_cast<const uint4*>(a.q + (int64_t)b * a.ld_q +
                                              (int64_t)(g * a.group + row) * D + ch * 8);
        *reinterpret_cast<uint4*>(sQ + row * L::kQRow + ch * 16) = v;
      }
      bar_sync(1, kDecWarps * 32);
      uint32_t qa[D / 16][4];
      load_q_frags<D>(smem_u32(sQ), L::kQRow, qa);
      float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
      float o[D / 8][4];
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[nt][i] = 0.f;
      const int lim[2] = {pos, pos};
      // group grp takes tiles grp, grp + 2, ... of the segment; every warp of
      // it takes its own 16 keys of the tile, so a stage is released after a
      // quarter of that tile's work and the other stages keep streaming
      const int grp = warp / kDecGroupWarps, wq = warp % kDecGroupWarps;
      constexpr int kWarpKeys = kKeyTile / kDecGroupWarps;
      for (int i = grp; i < len; i += kDecGroups) {
        const uint32_t n = n_base + i;
        const uint32_t s = n % S, ph = (n / S) & 1;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&full[s], ph, a.status);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) { alive = false; break; }
        const int key0 = (tile0 + i) * kKeyTile + wq * kWarpKeys;
        if (key0 <= pos) {
          const uint32_t st = smem_u32(tiles + s * L::kStageBytes);
          attn_tile<D, kWarpKeys / 8>(qa, st, st + L::kTileBytes, wq * kWarpKeys, key0, lim,
                                      a.scale_log2, m, l, o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      n_base += len;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
      }
      // combine: every warp's (m, l, O) meets the others in smem
      constexpr int CL = L::kCombLd;
      float* cw = comb + warp * 16 * CL;
      const int r0 = lane >> 2;
#pragma unroll
      for (int nt = 0; nt < D / 8; ++nt) {
        const int col = nt * 8 + (lane & 3) * 2;
        *reinterpret_cast<float2*>(cw + r0 * CL + col) = make_float2(o[nt][0], o[nt][1]);
        *reinterpret_cast<float2*>(cw + (r0 + 8) * CL + col) = make_float2(o[nt][2], o[nt][3]);
      }
      if ((lane & 3) == 0) {
        cw[r0 * CL + D] = m[0]; cw[r0 * CL + D + 1] = l[0];
        cw[(r0 + 8) * CL + D] = m[1]; cw[(r0 + 8) * CL + D + 1] = l[1];
      }
      const bool any_dead = bar_sync_or(1, kDecWarps * 32, !alive);
      // 256 threads: row = ctid / 16, D/16 columns each (8 for D = 128): columns
      // cl, cl + 16, ... so that a row's 16 threads read 16 consecutive floats
      constexpr int CPT = D / 16;
      const int row = ctid >> 4, cl = ctid & 15;
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, comb[(w * 16 + row) * CL + D]);
      float ll = 0.f, acc[CPT];
#pragma unroll
      for (int j = 0; j < CPT; ++j) acc[j] = 0.f;
#pragma unroll 2
      for (int w = 0; w < kDecWarps; ++w) {
        const float* cr = comb + (w * 16 + row) * CL;
        const float mw = cr[D];
        if (mw == -INFINITY) continue;
        const float sc = exp2f(mw - mm);
        ll += cr[D + 1] * sc;
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[j] += cr[cl + 16 * j] * sc;
      }
      const int nseg = owner_of((bg + 1) * TB - 1, T, G) - owner_of(bg * TB, T, G) + 1;
      uint16_t* orow = a.o + (int64_t)b * a.ld_o + (int64_t)(g * a.group + row) * D + cl;
      if (nseg == 1) {
        if (row < a.group) store_out_row<CPT>(orow, acc, 1.f / ll);
      } else {
        const int first_c = owner_of(bg * TB, T, G);
        const int my_slot = (beg / TB == bg) ? 0 : 1;
        float* rec = a.partials + (int64_t)(c * 2 + my_slot) * (16 * (D + 2));
#pragma unroll
        for (int j = 0; j < CPT; ++j) rec[row * (D + 2) + cl + 16 * j] = acc[j];
        if ((ctid & 15) == 0) { rec[row * (D + 2) + D] = mm; rec[row * (D + 2) + D + 1] = ll; }
        __threadfence();
        bar_sync(1, kDecWarps * 32);
        if (ctid == 0) {
          const int old = atomicAdd(&a.tickets[bg], 1);
          *last_flag = (old == nseg - 1) ? 1 : 0;
        }
        bar_sync(1, kDecWarps * 32);
        if (*last_flag) {
          __threadfence();
          float M2 = -INFINITY;
          for (int sgi = 0; sgi < nseg; ++sgi) {
            const int cc = first_c + sgi;
            const int slot = (range_begin(cc, T, G) / TB == bg) ? 0 : 1;
            const float* src = a.partials + (int64_t)(cc * 2 + slot) * (16 * (D + 2));
            M2 = fmaxf(M2, __ldcg(&src[row * (D + 2) + D]));
          }
          float L2 = 0.f, acc2[CPT];
#pragma unroll
          for (int j = 0; j < CPT; ++j) acc2[j] = 0.f;
          for (int sgi = 0; sgi < nseg; ++sgi) {
            const int cc = first_c + sgi;
            const int slot = (range_begin(cc, T, G) / TB == bg) ? 0 : 1;
            const float* src = a.partials + (int64_t)(cc * 2 + slot) * (16 * (D + 2));
            const float ms = __ldcg(&src[row * (D + 2) + D]);
            if (ms == -INFINITY) continue;
            const float sc = exp2f(ms - M2);
            L2 += __ldcg(&src[row * (D + 2) + D + 1]) * sc;
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc2[j] += __ldcg(&src[row * (D + 2) + cl + 16 * j]) * sc;
          }
          if (row < a.group) store_out_row<CPT>(orow, acc2, 1.f / L2);
          if (ctid == 0) a.tickets[bg] = 0;
        }
      }
      bar_sync(1, kDecWarps * 32);  // smem (q, comb, flag) reused by the next segment
      if (any_dead) break;
      u0 = seg_end;
    }
  }
  __syncthreads();
}

// ============================================================================
// prefill (causal within each sequence)
// ============================================================================
constexpr int kPreThreads = 128;
constexpr int kPreStages = 2;

template <int D>
struct PreSmem {
  static constexpr int kTileBytes = (D / 64) * 8192;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kQRow = D * 2 + 16;
  static constexpr size_t bytes() {
    return 1024 + (size_t)kPreStages * kStageBytes + 64 * kQRow + 128;
  }
};

template <int D>
__global__ void __launch_bounds__(kPreThreads) attn_prefill_kernel(const __grid_constant__ AttnArgs a) {
  using L = PreSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem;
  uint8_t* sQ = tiles + kPreStages * L::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sQ + 64 * L::kQRow);
  int* flags = reinterpret_cast<int*>(full + kPreStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  pdl_wait();  // q and the cache were written by the preceding kernels
  const int b = blockIdx.z, h = blockIdx.y;
  const int n_qb = gridDim.x;
  const int qb = n_qb - 1 - blockIdx.x;  // longest blocks first
  const int t0 = a.seq_start[b], t1 = a.seq_start[b + 1];
  const int q0 = t0 + qb * 64;
  if (q0 >= t1) return;
  const int nrows = min(64, t1 - q0);
  const int g = h / a.group;
  const int slice = ((g / a.kv_r) * a.n_seqs + b) * a.kv_r + (g % a.kv_r);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPreStages; ++i) mbar_init(&full[i], 1);
    fence_barrier_init();
    fence_proxy_async_smem();
    int mx = 0;
    for (int i = 0; i < nrows; ++i) mx = max(mx, a.positions[q0 + i]);
    flags[0] = mx;
  }
  // stage q rows
  for (int i = threadIdx.x; i < 64 * (D / 8); i += kPreThreads) {
    const int row = i / (D / 8), ch = i % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < nrows) v = *reinterpret_cast<const uint4*>(a.q + (int64_t)(q0 + row) * a.ld_q + (int64_t)h * D + ch * 8);
    *reinterpret_cast<uint4*>(sQ + row * L::kQRow + ch * 16) = v;
  }
  __syncthreads();
  const int max_pos = min(flags[0], a.l_max - 1);
  const int n_tiles = max_pos / kKeyTile + 1;
  const uint64_t pol = policy_evict_last();
  auto issue = [&](int tile) {
    const int s = tile % kPreStages;
    uint8_t* kt = tiles + s * L::kStageBytes;
    mbar_arrive_expect_tx(&full[s], L::kStageBytes);
#pragma unroll
    for (int bx = 0; bx < D / 64; ++bx) {
      tma_load_3d(kt + bx * 8192, &a.tmK, &full[s], bx * 64, tile * kKeyTile, slice, pol);
      tma_load_3d(kt + L::kTileBytes + bx * 8192, &a.tmV, &full[s], bx * 64, tile * kKeyTile, slice, pol);
    }
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < min(kPreStages, n_tiles); ++i) issue(i);

  uint32_t qa[D / 16][4];
  load_q_frags<D>(smem_u32(sQ) + warp * 16 * L::kQRow, L::kQRow, qa);
  const int r0 = warp * 16 + (lane >> 2);
  int lim[2];
  lim[0] = r0 < nrows ? a.positions[q0 + r0] : -1;
  lim[1] = r0 + 8 < nrows ? a.positions[q0 + r0 + 8] : -1;
  int warp_max = max(lim[0], lim[1]);
  warp_max = max(warp_max, __shfl_xor_sync(0xffffffffu, warp_max, 4));
  warp_max = max(warp_max, __shfl_xor_sync(0xffffffffu, warp_max, 8));
  warp_max = max(warp_max, __shfl_xor_sync(0xffffffffu, warp_max, 16));
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int nt = 0; nt < D / 8; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[nt][i] = 0.f;

  bool alive = true;
  for (int tile = 0; tile < n_tiles; ++tile) {
    const int s = tile % kPreStages;
    bool ok = true;
    if (lane == 0) ok = mbar_wait(&full[s], (tile / kPreStages) & 1, a.status);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    const bool dead = __syncthreads_or(!ok);
    if (dead) { alive = false; break; }
    const int key0 = tile * kKeyTile;
    if (key0 <= warp_max) {
      const uint32_t st = smem_u32(tiles + s * L::kStageBytes);
      attn_tile<D, 8>(qa, st, st + L::kTileBytes, 0, key0, lim, a.scale_log2, m, l, o);
    }
    __syncthreads();
    if (threadIdx.x == 0 && tile + kPreStages < n_tiles) issue(tile + kPreStages);
  }
  if (!alive) {
    // let copies in flight land before the CTA exits
    if (threadIdx.x == 0)
      for (int tile = 0; tile < n_tiles; ++tile)
        mbar_wait(&full[tile % kPreStages], (tile / kPreStages) & 1, a.status);
    __syncthreads();
    return;
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 1);
    l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 2);
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int row = r0 + hh * 8;
    if (row >= nrows) continue;
    const float inv = 1.f / l[hh];
    uint16_t* orow = a.o + (int64_t)(q0 + row) * a.ld_o + (int64_t)h * D;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) {
      const int col = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<uint32_t*>(orow + col) = pack2(o[nt][hh * 2] * inv, o[nt][hh * 2 + 1] * inv);
    }
  }
}

// ============================================================================
// host launchers
// ============================================================================
template <int D>
static cudaError_t launch_decode_t(const AttnArgs& a, cudaStream_t st) {
  const size_t smem = DecSmem<D>::bytes(0);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_k(attn_decode_kernel<D>, dim3(a.grid), dim3(kDecThreads), smem, st, a);
}

template <int D>
static cudaError_t launch_prefill_t(const AttnArgs& a, int n_qb, cudaStream_t st) {
  const size_t smem = PreSmem<D>::bytes();
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  dim3 grid(n_qb, a.n_heads, a.n_seqs);
  return launch_k(attn_prefill_kernel<D>, grid, dim3(kPreThreads), smem, st, a);
}

cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t st) {
  return a.head_dim == 128 ? launch_decode_t<128>(a, st) : launch_decode_t<64>(a, st);
}

cudaError_t launch_attn_prefill(const AttnArgs& a, int n_qb, cudaStream_t st) {
  return a.head_dim == 128 ? launch_prefill_t<128>(a, n_qb, st) : launch_prefill_t<64>(a, n_qb, st);
}

size_t attn_decode_partial_floats(int head_dim) { return 16 * (size_t)(head_dim + 2); }

}  // namespace tpk

namespace tpk {
size_t attn_decode_smem_bytes(int head_dim) {
  return head_dim == 128 ? DecSmem<128>::bytes(0) : DecSmem<64>::bytes(0);
}
}  // namespace tpk
