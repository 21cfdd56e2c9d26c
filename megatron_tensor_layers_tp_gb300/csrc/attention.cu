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
#include "rms.cuh"

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
  // from the one it wants).  The host takes the largest even count up to
  // kMaxStages that fits next to the combine buffer.
  static constexpr int kMaxStages = 8;
  // combine rows: O, m, l of every warp for each of the KV head's query rows
  // (n_heads / n_kv of the 16 MMA rows); the pitch keeps the two rows a warp
  // reads at once 18 banks apart (16 lanes per row, columns lane + 16 j)
  static constexpr int kCombLd = D + 18;
  struct Layout {
    size_t tiles, sq, comb, bars, misc, knew, total;
  };
  __host__ __device__ static constexpr Layout layout(int stages, int rows) {
    Layout L{};
    size_t off = 0;
    L.tiles = off;
    off += (size_t)stages * kStageBytes;
    L.sq = off;
    off += 16 * kQRow;
    L.comb = off;  // also the deferred qkv's unscaled sums before the tile loop
    off += (size_t)kDecWarps * rows * kCombLd * 4;
    off = (off + 15) & ~(size_t)15;
    L.bars = off;
    off += 2 * kMaxStages * 8;
    L.misc = off;
    off += 64;     // flag, the prologue's per-warp sums, the token's 1/rms
    L.knew = off;
    off += 2 * D * 4;
    L.total = off + 1024;
    return L;
  }
  __host__ __device__ static constexpr size_t bytes(int stages, int rows) {
    return layout(stages, rows).total;
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

// The 1/rms of token b for the RMSNorm folded into the qkv weights, by the
// 256 consumer threads (red: 8 floats of shared scratch): from the token's
// hidden row (norm_mode 1), from the partial sums of squares the kernel that
// wrote the row left (norm_mode 2), or 1 (norm_mode 0: the GEMM read the
// normalised rows).  Reads only what earlier kernels wrote, so it may run
// before the dependency wait on the qkv GEMM.
template <int D>
__device__ float token_rs(const AttnArgs& a, int b, float* red) {
  const int ctid = threadIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int NT = kDecWarps * 32;
  if (a.norm_mode == 0) return 1.f;
  float ss = 0.f;
  if (a.norm_mode == 1) {
    const uint4* xr = reinterpret_cast<const uint4*>(a.norm_src + (int64_t)b * a.norm_ld);
    const int nv = a.norm_width >> 3;
    uint4 hv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      hv[k] = ctid + k * NT < nv ? __ldcg(xr + ctid + k * NT) : make_uint4(0, 0, 0, 0);
    auto add_sq = [&](const uint4& p) {
      const uint32_t w4[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = __uint_as_float(w4[q] << 16), hi = __uint_as_float(w4[q] & 0xFFFF0000u);
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
      }
    };
#pragma unroll
    for (int k = 0; k < 4; ++k) add_sq(hv[k]);
    for (int v = ctid + 4 * NT; v < nv; v += NT) add_sq(__ldcg(xr + v));
  } else {
    const float4* pr = reinterpret_cast<const float4*>(a.norm_partials + (int64_t)b * a.norm_slots);
    for (int i4 = ctid; i4 < (a.norm_slots >> 2); i4 += NT) {
      const float4 p = __ldcg(pr + i4);
      ss += (p.x + p.y) + (p.z + p.w);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  bar_sync(1, NT);
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kDecWarps; ++w) t += red[w];
  bar_sync(1, NT);  // red is reused
  return 1.0f / sqrtf(t / (float)a.norm_width + a.norm_eps);
}

// Deferred qkv epilogue of one (sequence b, KV head g): the qkv GEMM left
// stream-K pieces of fp32 accumulators; sum the pieces of every q row of the
// group's query heads and of the K and V rows of head g at token b, in K
// order, then do what the GEMM epilogue would have done: scale by the token's
// 1/rms rs (the norm weight is folded into the weights), add the bias, rotate
// the RoPE pairs (shard rows 2i, 2i+1 hold features i and i + d/2 of a Q or K
// head), round to bf16.  q goes to the CTA's query rows sQ, k and v to knew /
// vnew; `write` also stores the new K/V row into the cache at the token's
// position.  All 256 consumer threads take part, two items (row pairs) per
// thread per round; every load of a round (the pieces, the RoPE factors, the
// biases) is issued before any is used, so a round costs one trip to L2.
template <int D>
__device__ void qkv_from_pieces(const AttnArgs& a, int b, int g, int pos, float rs, bool write,
                                uint8_t* sQ, int qrow_bytes, float* knew, float* vnew) {
  const int ctid = threadIdx.x;
  constexpr int NT = kDecWarps * 32;
  constexpr int kMaxPieces = 6;  // pieces loaded together per row pair
  const int half = D / 2, nq = a.q_per_rank, kvr = a.kv_r;
  const int kv_rank = a.kv_replicas == 1 ? g / kvr : g * a.kv_replicas;  // first holder of head g
  const int kv_local = g % kvr;
  const int n_items = (a.group + 2) * half;
  const bool pos_ok = pos >= 0 && pos < a.l_max;
  // (32-bit piece arithmetic: the host keeps pc_total * pc_grid below 2^31;
  // the divisions by pc_total, pc_grid and q_per_rank are multiply-shifts)
  const int T = static_cast<int>(a.pc_total), Gp = a.pc_grid, K = a.pc_k;
  const int64_t piece = (int64_t)a.pc_bn * 128;
  const float* pcb = a.pc + (int64_t)b * 128;
  for (int base_it = 0; base_it < n_items; base_it += 2 * NT) {
    int kind[2], hq[2], ii[2], r[2], lr[2], c0[2], ns[2], sl0[2];
    bool have[2];
    float2 pcs[2][kMaxPieces], cs[2], bs[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int it = base_it + u * NT + ctid;
      have[u] = it < n_items;
      const int itc = have[u] ? it : 0;
      if (itc < a.group * half) {
        kind[u] = 0;
        hq[u] = itc / half;
        ii[u] = itc - hq[u] * half;
        const int j = g * a.group + hq[u];
        r[u] = static_cast<int>(fast_div(static_cast<uint32_t>(j), a.pc_div_q));
        lr[u] = (j - r[u] * nq) * D + 2 * ii[u];
      } else {
        kind[u] = itc < (a.group + 1) * half ? 1 : 2;
        hq[u] = 0;
        ii[u] = itc - (a.group + kind[u] - 1) * half;
        r[u] = kv_rank;
        lr[u] = (nq + (kind[u] == 2 ? kvr : 0) + kv_local) * D + 2 * ii[u];
      }
      const int ts = r[u] * a.pc_a_tiles + lr[u] / 128;
      // owner of the tile's first step, pieces of the tile, slot of the first piece
      c0[u] = static_cast<int>(fast_div(static_cast<uint32_t>((ts * K + 1) * Gp - 1), a.pc_div_total));
      ns[u] = static_cast<int>(fast_div(static_cast<uint32_t>(((ts + 1) * K) * Gp - 1), a.pc_div_total)) -
              c0[u] + 1;
      sl0[u] = static_cast<int>(fast_div(static_cast<uint32_t>(c0[u] * T), a.pc_div_grid)) == ts * K ? 0 : 1;
      const float* src = pcb + lr[u] % 128;
#pragma unroll
      for (int q = 0; q < kMaxPieces; ++q)
        pcs[u][q] = have[u] && q < ns[u]
                        ? __ldcg(reinterpret_cast<const float2*>(
                              src + ((int64_t)(c0[u] + q) * 2 + (q == 0 ? sl0[u] : 0)) * piece))
                        : make_float2(0.f, 0.f);
      cs[u] = (have[u] && kind[u] != 2 && pos_ok) ? __ldg(a.rope + (int64_t)pos * half + ii[u])
                                                  : make_float2(1.f, 0.f);
      bs[u] = make_float2(0.f, 0.f);
      if (have[u] && a.qkv_bias) {
        const uint16_t* bb = a.qkv_bias + (int64_t)r[u] * a.nqkv_r + lr[u];
        bs[u] = make_float2(bf16_to_f(bb[0]), bf16_to_f(bb[1]));
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!have[u]) continue;
      float2 x = pcs[u][0];
#pragma unroll
      for (int q = 1; q < kMaxPieces; ++q)
        if (q < ns[u]) { x.x += pcs[u][q].x; x.y += pcs[u][q].y; }
      // a tile cut in more pieces than were loaded together (small grids)
      const float* src = pcb + lr[u] % 128;
      for (int q = kMaxPieces; q < ns[u]; ++q) {
        const float2 p2 = __ldcg(reinterpret_cast<const float2*>(src + (int64_t)(c0[u] + q) * 2 * piece));
        x.x += p2.x;
        x.y += p2.y;
      }
      x.x = x.x * rs + bs[u].x;
      x.y = x.y * rs + bs[u].y;
      const int i = ii[u];
      if (kind[u] == 2) {
        // V rows in natural order: features 2i and 2i + 1
        const uint16_t v0 = f_to_bf16(x.x), v1 = f_to_bf16(x.y);
        vnew[2 * i] = bf16_to_f(v0);
        vnew[2 * i + 1] = bf16_to_f(v1);
        if (write && pos_ok) {
          uint16_t* dst = a.v_cache + (int64_t)(g / kvr) * a.kv_copy_stride +
                          (((int64_t)b * kvr + kv_local) * a.l_max + pos) * D;
          *reinterpret_cast<uint32_t*>(dst + 2 * i) = (uint32_t)v0 | ((uint32_t)v1 << 16);
        }
        continue;
      }
      const uint16_t y1 = f_to_bf16(x.x * cs[u].x - x.y * cs[u].y);  // feature i
      const uint16_t y2 = f_to_bf16(x.y * cs[u].x + x.x * cs[u].y);  // feature i + d/2
      if (kind[u] == 0) {
        uint16_t* qr = reinterpret_cast<uint16_t*>(sQ + hq[u] * qrow_bytes);
        qr[i] = y1;
        qr[i + half] = y2;
      } else {
        knew[i] = bf16_to_f(y1);
        knew[i + half] = bf16_to_f(y2);
        if (write && pos_ok) {
          uint16_t* dst = a.k_cache + (int64_t)(g / kvr) * a.kv_copy_stride +
                          (((int64_t)b * kvr + kv_local) * a.l_max + pos) * D;
          dst[i] = y1;
          dst[i + half] = y2;
        }
      }
    }
  }
}

// Score of the new key against query row `row` (log2 units): the row's 16
// threads (one half-warp) each take features cl, cl + 16, ... and combine.
template <int D>
__device__ __forceinline__ float new_key_score(const uint8_t* sQ, int qrow_bytes, const float* knew,
                                               int row, int cl, float scale_log2) {
  const uint16_t* qr = reinterpret_cast<const uint16_t*>(sQ + row * qrow_bytes);
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < D / 16; ++j) s = fmaf(bf16_to_f(qr[cl + 16 * j]), knew[cl + 16 * j], s);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s * scale_log2;
}


// TQ: at most 8 query rows per KV head, taken on the MMA N side (attn_tile_t).
// N32: AttnArgs::idx32 (the schedule's divisions as multiply-shifts).
template <int D, bool TQ, bool N32>
__global__ void __launch_bounds__(kDecThreads, 1) attn_decode_kernel(const __grid_constant__ AttnArgs a) {
  using L = DecSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const typename L::Layout LY = L::layout(a.stages, a.group);
  uint8_t* tiles = smem + LY.tiles;
  uint8_t* sQ = smem + LY.sq;
  float* comb = reinterpret_cast<float*>(smem + LY.comb);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + LY.bars);
  uint64_t* empty = full + L::kMaxStages;
  int* last_flag = reinterpret_cast<int*>(smem + LY.misc);
  float* red = reinterpret_cast<float*>(smem + LY.misc + 16);  // 8 floats
  float* knew = reinterpret_cast<float*>(smem + LY.knew);       // [D]
  float* vnew = knew + D;                                        // [D]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.stages;
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
  // the schedule's divisions (by total_units T, the grid G, tiles_per_bg TB
  // and n_kv): multiply-shifts when every index fits 32 bits
  auto start_of = [&](int cc) -> int64_t {
    if constexpr (N32) return fast_div(static_cast<uint32_t>(cc * T), a.div_grid);
    return range_begin(cc, T, G);
  };
  auto owner = [&](int64_t x) -> int {
    if constexpr (N32) return static_cast<int>(fast_div(static_cast<uint32_t>((x + 1) * G - 1), a.div_units));
    return owner_of(x, T, G);
  };
  auto pair_of = [&](int64_t u) -> int64_t {
    if constexpr (N32) return fast_div(static_cast<uint32_t>(u), a.div_tb);
    return u / TB;
  };
  auto seq_of = [&](int64_t bg) -> int {
    if constexpr (N32) return static_cast<int>(fast_div(static_cast<uint32_t>(bg), a.div_kv));
    return static_cast<int>(bg / a.n_kv);
  };
  const int64_t beg = start_of(c), end = start_of(c + 1);

  if (warp == kDecWarps) {
    // producer
    if (lane == 0) {
      uint32_t n = 0;
      // (sequence, KV head, tile) of unit u, walked incrementally
      const int64_t bg0 = pair_of(beg);
      int tile = static_cast<int>(beg - bg0 * TB);
      int b = seq_of(bg0), g = static_cast<int>(bg0 - (int64_t)b * a.n_kv);
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
      while (u < end && n < (uint32_t)S &&
             (a.qkv_pieces || (tile + 1) * kKeyTile <= a.positions[b])) {
        issue(n);
        ++n;
        if (++u < end) advance();
      }
      // The next kL2AheadUnits of this CTA's cache tiles go to L2 now, while
      // the stages above wait for the prologue (at most 12 x 32 KB per CTA,
      // well inside L2 over all SMs): a 64-key K or V tile is 16 KB
      // contiguous in the cache ([copy][sequence][head][position][d]).  A
      // prefetch only warms L2, the point of coherence, so rows this step
      // still writes are read correctly later all the same.
      {
        constexpr int kL2AheadUnits = 12;
        int pt = tile, pg = g, pb = b;
        for (int64_t v = u; v < end && v < u + kL2AheadUnits; ++v) {
          const int slice = ((pg / a.kv_r) * a.n_seqs + pb) * a.kv_r + (pg % a.kv_r);
          const int p0 = pt * kKeyTile;
          const int rows = min(kKeyTile, a.l_max - p0);
          if (rows > 0) {
            const int64_t off = ((int64_t)slice * a.l_max + p0) * D;
            l2_prefetch_bulk(a.k_cache + off, static_cast<uint32_t>(rows) * D * 2);
            l2_prefetch_bulk(a.v_cache + off, static_cast<uint32_t>(rows) * D * 2);
          }
          if (++pt == TB) {
            pt = 0;
            if (++pg == a.n_kv) { pg = 0; ++pb; }
          }
        }
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
    const int ctid = threadIdx.x;  // 0..255
    // The first segment's position and, with the deferred qkv, its token's
    // 1/rms: they read only the batch and the hidden state, which every kernel
    // before the qkv GEMM has finished writing when this kernel starts (the
    // GEMM signals its dependents after its own wait), so they overlap the
    // GEMM's end.
    int first_pos = 0;
    float first_rs = 1.f;
    if (beg < end) {
      const int b0 = seq_of(pair_of(beg));
      first_pos = a.positions[b0];
      if (a.qkv_pieces) first_rs = token_rs<D>(a, b0, red);
    }
    pdl_wait();  // q and the newest cache rows were written by the preceding kernels
    uint32_t n_base = 0;           // CTA-local index of the segment's first unit
    bool alive = true;
    for (int64_t u0 = beg; u0 < end;) {
      const int64_t bg = pair_of(u0);
      const int64_t seg_end = min(end, (bg + 1) * TB);
      const int len = static_cast<int>(seg_end - u0);
      const int tile0 = static_cast<int>(u0 - bg * TB);
      const int b = seq_of(bg), g = static_cast<int>(bg - (int64_t)b * a.n_kv);
      const bool first_seg = u0 == beg;
      const int pos = first_seg ? first_pos : a.positions[b];
      // stage the group's query rows (16 rows, zero beyond the group)
      for (int i = ctid; i < 16 * (D / 8); i += kDecWarps * 32) {
        const int row = i / (D / 8), ch = i % (D / 8);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < a.group && !a.qkv_pieces)
          v = *reinterpret_cast<const uint4*>(a.q + (int64_t)b * a.ld_q +
                                              (int64_t)(g * a.group + row) * D + ch * 8);
        *reinterpret_cast<uint4*>(sQ + row * L::kQRow + ch * 16) = v;
      }
      bar_sync(1, kDecWarps * 32);
      if (a.qkv_pieces) {
        // q, and the new token's k and v, from the qkv GEMM's pieces; the
        // pair's first CTA stores the new K/V row in the cache
        const bool writer = owner(bg * TB) == c;
        const float rs = first_seg ? first_rs : token_rs<D>(a, b, red);
        qkv_from_pieces<D>(a, b, g, pos, rs, writer, sQ, L::kQRow, knew, vnew);
        bar_sync(1, kDecWarps * 32);
      }
      // Q fragments: A of 16 query rows, or (TQ) B of Q^T over 8 query rows
      constexpr int QR = TQ ? 2 : 4;   // registers per 16-wide d step
      constexpr int ON = TQ ? D / 16 : D / 8;  // accumulator fragments
      uint32_t qa[D / 16][QR];
      if constexpr (TQ) load_qt_frags<D>(smem_u32(sQ), L::kQRow, qa);
      else load_q_frags<D>(smem_u32(sQ), L::kQRow, qa);
      float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
      float o[ON][4];
#pragma unroll
      for (int nt = 0; nt < ON; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[nt][i] = 0.f;
      // with the deferred qkv the new key is merged at the end, not read from the cache
      const int last_key = a.qkv_pieces ? pos - 1 : pos;
      const int lim[2] = {last_key, last_key};
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
        if (key0 <= last_key) {
          const uint32_t st = smem_u32(tiles + s * L::kStageBytes);
          if constexpr (TQ) {
            static_assert(kWarpKeys == 16, "one 16-key step per warp and tile");
            attn_tile_t<D>(qa, st, st + L::kTileBytes, wq * kWarpKeys, key0, last_key,
                           a.scale_log2, m, l, o);
          } else {
            attn_tile<D, kWarpKeys / 8>(qa, st, st + L::kTileBytes, wq * kWarpKeys, key0, lim,
                                        a.scale_log2, m, l, o);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      n_base += len;
      // each query row's l: the row's threads hold shares of it (TQ: the 8
      // lanes of a column; otherwise the 4 lanes of a row)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if constexpr (TQ) {
          l[h] += __shfl_xor_sync(0xffffffffu, l[h], 4);
          l[h] += __shfl_xor_sync(0xffffffffu, l[h], 8);
          l[h] += __shfl_xor_sync(0xffffffffu, l[h], 16);
        } else {
          l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
          l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
        }
      }
      // combine: every warp's (m, l, O) meets the others in smem
      // (only the KV head's query rows: rows >= group hold no query)
      constexpr int CL = L::kCombLd;
      const int GR = a.group;
      float* cw = comb + warp * GR * CL;
      if constexpr (TQ) {
        // o[dt]: O^T rows (features) 16 dt + lane/4 and + 8, query columns
        // 2 (lane % 4) and + 1
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int q = (lane & 3) * 2 + c;
          if (q >= GR) continue;
#pragma unroll
          for (int dt = 0; dt < D / 16; ++dt) {
            cw[q * CL + dt * 16 + (lane >> 2)] = o[dt][c];
            cw[q * CL + dt * 16 + 8 + (lane >> 2)] = o[dt][2 + c];
          }
          if ((lane >> 2) == 0) { cw[q * CL + D] = m[c]; cw[q * CL + D + 1] = l[c]; }
        }
      } else {
        const int r0 = lane >> 2;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = r0 + hh * 8;
          if (r >= GR) continue;
#pragma unroll
          for (int nt = 0; nt < D / 8; ++nt) {
            const int col = nt * 8 + (lane & 3) * 2;
            *reinterpret_cast<float2*>(cw + r * CL + col) =
                make_float2(o[nt][hh * 2], o[nt][hh * 2 + 1]);
          }
          if ((lane & 3) == 0) { cw[r * CL + D] = m[hh]; cw[r * CL + D + 1] = l[hh]; }
        }
      }
      const bool any_dead = bar_sync_or(1, kDecWarps * 32, !alive);
      const int nseg = owner((bg + 1) * TB - 1) - owner(bg * TB) + 1;
      if (TQ && nseg == 1) {
        // A whole pair with at most 8 query rows: all 256 threads on the real
        // rows (64 threads per row for up to 4 rows, 32 for up to 8), 2-4
        // columns each, instead of 16 threads on each of 16 rows.  The new
        // key's score of each row comes first (16 threads per row).
        if (a.qkv_pieces) {
          const float sn = new_key_score<D>(sQ, L::kQRow, knew, ctid >> 4, ctid & 15, a.scale_log2);
          if ((ctid & 15) == 0 && (ctid >> 4) < 8) red[ctid >> 4] = sn;
          bar_sync(1, kDecWarps * 32);
        }
        const int tpr = GR <= 4 ? (kDecWarps * 32) / 4 : (kDecWarps * 32) / 8;
        const int row = ctid / tpr, cl = ctid % tpr;
        constexpr int kMaxCpt = D / 32;  // columns per thread at 32 threads per row
        const int cpt = D / tpr;
        if (row < GR) {
          float mm = -INFINITY;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, comb[(w * GR + row) * CL + D]);
          float ll = 0.f, acc[kMaxCpt];
#pragma unroll
          for (int j = 0; j < kMaxCpt; ++j) acc[j] = 0.f;
#pragma unroll
          for (int w = 0; w < kDecWarps; ++w) {
            const float* cr = comb + (w * GR + row) * CL;
            const float mw = cr[D];
            if (mw == -INFINITY) continue;
            const float sc = exp2f(mw - mm);
            ll += cr[D + 1] * sc;
#pragma unroll
            for (int j = 0; j < kMaxCpt; ++j)
              if (j < cpt) acc[j] += cr[cl + tpr * j] * sc;
          }
          if (a.qkv_pieces) {
            // the new key's state (score, weight 1, value vnew) joins in
            const float s_new = red[row];
            const float mn = fmaxf(mm, s_new);
            const float so = mm == -INFINITY ? 0.f : exp2f(mm - mn);
            const float sw = exp2f(s_new - mn);
            ll = ll * so + sw;
#pragma unroll
            for (int j = 0; j < kMaxCpt; ++j)
              if (j < cpt) acc[j] = acc[j] * so + vnew[cl + tpr * j] * sw;
          }
          const float inv = 1.f / ll;
          uint16_t* orow = a.o + (int64_t)b * a.ld_o + (int64_t)(g * a.group + row) * D + cl;
#pragma unroll
          for (int j = 0; j < kMaxCpt; ++j)
            if (j < cpt) orow[tpr * j] = f_to_bf16(acc[j] * inv);
        }
      } else {
        // 256 threads: row = ctid / 16, D/16 columns each (8 for D = 128): columns
        // cl, cl + 16, ... so that a row's 16 threads read 16 consecutive floats
        constexpr int CPT = D / 16;
        const int row = ctid >> 4, cl = ctid & 15;
        const float s_new =
            a.qkv_pieces ? new_key_score<D>(sQ, L::kQRow, knew, row, cl, a.scale_log2) : -INFINITY;
        const int crow = row < GR ? row : 0;  // rows >= group: computed, never stored
        float mm = -INFINITY;
  #pragma unroll
        for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, comb[(w * GR + crow) * CL + D]);
        float ll = 0.f, acc[CPT];
  #pragma unroll
        for (int j = 0; j < CPT; ++j) acc[j] = 0.f;
  #pragma unroll 2
        for (int w = 0; w < kDecWarps; ++w) {
          const float* cr = comb + (w * GR + crow) * CL;
          const float mw = cr[D];
          if (mw == -INFINITY) continue;
          const float sc = exp2f(mw - mm);
          ll += cr[D + 1] * sc;
  #pragma unroll
          for (int j = 0; j < CPT; ++j) acc[j] += cr[cl + 16 * j] * sc;
        }
        uint16_t* orow = a.o + (int64_t)b * a.ld_o + (int64_t)(g * a.group + row) * D + cl;
        // the new key's state (score s_new, weight 1, value vnew) joins the
        // pair's final combination
        auto add_new_key = [&](float& m_, float& l_, float (&o_)[CPT]) {
          const float mn = fmaxf(m_, s_new);
          const float so = m_ == -INFINITY ? 0.f : exp2f(m_ - mn);
          const float sn = exp2f(s_new - mn);
          l_ = l_ * so + sn;
  #pragma unroll
          for (int j = 0; j < CPT; ++j) o_[j] = o_[j] * so + vnew[cl + 16 * j] * sn;
          m_ = mn;
        };
        if (nseg == 1) {
          if (a.qkv_pieces) add_new_key(mm, ll, acc);
          if (row < a.group) store_out_row<CPT>(orow, acc, 1.f / ll);
        } else {
          const int first_c = owner(bg * TB);
          const int my_slot = (pair_of(beg) == bg) ? 0 : 1;
          float* rec = a.partials + (int64_t)(c * 2 + my_slot) * (16 * (D + 2));
  #pragma unroll
          for (int j = 0; j < CPT; ++j) rec[row * (D + 2) + cl + 16 * j] = acc[j];
          if ((ctid & 15) == 0) { rec[row * (D + 2) + D] = mm; rec[row * (D + 2) + D + 1] = ll; }
          // publish the record and take the pair's ticket: one thread fences
          // for the CTA around the increment (the barriers carry the ordering)
          bar_sync(1, kDecWarps * 32);
          if (ctid == 0) {
            fence_acq_rel_gpu();
            const int old = atomicAdd(&a.tickets[bg], 1);
            fence_acq_rel_gpu();
            *last_flag = (old == nseg - 1) ? 1 : 0;
          }
          bar_sync(1, kDecWarps * 32);
          if (*last_flag) {
            float M2 = -INFINITY;
            for (int sgi = 0; sgi < nseg; ++sgi) {
              const int cc = first_c + sgi;
              const int slot = (pair_of(start_of(cc)) == bg) ? 0 : 1;
              const float* src = a.partials + (int64_t)(cc * 2 + slot) * (16 * (D + 2));
              M2 = fmaxf(M2, __ldcg(&src[row * (D + 2) + D]));
            }
            float L2 = 0.f, acc2[CPT];
  #pragma unroll
            for (int j = 0; j < CPT; ++j) acc2[j] = 0.f;
            for (int sgi = 0; sgi < nseg; ++sgi) {
              const int cc = first_c + sgi;
              const int slot = (pair_of(start_of(cc)) == bg) ? 0 : 1;
              const float* src = a.partials + (int64_t)(cc * 2 + slot) * (16 * (D + 2));
              const float ms = __ldcg(&src[row * (D + 2) + D]);
              if (ms == -INFINITY) continue;
              const float sc = exp2f(ms - M2);
              L2 += __ldcg(&src[row * (D + 2) + D + 1]) * sc;
  #pragma unroll
              for (int j = 0; j < CPT; ++j) acc2[j] += __ldcg(&src[row * (D + 2) + cl + 16 * j]) * sc;
            }
            if (a.qkv_pieces) add_new_key(M2, L2, acc2);
            if (row < a.group) store_out_row<CPT>(orow, acc2, 1.f / L2);
            if (ctid == 0) a.tickets[bg] = 0;
          }
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

// Shared memory is the K/V ring alone (the Q fragments go straight from
// global memory to registers), so that three CTAs fit on an SM: the kernel is
// latency-bound (each CTA walks at most a few key tiles), and with 32-key
// score sub-tiles its registers also allow three.
template <int D>
struct PreSmem {
  static constexpr int kTileBytes = (D / 64) * 8192;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr size_t bytes() { return 1024 + (size_t)kPreStages * kStageBytes + 128; }
};

template <int D>
__global__ void __launch_bounds__(kPreThreads) attn_prefill_kernel(const __grid_constant__ AttnArgs a) {
  using L = PreSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(tiles + kPreStages * L::kStageBytes);
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

  // A fragments of the warp's 16 query rows (m16n8k16 layout: rows r0 and
  // r0 + 8, column pairs c2 and c2 + 8 of every 16-wide K step)
  const int r0 = warp * 16 + (lane >> 2);
  uint32_t qa[D / 16][4];
  {
    const int c2 = (lane & 3) * 2;
    const uint16_t* q_lo = a.q + (int64_t)(q0 + r0) * a.ld_q + (int64_t)h * D + c2;
    const uint16_t* q_hi = q_lo + 8 * a.ld_q;
    const bool v_lo = r0 < nrows, v_hi = r0 + 8 < nrows;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      qa[kk][0] = v_lo ? *reinterpret_cast<const uint32_t*>(q_lo + kk * 16) : 0u;
      qa[kk][1] = v_hi ? *reinterpret_cast<const uint32_t*>(q_hi + kk * 16) : 0u;
      qa[kk][2] = v_lo ? *reinterpret_cast<const uint32_t*>(q_lo + kk * 16 + 8) : 0u;
      qa[kk][3] = v_hi ? *reinterpret_cast<const uint32_t*>(q_hi + kk * 16 + 8) : 0u;
    }
  }
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
      // two 32-key halves: fewer live score registers than one 64-key pass
      attn_tile<D, 4>(qa, st, st + L::kTileBytes, 0, key0, lim, a.scale_log2, m, l, o);
      if (key0 + 32 <= warp_max)
        attn_tile<D, 4>(qa, st, st + L::kTileBytes, 32, key0 + 32, lim, a.scale_log2, m, l, o);
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
template <int D, bool TQ, bool N32>
static cudaError_t launch_decode_tq(const AttnArgs& a, cudaStream_t st) {
  const size_t smem = DecSmem<D>::bytes(a.stages, a.group);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<D, TQ, N32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_k(attn_decode_kernel<D, TQ, N32>, dim3(a.grid), dim3(kDecThreads), smem, st, a);
}

// up to 8 query rows per KV head: query rows on the MMA N side
template <int D>
static cudaError_t launch_decode_t(const AttnArgs& a, cudaStream_t st) {
  if (a.idx32)
    return a.group <= 8 ? launch_decode_tq<D, true, true>(a, st) : launch_decode_tq<D, false, true>(a, st);
  return a.group <= 8 ? launch_decode_tq<D, true, false>(a, st) : launch_decode_tq<D, false, false>(a, st);
}

// The most K/V stages (even, at most DecSmem::kMaxStages) whose shared memory
// fits next to the combine buffer of `rows` query rows per KV head.
template <int D>
static int decode_stages_t(int rows) {
  for (int s = DecSmem<D>::kMaxStages; s >= 2; s -= 2)
    if (DecSmem<D>::bytes(s, rows) <= 227 * 1024) return s;
  return 0;
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

int attn_decode_stages(int head_dim, int rows) {
  return head_dim == 128 ? decode_stages_t<128>(rows) : decode_stages_t<64>(rows);
}

}  // namespace tpk

