// Prefill-orientation GEMM on CTA pairs (tcgen05 cta_group::2): tokens on the
// MMA M side in tiles of 256 rows, output features on N (BN), one tile per
// pair of SMs at a time.  The two CTAs of a cluster of 2 each load their own
// 128 token rows of A and half of the tile's BN weight rows of B; the MMA of
// the even CTA reads both CTAs' shared memory and accumulates each CTA's 128
// rows in that CTA's tensor memory.  Per SM and 64-wide K step that moves
// 16 KB of A and BN/2 x 128 B of B instead of 16 KB + BN x 128 B, and the
// smaller stages leave room for a deeper ring: the single-CTA prefill GEMM is
// bound by that operand traffic (about the same bytes per SM per second at
// every tile width), the pair halves the weight part of it.
//
// Work: whole tiles in waves, pair p taking tiles p, p + P, ... (P pairs).
// Roles: warp 0 loads (both CTAs), warp 1 of the even CTA issues the MMAs,
// the epilogue warps of both CTAs drain their accumulators through the fused
// epilogues of the single-CTA kernel.  The last tile's epilogue is not hidden
// behind a mainloop (with four warps it took 6-12 us of a 55-275 us GEMM), so
// eight warps run it, two per TMEM lane quadrant on alternate 16-column units
// (measured, same box: Llama-8B prefill o_proj 60.0 -> 58.3 us, gate_up and
// down 1 us less); the qkv epilogue keeps four (its stores then overlap the
// next tile's loads less: 81.7 -> 83.6 us with eight).  Barriers: the even
// CTA's full[s] counts both CTAs' bytes; each commit arrives on empty[s] /
// acc_full[b] of both CTAs; the even CTA's acc_empty[b] takes the epilogue
// warps of both.  Every wait is bounded.
#pragma once
#include "gemm_kernel.cuh"

namespace tpk {

template <int EPI>
constexpr int kPairEpiWarps = EPI == EPI_QKV ? 4 : 8;
template <int EPI>
constexpr int kPairThreads = (2 + kPairEpiWarps<EPI>) * 32;  // loader, MMA, epilogue warps

template <int EPI>
__global__ void __launch_bounds__(kPairThreads<EPI>, 1)
    gemm_pair_kernel(const __grid_constant__ GemmArgs a) {
  constexpr int NH = kPairEpiWarps<EPI> / 4;  // epilogue warps per TMEM lane quadrant
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int BN = a.BN, S = a.stages;
  const int HB = BN / 2;                 // weight rows of the tile in this CTA
  const int b_half_bytes = HB * 128;
  const uint32_t stage_tx = 2u * (kATileBytes + b_half_bytes);  // both CTAs' bytes
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * kATileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + S * b_half_bytes);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 2 * kPairEpiWarps<EPI>);  // the epilogue warps of both CTAs
    }
    mbar_init(drain, 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) { tma_prefetch_desc(&a.tmA); tma_prefetch_desc(&a.tmB); }
  if (warp == 1) { tmem_alloc_pair(tmem_slot, a.tmem_cols); tmem_relinquish_pair(); }
  tc_fence_before();
  // both CTAs' barriers exist before either CTA signals the other
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int P = gridDim.x >> 1, pair = blockIdx.x >> 1;
  const int64_t n_tiles = (int64_t)a.n_groups * a.a_tiles * a.b_tiles;
  const int K = a.k_slices * a.k_iters_slice;
  auto tile_coords = [&](int64_t tile, int& g, int& ia, int& ib) {
    ia = static_cast<int>(tile % a.a_tiles);
    const int64_t rest = tile / a.a_tiles;
    ib = static_cast<int>(rest % a.b_tiles);
    g = static_cast<int>(rest / a.b_tiles);
  };

  // as in the single-CTA kernel: the qkv projection signals its dependents
  // only after its own wait
  constexpr bool kLateSignal = EPI == EPI_QKV;
  if constexpr (!kLateSignal) pdl_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t polA = make_policy(a.a_policy), polB = make_policy(a.b_policy);
      const int kis = a.k_iters_slice;
      const uint32_t full0 = mapa_shared(smem_u32(full), 0);  // the even CTA's full[0]
      auto load = [&](int g, int ia, int ib, int ks, int kk, uint32_t s, bool weights) {
        const uint32_t bar = full0 + s * 8;
        if (weights) {  // 4-D map over the K-blocked shards: (0, row, K block, rank)
          const int sb = slice_of(a.b_slice_mode, g, ks);
          const int r0 = ib * BN + static_cast<int>(rank) * HB;
          tma_load_4d_pair(sB + s * b_half_bytes, &a.tmB, bar, 0, r0, kk, sb, polB);
        } else {
          const int sa = slice_of(a.a_slice_mode, g, ks);
          const int r0 = ia * 256 + static_cast<int>(rank) * 128;
          if (a.a_slice_mid)
            tma_load_3d_pair(sA + s * kATileBytes, &a.tmA, bar, kk * 64, sa, r0, polA);
          else
            tma_load_3d_pair(sA + s * kATileBytes, &a.tmA, bar, kk * 64, r0, sa, polA);
        }
      };
      // the weight halves of the first S loads go out before the dependency
      // wait (weights are never written by the step)
      uint32_t pre = 0;
      for (int64_t tile = pair; tile < n_tiles && pre < (uint32_t)S; tile += P) {
        int g, ia, ib;
        tile_coords(tile, g, ia, ib);
        int ks = 0, kk = 0;
        for (int k = 0; k < K && pre < (uint32_t)S; ++k, ++pre) {
          if (rank == 0) mbar_arrive_expect_tx(&full[pre], stage_tx);
          load(g, ia, ib, ks, kk, pre, true);
          if (++kk == kis) { kk = 0; ++ks; }
        }
      }
      pdl_wait();
      uint32_t n = 0, s = 0, ph = 0;  // load count, stage, stage phase
      bool ok = true;
      for (int64_t tile = pair; ok && tile < n_tiles; tile += P) {
        int g, ia, ib;
        tile_coords(tile, g, ia, ib);
        int ks = 0, kk = 0;
        for (int k = 0; k < K; ++k, ++n) {
          if (n >= pre) {
            if (!mbar_wait(&empty[s], ph ^ 1, a.status)) { ok = false; break; }
            if (rank == 0) mbar_arrive_expect_tx(&full[s], stage_tx);
            load(g, ia, ib, ks, kk, s, true);
          }
          load(g, ia, ib, ks, kk, s, false);
          if (++kk == kis) { kk = 0; ++ks; }
          if (++s == (uint32_t)S) { s = 0; ph ^= 1; }
        }
      }
      // never leave with bulk copies still landing: the even CTA's full
      // barriers count both CTAs' copies (the odd CTA stays until the final
      // cluster barrier, which the even CTA reaches only after this)
      if (rank == 0)
        for (uint32_t i = (n > (uint32_t)S ? n - S : 0); i < n; ++i)
          mbar_wait(&full[i % S], (i / S) & 1, a.status);
    } else {
      pdl_wait();
    }
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = idesc_bf16_f32(256, BN);
      uint32_t seg = 0, s = 0, ph = 0;  // tile count, stage, stage phase
      bool ok = true;
      for (int64_t tile = pair; ok && tile < n_tiles; tile += P) {
        const uint32_t buf = seg & 1, use = seg >> 1;
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, a.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int k = 0; k < K; ++k) {
          if (!mbar_wait(&full[s], ph, a.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t da = smem_desc_sw128(sA + s * kATileBytes);
          const uint64_t db = smem_desc_sw128(sB + s * b_half_bytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_f16_pair(d_tmem, da + 2 * kk, db + 2 * kk, idesc, (k > 0 || kk > 0) ? 1u : 0u);
          tc_commit_pair(&empty[s], 0x3);
          if (++s == (uint32_t)S) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc_commit_pair(&acc_full[buf], 0x3);
        ++seg;
      }
      tc_commit_pair(drain, 0x1);
      mbar_wait(drain, 0, a.status);
    }
  } else {
    pdl_wait();
    if constexpr (kLateSignal) pdl_launch_dependents();
    // epilogue warp w reads TMEM lanes of quadrant w % 4 (token rows of this
    // CTA) and the 16-column units half, half + NH, ... of the tile
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const uint32_t acc_empty0 = mapa_shared(smem_u32(acc_empty), 0);
    const int* tok = nullptr;  // token tables live in EpiArgs in this orientation
    // the folded norm's 1/rms of this thread's row in the last two 256-row
    // blocks seen: a pair's tiles p, p + P, ... revisit few row blocks (two
    // when P is a multiple of half the row-block count), so the row's sums are
    // read once per block rather than once per tile
    int rs_blk0 = -1, rs_blk1 = -1;
    float rs_val0 = 1.f, rs_val1 = 1.f;
    bool rs_next1 = false;
    uint32_t seg = 0;
    for (int64_t tile = pair; tile < n_tiles; tile += P) {
      int g, ia, ib;
      tile_coords(tile, g, ia, ib);
      const uint32_t buf = seg & 1, use = seg >> 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&acc_full[buf], use & 1, a.status);
      if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + buf * BN;
      const int arow = ia * 256 + static_cast<int>(rank) * 128 + row;
      const int brow = ib * BN;
      // inputs of the next unit are fetched before the current one is stored;
      // the token's 1/rms (folded norm) once per tile, its sum of squares over
      // this thread's units (EPI_RESID_SQ)
      float rs = 1.f, ss = 0.f;
      if constexpr (kEpiNorm<EPI>) {
        const int blk = g * a.a_tiles + ia;
        if (rs_blk0 == blk) {
          rs = rs_val0;
        } else if (rs_blk1 == blk) {
          rs = rs_val1;
        } else {
          rs = prefill_row_rs(a.e, arow);
          if (rs_next1) { rs_blk1 = blk; rs_val1 = rs; }
          else { rs_blk0 = blk; rs_val0 = rs; }
          rs_next1 = !rs_next1;
        }
      }
      EpiIn cur, nxt;
      const int c_first = half * 16;
      if (c_first < BN) epi_load<false, EPI>(a, g, arow, brow + c_first, tok, cur);
      cur.rs = rs;
      for (int c0 = c_first; c0 < BN; c0 += NH * 16) {
        if (c0 + NH * 16 < BN) {
          epi_load<false, EPI>(a, g, arow, brow + c0 + NH * 16, tok, nxt);
          nxt.rs = rs;
        }
        float v[16];
        tmem_ld16(taddr + c0, v);
        tmem_ld_wait();
        ss += epi_chunk<false, EPI>(a, g, arow, brow + c0, tok, v, cur);
        cur = nxt;
      }
      if constexpr (EPI == EPI_RESID_SQ) store_row_sq(a, arow, ib, half, ss, NH == 1);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + buf * 8);
      ++seg;
    }
  }

  // both CTAs' epilogues are done with the accumulators and the even CTA's
  // MMAs have drained before either CTA frees tensor memory or exits
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, a.tmem_cols);
  }
}

}  // namespace tpk
