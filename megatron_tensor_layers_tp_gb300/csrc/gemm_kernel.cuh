// Sharded GEMM on the 5th-generation tensor cores: D = A * B^T, both operands
// K-major bf16 fed by TMA (128-byte swizzle), fp32 accumulators in tensor
// memory, fused epilogues for the tensor-parallel layer.
//
// One launch covers all t emulated ranks.  Operands are 3-D tensor maps
// (K, rows, slice) where the slice coordinate is the rank shard.  Work is the
// flat sequence of (output tile, 64-wide K step) pairs, scheduled (on the
// host) one of three ways:
//  - stream-K: CTA c of G processes the contiguous range [c*T/G, (c+1)*T/G),
//    so every CTA streams the same number of bytes.  A tile cut between CTAs
//    leaves fp32 partials in the workspace; the last CTA to finish a piece of
//    the tile (atomic ticket, no waiting) adds the pieces in K order — which
//    is rank order for the fused row-parallel reduction — and runs the
//    epilogue;
//  - cluster split-K (decode orientation, few tiles): a cluster of s CTAs per
//    tile, each taking 1/s of its K range; the pieces meet in distributed
//    shared memory and are added in K order after a cluster barrier;
//  - data-parallel waves of whole tiles (prefill orientation), the remainder
//    as a last, partial wave of whole tiles.
// The result is deterministic for a given grid.  (Prefill GEMMs with at least
// one wave of 256-row tiles run on CTA pairs instead: gemm_pair.cuh, with the
// epilogues defined here.)
//
// Roles: warp 0 issues TMA loads, warp 1 issues tcgen05.mma from one thread
// into one of two TMEM accumulators, and the epilogue warps (eight in the
// decode orientation, 320 threads; four in the prefill orientation, 192)
// drain the other accumulator (tcgen05.ld) and run the epilogue.  The qkv and
// gate_up epilogues also apply the RMSNorm folded into those GEMMs: each
// token's 1/rms from h's rows (decode orientation, worked out by the epilogue
// warps while the weights stream) or from the sums of squares the kernel
// that wrote h left.  Every wait is bounded.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"
#include "rms.cuh"

namespace tpk {

constexpr int kATileBytes = 128 * 128;  // 128 rows x 64 bf16

__device__ __forceinline__ uint64_t make_policy(int kind) {
  if (kind == 1) return policy_evict_first();
  if (kind == 2) return policy_evict_last();
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ int slice_of(int mode, int g, int ks) {
  return mode == 1 ? g : (mode == 2 ? ks : 0);
}

// --------------------------------------------------------------------------
// epilogues: one call handles 16 accumulator columns of one TMEM lane.
// SWAP (decode): lane = feature row of the weight, columns = tokens.
// !SWAP (prefill): lane = token, columns = feature rows.
// --------------------------------------------------------------------------
__device__ __forceinline__ void qkv_classify(const EpiArgs& e, int f, int& kind, int& head,
                                             int& w) {
  const int d = e.head_dim;
  const int nq = e.q_heads_per_rank * d, nk = e.kv_heads_per_rank * d;
  if (f < nq) { kind = 0; head = f / d; w = f - head * d; }
  else if (f < nq + nk) { kind = 1; head = (f - nq) / d; w = f - nq - head * d; }
  else { kind = 2; head = (f - nq - nk) / d; w = f - nq - nk - head * d; }
}

// Standard per-rank column of shard row f (undoes the pair interleaving).
__device__ __forceinline__ int plain_col(const EpiArgs& e, int f) {
  if (e.which == 1) return (f & 1) ? e.inter_per_rank + (f >> 1) : (f >> 1);
  int kind, head, w;
  qkv_classify(e, f, kind, head, w);
  const int d = e.head_dim;
  const int base = f - w;
  if (kind == 2) return f;
  return base + ((w & 1) ? (w >> 1) + d / 2 : (w >> 1));
}

// Inputs of the epilogues (residual values; token positions, sequences and
// RoPE factors), fetched by epi_load ahead of the arithmetic so their latency
// overlaps the other loads of a fix-up.  In the decode orientation the
// tokens' positions come from the CTA's shared-memory copy (tok: positions of
// tokens 0..kSwapMaxTokens-1, their sequences, then each token's part of a
// K/V cache index as int64).
struct EpiIn {
  float r[16];
  int pos[16];
  float2 cs[16];
  float b[16];  // output bias: one value per row (decode) or per column (prefill)
  float rs;     // prefill orientation, folded RMSNorm: the token's 1/rms (set by the caller)
};

// Prefill orientation, folded RMSNorm (norm_mode 2): token m's 1/rms from the
// sums of squares the kernel that wrote h left (norm_slots per token, fixed
// order); 1 for any other norm mode.
// (norm_slots is a multiple of 4: a row's slots are read as 16-byte vectors,
// eight in flight together)
__device__ __forceinline__ float prefill_row_rs(const EpiArgs& e, int m) {
  if (e.norm_mode != 2 || m >= e.M) return 1.f;
  const float4* p = reinterpret_cast<const float4*>(e.norm_partials + (int64_t)m * e.norm_slots);
  const int n4 = e.norm_slots >> 2;
  float ss = 0.f;
  for (int i0 = 0; i0 < n4; i0 += 8) {
    float4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = i0 + k < n4 ? __ldcg(p + i0 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k) ss += (v[k].x + v[k].y) + (v[k].z + v[k].w);
  }
  return 1.0f / sqrtf(ss / (float)e.norm_width + e.norm_eps);
}

// Epilogues that add the GEMM's output bias (the unfused row-parallel
// partials leave it to the rank reduction; the LM head has none).
// Columns one epilogue thread finishes at a time: 8 tokens in the decode
// orientation (two warps share each TMEM lane quadrant, each taking alternate
// 8-column units), 16 features in the prefill orientation.
template <bool SWAP>
constexpr int kUnit = SWAP ? 8 : 16;
// epilogue warps: 8 in the decode orientation, 4 in the prefill orientation
template <bool SWAP>
constexpr int kEpiWarps = SWAP ? 8 : 4;
template <bool SWAP>
constexpr int kThreadsOf = (2 + kEpiWarps<SWAP>) * 32;

// the fused row-parallel epilogues: residual + rank sum (+ the next norm's sums of squares)
template <int EPI>
constexpr bool kResid = EPI == EPI_RESID || EPI == EPI_RESID_SQ;
template <int EPI>
constexpr bool kEpiBias = EPI == EPI_PLAIN || EPI == EPI_QKV || EPI == EPI_SILU || kResid<EPI>;
// Epilogues that can scale by a folded RMSNorm's 1/rms (decode orientation):
// the two column-parallel GEMMs that follow a norm in the decoder layer.
template <int EPI>
constexpr bool kEpiNorm = EPI == EPI_QKV || EPI == EPI_SILU;
// Multi-chunk epilogues fetch the next chunk's inputs before storing the
// current one, except qkv, whose inputs (positions, RoPE factors) would not
// fit in registers twice next to the fix-up's pieces.
template <int EPI>
constexpr bool kEpiAhead = EPI != EPI_QKV;

template <bool SWAP, int EPI>
__device__ __forceinline__ void epi_load(const GemmArgs& a, int g, int arow, int brow0,
                                         const int* tok, EpiIn& in) {
  const EpiArgs& e = a.e;
  const int f = arow;
  const bool fval = f < a.a_rows_valid;
  if constexpr (kEpiBias<EPI>) {
    if (e.bias) {
      const uint16_t* bg = e.bias + (int64_t)g * e.bias_group_stride;
      if constexpr (SWAP) {
        in.b[0] = fval ? bf16_to_f(bg[f]) : 0.f;
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          in.b[j] = brow0 + j < a.b_rows_valid ? bf16_to_f(bg[brow0 + j]) : 0.f;
      }
    }
  }
  if constexpr (SWAP && kResid<EPI>) {
#pragma unroll
    for (int j = 0; j < kUnit<SWAP>; ++j) {
      const int m = brow0 + j;
      in.r[j] = (e.residual && fval && m < e.M) ? bf16_to_f(e.residual[(int64_t)m * e.ld_res + f])
                                                : 0.f;
    }
  } else if constexpr (SWAP && EPI == EPI_QKV) {
    int kind = 2, head = 0, w = 0;
    if (fval) qkv_classify(e, f, kind, head, w);
    const int half = e.head_dim / 2, jp = w >> 1;
#pragma unroll
    for (int j = 0; j < kUnit<SWAP>; ++j) {
      const int m = brow0 + j;
      in.pos[j] = (fval && m < e.M) ? tok[m] : -1;
    }
#pragma unroll
    for (int j = 0; j < kUnit<SWAP>; ++j) {
      const bool ok = in.pos[j] >= 0 && in.pos[j] < e.l_max;
      in.cs[j] = (ok && kind != 2) ? e.rope[(int64_t)in.pos[j] * half + jp] : make_float2(1.f, 0.f);
    }
  } else if constexpr (!SWAP && kResid<EPI>) {
    // prefill orientation: lane = token m, 16 consecutive features f0..f0+15
    const int m = arow, f0 = brow0;
    if (e.residual && m < e.M && f0 < a.b_rows_valid) {
      const uint4* rp = reinterpret_cast<const uint4*>(e.residual + (int64_t)m * e.ld_res + f0);
      const uint4 r0 = rp[0], r1 = rp[1];
      const uint16_t* rb0 = reinterpret_cast<const uint16_t*>(&r0);
      const uint16_t* rb1 = reinterpret_cast<const uint16_t*>(&r1);
#pragma unroll
      for (int j = 0; j < 8; ++j) { in.r[j] = bf16_to_f(rb0[j]); in.r[8 + j] = bf16_to_f(rb1[j]); }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) in.r[j] = 0.f;
    }
  } else if constexpr (!SWAP && EPI == EPI_QKV) {
    // pos[0]: the token's position, pos[1]: its sequence (K/V rows only)
    const int m = arow, f0 = brow0;
    int kind, head, w;
    qkv_classify(e, f0, kind, head, w);
    const bool mval = m < e.M && f0 < a.b_rows_valid;
    in.pos[0] = mval ? e.positions[m] : -1;
    in.pos[1] = (mval && kind != 0) ? e.token_seq[m] : 0;
    const bool ok = in.pos[0] >= 0 && in.pos[0] < e.l_max && kind != 2;
    const float2* cs = e.rope + (int64_t)(ok ? in.pos[0] : 0) * (e.head_dim / 2) + (w >> 1);
#pragma unroll
    for (int j = 0; j < 8; ++j) in.cs[j] = ok ? cs[j] : make_float2(1.f, 0.f);
  }
}

// Returns, in the prefill orientation with EPI_RESID_SQ, the sum of the
// squares of the 16 values it stored (0 otherwise).
template <bool SWAP, int EPI>
__device__ __forceinline__ float epi_chunk(const GemmArgs& a, int g, int arow, int brow0,
                                           const int* tok, float (&v)[16], const EpiIn& in) {
  const EpiArgs& e = a.e;
  if constexpr (SWAP && kEpiNorm<EPI>) {
    if (e.norm_mode) {  // the token's 1/rms, staged in shared memory after tok
      const float* rs = reinterpret_cast<const float*>(tok + 4 * kSwapMaxTokens);
#pragma unroll
      for (int j = 0; j < kUnit<SWAP>; ++j) v[j] *= rs[brow0 + j];
    }
  } else if constexpr (!SWAP && kEpiNorm<EPI>) {
    if (e.norm_mode == 2) {  // the token's 1/rms, fetched by the caller once per tile
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] *= in.rs;
    }
  }
  if constexpr (kEpiBias<EPI>) {
    if (e.bias) {  // before RoPE / SiLU pairing and the residual
#pragma unroll
      for (int j = 0; j < kUnit<SWAP>; ++j) v[j] += SWAP ? in.b[0] : in.b[j];
    }
  }
  if constexpr (SWAP) {
    const int f = arow;
    const bool fval = f < a.a_rows_valid;
    if constexpr (EPI == EPI_RESID) {
      // The residual is usually the output buffer itself (in-place update of
      // the hidden state): read all 16 values before the first store so the
      // loads are not serialised behind stores to the same buffer.
      uint16_t* out = static_cast<uint16_t*>(e.out);
#pragma unroll
      for (int j = 0; j < kUnit<SWAP>; ++j) {
        const int m = brow0 + j;
        if (fval && m < e.M) out[(int64_t)m * e.ld_out + f] = f_to_bf16(v[j] + in.r[j]);
      }
    } else if constexpr (EPI == EPI_RESID_SQ) {
      uint16_t* out = static_cast<uint16_t*>(e.out);
      float sq[kUnit<SWAP>];
#pragma unroll
      for (int j = 0; j < kUnit<SWAP>; ++j) {
        const int m = brow0 + j;
        const uint16_t ob = f_to_bf16(v[j] + in.r[j]);
        const bool st = fval && m < e.M;
        if (st) out[(int64_t)m * e.ld_out + f] = ob;
        const float of = bf16_to_f(ob);
        sq[j] = st ? of * of : 0.f;
      }
      // the next RMSNorm's sums of squares over this warp's 32 features, per
      // token: halve the token set at each exchange (xor 16, 8, 4), then
      // finish the sum over lane bits 1 and 0; lane 4j ends with token j
      static_assert(kUnit<SWAP> == 8, "8 tokens per unit");
      const int lane = threadIdx.x & 31;
      float s4[4], s2[2];
      const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        s4[i] = (b4 ? sq[4 + i] : sq[i]) + __shfl_xor_sync(0xffffffffu, b4 ? sq[i] : sq[4 + i], 16);
#pragma unroll
      for (int i = 0; i < 2; ++i)
        s2[i] = (b3 ? s4[2 + i] : s4[i]) + __shfl_xor_sync(0xffffffffu, b3 ? s4[i] : s4[2 + i], 8);
      float s1 = (b2 ? s2[1] : s2[0]) + __shfl_xor_sync(0xffffffffu, b2 ? s2[0] : s2[1], 4);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
      s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
      if ((lane & 3) == 0) e.sq_out[(int64_t)(brow0 + (lane >> 2)) * e.sq_ld + (f >> 5)] = s1;
    } else if constexpr (EPI == EPI_PARTIAL) {
      float* out = static_cast<float*>(e.out) + (int64_t)g * e.out_group_stride;
#pragma unroll
      for (int j = 0; j < kUnit<SWAP>; ++j) {
        const int m = brow0 + j;
        if (fval && m < e.M) out[(int64_t)m * e.ld_out + f] = v[j];
      }
    } else if constexpr (EPI == EPI_PLAIN) {
      uint16_t* out = static_cast<uint16_t*>(e.out) + (int64_t)g * e.out_group_stride;
      const int col = fval ? plain_col(e, f) : 0;
#pragma unroll
      for (int j = 0; j < kUnit<SWAP>; ++j) {
        const int m = brow0 + j;
        if (fval && m < e.M) out[(int64_t)m * e.ld_out + col] = f_to_bf16(v[j]);
      }
    } else if constexpr (EPI == EPI_LOGITS) {
      uint16_t* out = static_cast<uint16_t*>(e.out);
      const int64_t col = (int64_t)g * e.vocab_per_rank + f;
      const bool ok = fval && f < e.vocab_per_rank && col < e.vocab;
#pragma unroll
      for (int j = 0; j < kUnit<SWAP>; ++j) {
        const int m = brow0 + j;
        if (ok && m < e.M) out[(int64_t)m * e.ld_out + col] = f_to_bf16(v[j]);
      }
    } else if constexpr (EPI == EPI_SILU) {
      uint16_t* out = static_cast<uint16_t*>(e.out);
      const int64_t col = (int64_t)g * e.inter_per_rank + (f >> 1);
#pragma unroll
      for (int j = 0; j < kUnit<SWAP>; ++j) {
        const float partner = __shfl_xor_sync(0xffffffffu, v[j], 1);
        const int m = brow0 + j;
        if (fval && !(f & 1) && m < e.M) {
          const float gt = v[j], up = partner;
          out[(int64_t)m * e.ld_out + col] = f_to_bf16(__fdividef(gt, 1.f + __expf(-gt)) * up);
        }
      }
    } else if constexpr (EPI == EPI_QKV) {
      int kind = 2, head = 0, w = 0;
      if (fval) qkv_classify(e, f, kind, head, w);
      const int d = e.head_dim, half = d / 2;
      const int jp = w >> 1;
      const bool second = (w & 1) != 0;
      const int feat = kind == 2 ? w : (second ? jp + half : jp);
      const bool primary = (g % e.kv_replicas) == 0;
      const int copy = g / e.kv_replicas;
      uint16_t* qout = static_cast<uint16_t*>(e.out);
      // this thread's (copy, KV head, feature) part of a cache index; the
      // token's part ((seq * kv_r) * l_max + pos) * d is staged in shared memory
      uint16_t* cache_row = (kind == 1 ? e.k_cache : e.v_cache) + copy * e.kv_copy_stride +
                            (int64_t)head * e.l_max * d + feat;
#pragma unroll
      for (int j = 0; j < kUnit<SWAP>; ++j) {
        const float partner = __shfl_xor_sync(0xffffffffu, v[j], 1);
        const int m = brow0 + j;
        if (!fval || m >= e.M) continue;
        const int pos = in.pos[j];
        if (pos < 0 || pos >= e.l_max) continue;  // never index the cache or table out of range
        float val = v[j];
        if (kind != 2) {
          const float2 cs = in.cs[j];
          val = second ? (v[j] * cs.x + partner * cs.y) : (v[j] * cs.x - partner * cs.y);
        }
        if (kind == 0) {
          qout[(int64_t)m * e.ld_out + (int64_t)(g * e.q_heads_per_rank + head) * d + feat] =
              f_to_bf16(val);
        } else if (primary) {
          cache_row[reinterpret_cast<const int64_t*>(tok + 2 * kSwapMaxTokens)[m]] =
              f_to_bf16(val);
        }
      }
    }
  } else {
    const int m = arow;
    const int f0 = brow0;
    if (m >= e.M || f0 >= a.b_rows_valid) return 0.f;
    if constexpr (kResid<EPI>) {
      uint16_t* out = static_cast<uint16_t*>(e.out) + (int64_t)m * e.ld_out + f0;
      const float* r = in.r;
      uint4 o0, o1;
      uint32_t* p0 = reinterpret_cast<uint32_t*>(&o0);
      uint32_t* p1 = reinterpret_cast<uint32_t*>(&o1);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        p0[j] = pack_bf16x2(v[2 * j] + r[2 * j], v[2 * j + 1] + r[2 * j + 1]);
        p1[j] = pack_bf16x2(v[8 + 2 * j] + r[8 + 2 * j], v[9 + 2 * j] + r[9 + 2 * j]);
      }
      reinterpret_cast<uint4*>(out)[0] = o0;
      reinterpret_cast<uint4*>(out)[1] = o1;
      if constexpr (EPI == EPI_RESID_SQ) {
        // the squares of the stored values, for the next RMSNorm
        float sq = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t w[2] = {p0[j], p1[j]};
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const float lo = __uint_as_float(w[q] << 16), hi = __uint_as_float(w[q] & 0xFFFF0000u);
            sq = fmaf(lo, lo, fmaf(hi, hi, sq));
          }
        }
        return sq;
      }
    } else if constexpr (EPI == EPI_PARTIAL) {
      float4* out = reinterpret_cast<float4*>(static_cast<float*>(e.out) +
                                              (int64_t)g * e.out_group_stride +
                                              (int64_t)m * e.ld_out + f0);
#pragma unroll
      for (int j = 0; j < 4; ++j) out[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else if constexpr (EPI == EPI_PLAIN) {
      uint16_t* row = static_cast<uint16_t*>(e.out) + (int64_t)g * e.out_group_stride +
                      (int64_t)m * e.ld_out;
      int kind = 2, head = 0, w = 0;
      if (e.which == 0) qkv_classify(e, f0, kind, head, w);
      if (e.which == 0 && kind == 2) {
        uint4 o0, o1;
        uint32_t* p0 = reinterpret_cast<uint32_t*>(&o0);
        uint32_t* p1 = reinterpret_cast<uint32_t*>(&o1);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          p0[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
          p1[j] = pack_bf16x2(v[8 + 2 * j], v[9 + 2 * j]);
        }
        reinterpret_cast<uint4*>(row + f0)[0] = o0;
        reinterpret_cast<uint4*>(row + f0)[1] = o1;
      } else {
        // 8 pairs: first halves go to one run of 8 columns, second halves to another
        uint4 lo, hi;
        uint32_t* pl = reinterpret_cast<uint32_t*>(&lo);
        uint32_t* ph = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          pl[j] = pack_bf16x2(v[4 * j], v[4 * j + 2]);
          ph[j] = pack_bf16x2(v[4 * j + 1], v[4 * j + 3]);
        }
        int c_lo, c_hi;
        if (e.which == 1) { c_lo = f0 >> 1; c_hi = e.inter_per_rank + (f0 >> 1); }
        else { c_lo = f0 - w + (w >> 1); c_hi = c_lo + e.head_dim / 2; }
        *reinterpret_cast<uint4*>(row + c_lo) = lo;
        *reinterpret_cast<uint4*>(row + c_hi) = hi;
      }
    } else if constexpr (EPI == EPI_LOGITS) {
      uint16_t* row = static_cast<uint16_t*>(e.out) + (int64_t)m * e.ld_out;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int f = f0 + j;
        const int64_t col = (int64_t)g * e.vocab_per_rank + f;
        if (f < e.vocab_per_rank && col < e.vocab) row[col] = f_to_bf16(v[j]);
      }
    } else if constexpr (EPI == EPI_SILU) {
      uint16_t* row = static_cast<uint16_t*>(e.out) + (int64_t)m * e.ld_out +
                      (int64_t)g * e.inter_per_rank + (f0 >> 1);
      uint4 o;
      uint32_t* p = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float g0 = v[4 * j], u0 = v[4 * j + 1], g1 = v[4 * j + 2], u1 = v[4 * j + 3];
        p[j] = pack_bf16x2(g0 / (1.f + expf(-g0)) * u0, g1 / (1.f + expf(-g1)) * u1);
      }
      *reinterpret_cast<uint4*>(row) = o;
    } else if constexpr (EPI == EPI_QKV) {
      int kind, head, w;
      qkv_classify(e, f0, kind, head, w);
      const int d = e.head_dim, half = d / 2;
      const int pos = in.pos[0];
      if (pos < 0 || pos >= e.l_max) return 0.f;  // never index the cache or table out of range
      float outv[16];
      if (kind == 2) {
#pragma unroll
        for (int j = 0; j < 16; ++j) outv[j] = v[j];
      } else {
  #pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float2 c = in.cs[j];
          const float x1 = v[2 * j], x2 = v[2 * j + 1];
          outv[j] = x1 * c.x - x2 * c.y;       // feature jp
          outv[8 + j] = x2 * c.x + x1 * c.y;   // feature jp + d/2
        }
      }
      uint4 lo, hi;
      uint32_t* pl = reinterpret_cast<uint32_t*>(&lo);
      uint32_t* ph = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pl[j] = pack_bf16x2(outv[2 * j], outv[2 * j + 1]);
        ph[j] = pack_bf16x2(outv[8 + 2 * j], outv[9 + 2 * j]);
      }
      // destination runs: V rows are in natural order; Q/K pairs split in two runs
      const int c_lo = kind == 2 ? w : (w >> 1);
      const int c_hi = kind == 2 ? w + 8 : (w >> 1) + half;
      if (kind == 0) {
        uint16_t* dst = static_cast<uint16_t*>(e.out) + (int64_t)m * e.ld_out +
                        (int64_t)(g * e.q_heads_per_rank + head) * d;
        *reinterpret_cast<uint4*>(dst + c_lo) = lo;
        *reinterpret_cast<uint4*>(dst + c_hi) = hi;
      } else if ((g % e.kv_replicas) == 0) {
        const int seq = in.pos[1];
        uint16_t* cache = kind == 1 ? e.k_cache : e.v_cache;
        uint16_t* dst = cache + (int64_t)(g / e.kv_replicas) * e.kv_copy_stride +
                        (((int64_t)seq * e.kv_heads_per_rank + head) * e.l_max + pos) * d;
        *reinterpret_cast<uint4*>(dst + c_lo) = lo;
        *reinterpret_cast<uint4*>(dst + c_hi) = hi;
      }
    }
  }
  return 0.f;
}

// Prefill orientation, EPI_RESID_SQ: token m's sum of squares over its units
// of output tile ib of b_tiles (half: which of two threads sharing the tile;
// whole: one thread covered the whole tile, so the other slot is zero).  The
// last tile's writers also zero the padding up to sq_ld (a multiple of 4).
__device__ __forceinline__ void store_row_sq(const GemmArgs& a, int m, int ib, int half, float ss,
                                             bool whole) {
  const EpiArgs& e = a.e;
  if (!e.sq_out || m >= e.M) return;
  float* row = e.sq_out + (int64_t)m * e.sq_ld;
  row[2 * ib + half] = ss;
  if (whole) row[2 * ib + 1] = 0.f;
  if (ib == a.b_tiles - 1 && half == 0)
    for (int i = 2 * a.b_tiles; i < e.sq_ld; ++i) row[i] = 0.f;
}

// --------------------------------------------------------------------------
// Work of CTA c: first W data-parallel waves — tile c + w*G over its whole K
// range, so all CTAs walk K in lockstep and the operand slices in flight are
// shared through L2 — then an even share of the flat (tile, K step) range of
// the remaining tiles (stream-K).  A tile split there is finished by the last
// CTA to deliver a piece.  Index arithmetic happens once per segment.
struct Segment {
  int64_t tile;   // global tile index
  int k0, k1;     // K steps [k0, k1) of the tile
  bool sk;        // from the stream-K part (may still be the whole tile)
};

struct SegIter {
  int G, c, K, W;
  int64_t dp_tiles, T, beg, end;
  int w;
  int64_t it;
  int split;   // cluster split-K: one segment, 1/split of tile c / split's K range
  bool used;
  const FastDiv* dk;  // division by K as a multiply-shift (null: 64-bit division)
  __device__ __forceinline__ bool next(Segment& s) {
    if (split > 1) {
      if (used) return false;
      used = true;
      const int r = c % split;
      s.tile = c / split;
      s.k0 = r * K / split;
      s.k1 = (r + 1) * K / split;
      s.sk = false;
      return true;
    }
    if (w < W) {
      s.tile = c + (int64_t)w * G;
      s.k0 = 0;
      s.k1 = K;
      s.sk = false;
      ++w;
      return true;
    }
    if (it >= end) return false;
    const int64_t ts = dk ? static_cast<int64_t>(fast_div(static_cast<uint32_t>(it), *dk)) : it / K;
    const int64_t seg_end = min(end, (ts + 1) * K);
    s.tile = dp_tiles + ts;
    s.k0 = static_cast<int>(it - ts * K);
    s.k1 = static_cast<int>(seg_end - ts * K);
    s.sk = true;
    it = seg_end;
    return true;
  }
};

template <bool SWAP, int EPI>
__global__ void __launch_bounds__(kThreadsOf<SWAP>, 1) gemm_kernel(const __grid_constant__ GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int BN = a.BN, S = a.stages;
  const int b_tile_bytes = BN * 128;
  uint8_t* sA = smem;
  uint8_t* sB = smem + S * kATileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + S * b_tile_bytes);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* last_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* tok = reinterpret_cast<int*>(last_flag + 3);  // decode: positions, sequences, cache offsets
  // then (decode, folded RMSNorm) kSwapMaxTokens floats: each token's 1/rms

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps<SWAP>);
    }
    mbar_init(drain, 1);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) { tma_prefetch_desc(&a.tmA); tma_prefetch_desc(&a.tmB); }
  if (warp == 1) { tmem_alloc(tmem_slot, a.tmem_cols); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int G = a.grid, c = blockIdx.x;
  const int64_t T = a.total_iters;  // stream-K iterations
  const int K = a.k_slices * a.k_iters_slice;  // K steps per tile
  const int64_t dp_tiles = (int64_t)a.dp_waves * G;
  const int Gs = a.sk_ctas > 0 ? a.sk_ctas : G;  // CTAs sharing the stream-K part
  const int64_t beg = c < Gs ? range_begin(c, T, Gs) : T;
  const int64_t end = c < Gs ? range_begin(c + 1, T, Gs) : T;
  // Index divisions: after the dependency wait (fast = true) they are
  // multiply-shifts when the host set fix32; the weight loads issued before
  // the wait keep 64-bit divisions (measured: speeding those up made the
  // decode step slower, its first loads then competing with the tail of the
  // kernel before)
  auto make_iter = [&](bool fast) {
    SegIter si;
    si.G = G; si.c = c; si.K = K; si.W = a.dp_waves;
    si.dp_tiles = dp_tiles; si.T = T; si.beg = beg; si.end = end;
    si.w = 0; si.it = beg;
    si.split = a.cluster_split; si.used = false;
    si.dk = fast && a.fix32 ? &a.div_k : nullptr;
    return si;
  };
  auto tile_coords = [&](int64_t tile, int& g, int& ia, int& ib, bool fast) {
    if (fast && a.fix32) {
      const uint32_t rest = fast_div(static_cast<uint32_t>(tile), a.div_a);
      ia = static_cast<int>(static_cast<uint32_t>(tile) - rest * a.a_tiles);
      const uint32_t gq = fast_div(rest, a.div_b);
      ib = static_cast<int>(rest - gq * a.b_tiles);
      g = static_cast<int>(gq);
      return;
    }
    ia = static_cast<int>(tile % a.a_tiles);
    const int64_t rest = tile / a.a_tiles;
    ib = static_cast<int>(rest % a.b_tiles);
    g = static_cast<int>(rest / a.b_tiles);
  };

  // Epilogue inputs of this CTA's last segment: that segment's epilogue (or
  // fix-up) ends the kernel, so in the decode orientation (few 8-column units
  // per thread) the inputs of its first unit are fetched as soon as the
  // epilogue warps may read them, long before the accumulator is ready.
  EpiIn pre;
  bool pre_ok = false;
  int n_segs = 0;

  // Launched with programmatic stream serialisation: the next kernel may start
  // its own set-up now.  Everything below that reads data written by an
  // earlier kernel comes after pdl_wait(); only the weight shards (written
  // once when the model was loaded) are fetched before it.  The qkv
  // projection is the exception that signals late (after its wait): decode
  // attention reads the cache rows of earlier steps before its own wait, which
  // is sound only if every kernel before this one has completed.
  constexpr bool kLateSignal = EPI == EPI_QKV || EPI == EPI_QKV_PIECES;
  if constexpr (!kLateSignal) pdl_launch_dependents();
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t polA = make_policy(a.a_policy), polB = make_policy(a.b_policy);
      // decode orientation: A holds the weights; prefill orientation: B does.
      // (ks, kk): rank slice and 64-wide step inside it, kept as counters.
      // The weights' tensor map is 4-D over the K-blocked shards (coordinates:
      // 0, row, K block, rank); the activations' is 3-D (K, rows, slice).
      auto issue = [&](int g, int ia, int ib, int ks, int kk, uint32_t s, bool weights) {
        if (weights == SWAP) {
          const int sa = slice_of(a.a_slice_mode, g, ks);
          if constexpr (SWAP)
            tma_load_4d(sA + s * kATileBytes, &a.tmA, &full[s], 0, ia * 128, kk, sa, polA);
          else if (a.a_slice_mid)
            tma_load_3d(sA + s * kATileBytes, &a.tmA, &full[s], kk * 64, sa, ia * 128, polA);
          else
            tma_load_3d(sA + s * kATileBytes, &a.tmA, &full[s], kk * 64, ia * 128, sa, polA);
        } else {
          const int sb = slice_of(a.b_slice_mode, g, ks);
          if constexpr (!SWAP)
            tma_load_4d(sB + s * b_tile_bytes, &a.tmB, &full[s], 0, ib * BN, kk, sb, polB);
          else if (a.b_slice_mid)
            tma_load_3d(sB + s * b_tile_bytes, &a.tmB, &full[s], kk * 64, sb, ib * BN, polB);
          else
            tma_load_3d(sB + s * b_tile_bytes, &a.tmB, &full[s], kk * 64, ib * BN, sb, polB);
        }
      };
      // first use of each stage needs no wait: put the weight tiles of the
      // first S loads in flight before waiting for the previous kernel
      const int kis = a.k_iters_slice;
      uint32_t pre = 0;
      {
        SegIter si = make_iter(false);
        Segment sg;
        while (pre < (uint32_t)S && si.next(sg)) {
          int g, ia, ib;
          tile_coords(sg.tile, g, ia, ib, false);
          int ks = sg.k0 / kis, kk = sg.k0 - ks * kis;
          for (int k = sg.k0; k < sg.k1 && pre < (uint32_t)S; ++k, ++pre) {
            mbar_arrive_expect_tx(&full[pre], kATileBytes + b_tile_bytes);
            issue(g, ia, ib, ks, kk, pre, true);
            if (++kk == kis) { kk = 0; ++ks; }
          }
        }
      }
      pdl_wait();
      uint32_t n = 0, s = 0, ph = 0;  // load count, stage, stage phase
      bool ok = true;
      SegIter si = make_iter(true);
      Segment sg;
      while (ok && si.next(sg)) {
        int g, ia, ib;
        tile_coords(sg.tile, g, ia, ib, true);
        int ks = sg.k0 / kis, kk = sg.k0 - ks * kis;
        for (int k = sg.k0; k < sg.k1; ++k, ++n) {
          if (n >= pre) {
            if (!mbar_wait(&empty[s], ph ^ 1, a.status)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[s], kATileBytes + b_tile_bytes);
            issue(g, ia, ib, ks, kk, s, true);
          }
          issue(g, ia, ib, ks, kk, s, false);
          if (++kk == kis) { kk = 0; ++ks; }
          if (++s == (uint32_t)S) { s = 0; ph ^= 1; }
        }
      }
      // never leave with bulk copies still landing in shared memory
      for (uint32_t i = (n > (uint32_t)S ? n - S : 0); i < n; ++i)
        mbar_wait(&full[i % S], (i / S) & 1, a.status);
    } else {
      pdl_wait();
    }
  } else if (warp == 1) {
    pdl_wait();
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, BN);
      uint32_t seg = 0, s = 0, ph = 0;  // segment count, stage, stage phase
      bool ok = true;
      SegIter si = make_iter(true);
      Segment sg;
      while (ok && si.next(sg)) {
        const uint32_t buf = seg & 1, use = seg >> 1;
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, a.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int k = sg.k0; k < sg.k1; ++k) {
          if (!mbar_wait(&full[s], ph, a.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t da = smem_desc_sw128(sA + s * kATileBytes);
          const uint64_t db = smem_desc_sw128(sB + s * b_tile_bytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_f16(d_tmem, da + 2 * kk, db + 2 * kk, idesc, (k > sg.k0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[s]);
          if (++s == (uint32_t)S) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
        ++seg;
      }
      tc_commit(drain);
      mbar_wait(drain, 0, a.status);
    }
  } else {
    pdl_wait();
    if constexpr (kLateSignal) pdl_launch_dependents();
    // Epilogue warp w reads TMEM lanes of quadrant w % 4 (its 32 rows); in the
    // decode orientation two warps share a quadrant and take alternate
    // U-column units of every 16-column span.
    constexpr int U = kUnit<SWAP>, NH = kEpiWarps<SWAP> / 4, ET = kEpiWarps<SWAP> * 32;
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    const int et = threadIdx.x - 64;  // 0..ET-1 over the epilogue warps
    auto tld = [&](uint32_t addr, float (&v)[16]) {
      if constexpr (SWAP) tmem_ld8(addr, v);
      else tmem_ld16(addr, v);
    };
    bool staged = false;
    if constexpr (SWAP && EPI == EPI_QKV) {
      // every tile of the decode orientation covers tokens 0..M-1
      if (et < kSwapMaxTokens) {
        const bool ok = et < a.e.M;
        const int pos = ok ? a.e.positions[et] : -1;
        const int seq = ok ? a.e.token_seq[et] : 0;
        tok[et] = pos;
        tok[kSwapMaxTokens + et] = seq;
        reinterpret_cast<int64_t*>(tok + 2 * kSwapMaxTokens)[et] =
            ((int64_t)seq * a.e.kv_heads_per_rank * a.e.l_max + pos) * a.e.head_dim;
      }
      staged = true;
    }
    if constexpr (SWAP && kEpiNorm<EPI>) {
      if (a.e.norm_mode == 2) {
        // the folded RMSNorm's 1/rms of every token from the sums of squares
        // the kernel that wrote h left behind (fixed order: deterministic)
        // (the warp's tokens m = ew + 8 q: one 16-byte load per lane and token,
        // all tokens' loads in flight together)
        float* rs = reinterpret_cast<float*>(tok + 4 * kSwapMaxTokens);
        const int ew = et >> 5, n4 = a.e.norm_slots >> 2;
        constexpr int QW = kSwapMaxTokens / kEpiWarps<SWAP>;
        float ss[QW];
#pragma unroll
        for (int q = 0; q < QW; ++q) ss[q] = 0.f;
        for (int i4 = lane; i4 < n4; i4 += 32) {
          float4 p[QW];
#pragma unroll
          for (int q = 0; q < QW; ++q) {
            const int m = ew + q * kEpiWarps<SWAP>;
            p[q] = m < a.e.M ? __ldcg(reinterpret_cast<const float4*>(
                                   a.e.norm_partials + (int64_t)m * a.e.norm_slots) + i4)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int q = 0; q < QW; ++q) ss[q] += (p[q].x + p[q].y) + (p[q].z + p[q].w);
        }
#pragma unroll
        for (int q = 0; q < QW; ++q) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss[q] += __shfl_xor_sync(0xffffffffu, ss[q], o);
          const int m = ew + q * kEpiWarps<SWAP>;
          if (lane == 0 && m < a.e.M)
            rs[m] = 1.0f / sqrtf(ss[q] / (float)a.e.norm_width + a.e.norm_eps);
        }
        if (et >= a.e.M && et < kSwapMaxTokens) rs[et] = 0.f;
        staged = true;
      } else if (a.e.norm_mode == 1) {
        // the folded RMSNorm's 1/rms of every token, one warp per token, while
        // the MMA warp streams the weights (the hidden rows come from L2)
        float* rs = reinterpret_cast<float*>(tok + 4 * kSwapMaxTokens);
        const int ew = et >> 5;
        for (int m = ew; m < a.e.M; m += kEpiWarps<SWAP>) {
          const float ss = warp_row_sumsq(a.e.norm_src + (int64_t)m * a.e.norm_ld, a.e.norm_width);
          if (lane == 0) rs[m] = 1.0f / sqrtf(ss / (float)a.e.norm_width + a.e.norm_eps);
        }
        if (et >= a.e.M && et < kSwapMaxTokens) rs[et] = 0.f;
        staged = true;
      }
    }
    if (staged) bar_sync(1, ET);
    // units this thread stores itself: columns c0 = u0, u0 + ustep, ... of a
    // tile; in a cluster split the (half, rank) workers of the cluster share
    // the units of the one tile
    const int rank = a.cluster_split > 1 ? static_cast<int>(c % a.cluster_split) : 0;
    const int worker = half * (a.cluster_split > 1 ? a.cluster_split : 1) + rank;
    const int u0 = worker * U;
    const int ustep = NH * (a.cluster_split > 1 ? a.cluster_split : 1) * U;
    const int chunk0 = a.cluster_split > 1 ? u0 : half * U;
    {
      SegIter t = make_iter(true);
      Segment last, x;
      while (t.next(x)) { last = x; ++n_segs; }
      if (SWAP && n_segs > 0 && chunk0 < BN) {
        int g, ia, ib;
        tile_coords(last.tile, g, ia, ib, true);
        epi_load<SWAP, EPI>(a, g, ia * 128 + row, ib * BN + chunk0, tok, pre);
        pre_ok = true;
      }
    }
    uint32_t seg = 0;
    SegIter si = make_iter(true);
    Segment sg;
    while (si.next(sg)) {
      const bool use_pre = pre_ok && (int)seg == n_segs - 1;
      int g, ia, ib;
      tile_coords(sg.tile, g, ia, ib, true);
      const uint32_t buf = seg & 1, use = seg >> 1;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&acc_full[buf], use & 1, a.status);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (bar_sync_or(1, ET, !ok)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + buf * BN;
      const int arow = ia * 128 + row;
      const int brow = ib * BN;
      if (a.cluster_split > 1) {
        // cluster split-K: park this CTA's piece in its own shared memory (the
        // operand stages are free: every load was consumed by the finished
        // MMAs); the pieces are summed after the cluster barrier
        float* red = reinterpret_cast<float*>(smem);
        for (int c0 = half * U; c0 < BN; c0 += NH * U) {
          float v[16];
          tld(taddr + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < kUnit<SWAP>; ++j) red[(c0 + j) * 128 + row] = v[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        ++seg;
        continue;
      }
      if constexpr (EPI == EPI_QKV_PIECES) {
        // slot 0: the segment where this CTA's range starts, slot 1: the next
        // (a range never spans more than two tiles: the host keeps the grid at
        // least as large as the tile count)
        const int64_t ts = sg.tile - dp_tiles;
        const int my_slot = (beg / K == ts) ? 0 : 1;
        float* mine = a.partials + ((int64_t)(c * 2 + my_slot) * BN) * 128;
        for (int c0 = half * U; c0 < BN; c0 += NH * U) {
          float v[16];
          tld(taddr + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < kUnit<SWAP>; ++j) mine[(c0 + j) * 128 + row] = v[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        ++seg;
        continue;
      }
      // pieces of this tile in the stream-K part (1 for a data-parallel tile);
      // with fix32 the divisions are multiply-shifts (they sit on the tail)
      auto owner_fx = [&](int64_t x) -> int {
        if (a.fix32)
          return static_cast<int>(fast_div(static_cast<uint32_t>((x + 1) * Gs - 1), a.div_total));
        return owner_of(x, T, Gs);
      };
      auto start_fx = [&](int cc) -> int64_t {
        if (a.fix32) return fast_div(static_cast<uint32_t>(cc * T), a.div_sk);
        return range_begin(cc, T, Gs);
      };
      auto step_tile = [&](int64_t x) -> int64_t {
        if (a.fix32) return fast_div(static_cast<uint32_t>(x), a.div_k);
        return x / K;
      };
      int nseg = 1, c_first = c;
      int64_t ts = 0;
      if (sg.sk) {
        ts = sg.tile - dp_tiles;
        c_first = owner_fx(ts * K);
        nseg = owner_fx((ts + 1) * K - 1) - c_first + 1;
      }
      if (nseg == 1) {
        if constexpr (SWAP) {
          for (int c0 = half * U; c0 < BN; c0 += NH * U) {
            float v[16];
            EpiIn in;
            if (use_pre && c0 == half * U) in = pre;
            else epi_load<SWAP, EPI>(a, g, arow, brow + c0, tok, in);
            tld(taddr + c0, v);
            tmem_ld_wait();
            epi_chunk<SWAP, EPI>(a, g, arow, brow + c0, tok, v, in);
          }
        } else {
          // inputs of chunk c0 + 16 are fetched before chunk c0 is stored
          float rs = 1.f, ss = 0.f;
          if constexpr (kEpiNorm<EPI>) rs = prefill_row_rs(a.e, arow);
          EpiIn cur, nxt;
          epi_load<SWAP, EPI>(a, g, arow, brow, tok, cur);
          cur.rs = rs;
          for (int c0 = 0; c0 < BN; c0 += 16) {
            if (c0 + 16 < BN) {
              epi_load<SWAP, EPI>(a, g, arow, brow + c0 + 16, tok, nxt);
              nxt.rs = rs;
            }
            float v[16];
            tld(taddr + c0, v);
            tmem_ld_wait();
            ss += epi_chunk<SWAP, EPI>(a, g, arow, brow + c0, tok, v, cur);
            cur = nxt;
          }
          if constexpr (EPI == EPI_RESID_SQ) store_row_sq(a, arow, ib, 0, ss, true);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      } else {
        // my piece of the tile -> workspace slot 0 (tile where my range starts) or 1
        const int my_slot = (step_tile(beg) == ts) ? 0 : 1;
        float* mine = a.partials + ((int64_t)(c * 2 + my_slot) * BN) * 128;
        for (int c0 = half * U; c0 < BN; c0 += NH * U) {
          float v[16];
          tld(taddr + c0, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < kUnit<SWAP>; ++j) mine[(c0 + j) * 128 + row] = v[j];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        // Publish the piece and take the tile's ticket: the named barrier
        // orders every epilogue thread's stores before one thread's GPU-scope
        // fence and ticket increment; a second fence after the increment, and
        // the barrier after it, order the last arriver's reads of the other
        // pieces after the others' increments (one fence pair per piece
        // instead of a fence per thread)
        bar_sync(1, ET);
        if (threadIdx.x == 64) {
          fence_acq_rel_gpu();
          const int old = atomicAdd(&a.tickets[sg.tile], 1);
          fence_acq_rel_gpu();
          *last_flag = (old == nseg - 1) ? 1 : 0;
        }
        bar_sync(1, ET);
        if (*last_flag) {
          // The pieces in K order are those of CTAs c_first, c_first + 1, ...;
          // only the first can have started its range before this tile (its
          // piece then sits in slot 1).  Loads of up to 4 pieces are in flight
          // together, and the first batch of the next chunk is fetched before
          // the current chunk is stored.
          const int slot0 = start_fx(c_first) == ts * K ? 0 : 1;
          const float* base = a.partials + (int64_t)c_first * 2 * BN * 128 + row;
          float tmp[4][16];
          auto load_batch = [&](int c0, int s0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (s0 + q < nseg) {
                const int pq = s0 + q;
                const float* src = base + ((int64_t)pq * 2 + (pq == 0 ? slot0 : 0)) * BN * 128 +
                                   c0 * 128;
#pragma unroll
                for (int j = 0; j < kUnit<SWAP>; ++j) tmp[q][j] = __ldcg(src + j * 128);
              }
            }
          };
          const int cs = NH * U;  // this thread's units: half * U, + cs, ...
          load_batch(half * U, 0);
          // prefill orientation: the token's 1/rms (folded norm) and its sum of
          // squares over the tile (EPI_RESID_SQ; one thread covers the tile)
          float rs = 1.f, ss = 0.f;
          if constexpr (!SWAP && kEpiNorm<EPI>) rs = prefill_row_rs(a.e, arow);
          EpiIn in;  // inputs of the current unit; those of the next are fetched ahead
          if (use_pre) in = pre;
          else epi_load<SWAP, EPI>(a, g, arow, brow + half * U, tok, in);
          in.rs = rs;
          for (int c0 = half * U; c0 < BN; c0 += cs) {
            EpiIn nxt;
            nxt.rs = rs;
            if constexpr (kEpiAhead<EPI>)
              if (c0 + cs < BN) epi_load<SWAP, EPI>(a, g, arow, brow + c0 + cs, tok, nxt);
            float v[16];
#pragma unroll
            for (int j = 0; j < kUnit<SWAP>; ++j) v[j] = 0.f;
            for (int s0 = 0; s0 < nseg; s0 += 4) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (s0 + q < nseg) {
#pragma unroll
                  for (int j = 0; j < kUnit<SWAP>; ++j) v[j] += tmp[q][j];
                }
              if (s0 + 4 < nseg) load_batch(c0, s0 + 4);
              else if (c0 + cs < BN) load_batch(c0 + cs, 0);
            }
            ss += epi_chunk<SWAP, EPI>(a, g, arow, brow + c0, tok, v, in);
            if constexpr (kEpiAhead<EPI>) in = nxt;
            else if (c0 + cs < BN) epi_load<SWAP, EPI>(a, g, arow, brow + c0 + cs, tok, in);
            in.rs = rs;
          }
          if constexpr (!SWAP && EPI == EPI_RESID_SQ) store_row_sq(a, arow, ib, 0, ss, true);
          if (threadIdx.x == 64) a.tickets[sg.tile] = 0;
        }
        bar_sync(1, ET);
      }
      ++seg;
    }
  }

  if (a.cluster_split > 1) {
    // every thread of the cluster: the pieces are in shared memory
    cluster_sync();
    if (warp >= 2) {
      constexpr int U = kUnit<SWAP>, NH = kEpiWarps<SWAP> / 4;
      const int rank = static_cast<int>(c % a.cluster_split);
      const int half = (warp - 2) >> 2;
      const int row = (warp & 3) * 32 + lane;
      const int64_t tile = c / a.cluster_split;
      int g, ia, ib;
      tile_coords(tile, g, ia, ib, true);
      const int arow = ia * 128 + row, brow = ib * BN;
      const uint32_t red_s = smem_u32(smem);
      // rank r sums and stores chunks r, r + s, ...; the pieces are added in
      // K order (rank 0 first), up to 4 remote loads in flight together
      // worker (half, rank) sums units c0 = (half * s + rank) * U, + NH * s * U, ...
      const int cfirst = (half * a.cluster_split + rank) * U;
      const int cstep = NH * a.cluster_split * U;
      EpiIn in;  // inputs of the current unit; those of the next are fetched ahead
      if (pre_ok) in = pre;
      else if (cfirst < BN) epi_load<SWAP, EPI>(a, g, arow, brow + cfirst, tok, in);
      for (int c0 = cfirst; c0 < BN; c0 += cstep) {
        EpiIn nxt;
        if constexpr (kEpiAhead<EPI>)
          if (c0 + cstep < BN) epi_load<SWAP, EPI>(a, g, arow, brow + c0 + cstep, tok, nxt);
        float v[16];
        for (int r0 = 0; r0 < a.cluster_split; r0 += 4) {
          float p[4][16];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (r0 + q < a.cluster_split) {
#pragma unroll
              for (int j = 0; j < kUnit<SWAP>; ++j)
                p[q][j] = ld_shared_cluster(mapa_shared(red_s + ((c0 + j) * 128 + row) * 4, r0 + q));
            }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (r0 + q < a.cluster_split) {
#pragma unroll
              for (int j = 0; j < kUnit<SWAP>; ++j) v[j] = (r0 + q == 0) ? p[q][j] : v[j] + p[q][j];
            }
        }
        epi_chunk<SWAP, EPI>(a, g, arow, brow + c0, tok, v, in);
        if constexpr (kEpiAhead<EPI>) in = nxt;
        else if (c0 + cstep < BN) epi_load<SWAP, EPI>(a, g, arow, brow + c0 + cstep, tok, in);
      }
    }
    cluster_sync();  // keep every piece readable until the sums are done
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, a.tmem_cols);
  }
}

}  // namespace tpk
