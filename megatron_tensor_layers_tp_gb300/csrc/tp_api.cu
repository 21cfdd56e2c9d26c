// Host side of the C ABI declared in include/tp.h: configuration rules, shard
// construction, TMA descriptors, work planning and kernel dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "tp.h"

using namespace tpk;

// Output-feature tile widths of the prefill orientation, widest first.
constexpr int kPrefillBNs[] = {256, 224, 192, 160, 128};
constexpr int kNumPrefillBN = 5;
constexpr int kPrefillBN = kPrefillBNs[0];

struct ShardedLinear {
  uint16_t* data = nullptr;  // [t][rows][cols]
  uint16_t* bias = nullptr;  // optional: [ranks][rows] (column-parallel) or [rows] (row-parallel)
  int rows = 0, cols = 0;    // per rank
  int ranks = 0;             // t, or attn_tp for the attention block
  CUtensorMap tm_a;          // box (64, 128, 1): weight on the MMA M side (decode)
  CUtensorMap tm_b[kNumPrefillBN];  // box (64, kPrefillBNs[i], 1): weight on the MMA N side (prefill)
  CUtensorMap tm_h[kNumPrefillBN];  // box (64, kPrefillBNs[i] / 2, 1): one CTA's half (CTA pairs)
};

struct LayerShards {
  ShardedLinear qkv, gate_up, o, down;
  // qkv and gate_up with the preceding RMSNorm's weight folded into their
  // columns (W[n][k] * w[k]): the decoder layer's GEMMs read these, and the
  // raw hidden state; tp_column_linear keeps the plain shards
  ShardedLinear qkv_folded, gate_up_folded;
  uint16_t* attn_norm = nullptr;
  uint16_t* mlp_norm = nullptr;
};

struct tp_model {
  tp_config_t cfg;
  int device = 0;
  int num_sms = 0;
  bool host_coherent = false;  // the GPU reaches host memory coherently (NVLink-C2C)
  std::vector<LayerShards> layers;
  uint16_t* embed = nullptr;  // [Vp][H] = t shards of [Vp/t][H]
  ShardedLinear lm;
  uint16_t* final_norm = nullptr;
  uint16_t* ones = nullptr;  // [H] bf16 1.0: the norm weight once it is folded
  float2* rope = nullptr;
  int* status = nullptr;
  std::vector<std::pair<void*, size_t>> allocs;  // device buffers and their sizes
  mutable tp_stats_t stats;
  // per-launch timing (tp_profile)
  bool profiling = false;
  struct Rec { const char* name; cudaEvent_t a, b; };
  mutable std::vector<Rec> recs;
  mutable std::vector<cudaEvent_t> pool;
  mutable size_t pool_used = 0;
};

namespace {

constexpr int kAttnWholeMaxTiles = 128;  // decode attention: whole pairs up to this many key tiles per CTA
constexpr int kNormInGemmTokens = 32;  // folded RMSNorm applied inside the GEMM up to here
constexpr size_t kAlign = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int cdiv(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 tensor map (inner K, rows, slices) with a (64, box_rows, 1) box and
// 128-byte swizzle; reads outside the extents return zeros.
// When the slices sit closer together than the rows (rank shards side by side
// in one [rows, t*K] buffer), the dimensions are ordered (K, slice, rows) so
// the strides increase; *slice_mid reports which order was used.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint64_t slices,
               uint64_t row_stride_bytes, uint64_t slice_stride_bytes, uint32_t box_rows,
               int* slice_mid = nullptr) {
  auto enc = get_encoder();
  if (!enc) return false;
  const bool mid = slices > 1 && slice_stride_bytes < row_stride_bytes;
  if (slice_mid) *slice_mid = mid ? 1 : 0;
  if (mid && !slice_mid) return false;
  cuuint64_t dims[3] = {inner, rows, slices};
  cuuint64_t strides[2] = {row_stride_bytes, slice_stride_bytes};
  cuuint32_t box[3] = {64, box_rows, 1};
  if (mid) {
    dims[1] = slices; dims[2] = rows;
    strides[0] = slice_stride_bytes; strides[1] = row_stride_bytes;
    box[1] = 1; box[2] = box_rows;
  }
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor map of a weight shard stored in K blocks, [ranks][cols / 64][rows][64]
// bf16: dims (64, rows, cols / 64, ranks), box (64, box_rows, 1, 1), 128-byte
// swizzle.  A box at (0, row, K block, rank) is box_rows x 128 contiguous
// bytes, the same tile (and shared-memory image) the row-major layout's
// (K step x 64, row, rank) box gives.
bool make_tmap_kblocked(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                        uint64_t ranks, uint32_t box_rows) {
  auto enc = get_encoder();
  if (!enc || cols % 64) return false;
  cuuint64_t dims[4] = {64, rows, cols / 64, ranks};
  cuuint64_t strides[3] = {128, rows * 128, rows * cols * 2};
  cuuint32_t box[4] = {64, box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

tp_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return TP_OK;
  if (e == cudaErrorMemoryAllocation) return TP_ERR_OOM;
  return TP_ERR_CUDA;
}

#define TP_CHECK_CUDA(expr)                         \
  do {                                              \
    cudaError_t _e = (expr);                        \
    if (_e != cudaSuccess) return cuda_status(_e);  \
  } while (0)

constexpr size_t kMaxProfiled = 16384;

// Every kernel launch of the library goes through here: counted, and timed
// with two events on the launch stream while profiling is enabled.
template <class F>
cudaError_t launch(const tp_model* m, const char* name, cudaStream_t st, F&& f) {
  m->stats.kernel_launches++;
  if (!m->profiling || m->recs.size() >= kMaxProfiled) return f();
  while (m->pool.size() < m->pool_used + 2) {
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreate(&ev);
    if (e != cudaSuccess) return e;
    m->pool.push_back(ev);
  }
  cudaEvent_t a = m->pool[m->pool_used++], b = m->pool[m->pool_used++];
  cudaError_t e = cudaEventRecord(a, st);
  if (e != cudaSuccess) return e;
  e = f();
  if (e != cudaSuccess) return e;
  m->recs.push_back({name, a, b});
  return cudaEventRecord(b, st);
}

template <class T>
tp_status dev_alloc(tp_model* m, T** p, size_t bytes) {
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
  if (e != cudaSuccess) return cuda_status(e);
  m->allocs.push_back({q, bytes});
  *p = static_cast<T*>(q);
  return TP_OK;
}

// ---------------------------------------------------------------- planning
struct GemmPlan {
  bool swap;
  bool pair;  // prefill orientation on CTA pairs
  int BN, stages, tmem_cols;
  size_t smem;
};

int prefill_bn_index(int bn) {
  for (int i = 0; i < kNumPrefillBN; ++i)
    if (kPrefillBNs[i] == bn) return i;
  return -1;
}

GemmPlan plan_gemm(int M, int bn = kPrefillBN, bool pair = false) {
  GemmPlan p;
  p.swap = M <= kSwapMaxTokens;
  p.pair = !p.swap && pair;
  p.BN = p.swap ? std::max(16, cdiv(M, 16) * 16) : bn;
  // one CTA's stage: 128 rows of A and its rows of B (half of them on a pair)
  const int stage = 128 * 128 + (p.pair ? p.BN / 2 : p.BN) * 128;
  const int budget = 200 * 1024;
  p.stages = std::min(8, budget / stage);
  int cols = 32;
  while (cols < 2 * p.BN) cols *= 2;
  p.tmem_cols = cols;
  p.smem = 1024 + (size_t)p.stages * stage + (2 * p.stages + 5) * 8 + 16 + 5 * kSwapMaxTokens * 4;
  return p;
}

// Prefill orientation: whether a GEMM runs on CTA pairs, and its
// output-feature tile width.
//  - CTA pairs (tcgen05 cta_group::2, tiles of 256 token rows) when the GEMM
//    has at least one whole wave of pair tiles at width 256: per SM they move
//    a third less operand data per K step than a single CTA's 128 x 256 tile,
//    and the single-CTA kernel is bound by that traffic.  Fewer tiles than
//    that run on single CTAs (the remainder stream-K over every SM).
//  - Whole tiles run in waves, so a GEMM whose tile count is just above a
//    multiple of the slots (SMs, or co-resident pairs) idles most of them in
//    its last wave (Llama-8B o_proj at 2048 tokens: 128 pair tiles of 256 on
//    76 pairs = 1.7 waves).  The width taken is the one whose
//    waves x (width + 16) is least (the 16 a per-tile cost, so that a narrower
//    tile pays only when it saves a wave: 224 gives that o_proj 152 pair
//    tiles, exactly 2 waves).
// cfg.prefill_bn fixes the width, cfg.prefill_cta_pairs the kernel.
struct PrefillChoice {
  int bi;     // index into kPrefillBNs
  bool pair;
};

int pair_slots(const tp_model* m, int epi) {
  const GemmPlan p = plan_gemm(kSwapMaxTokens + 1, kPrefillBN, true);
  return gemm_max_clusters(false, true, epi, 2, p.smem);
}

PrefillChoice choose_prefill(const tp_model* m, int epi, int64_t groups, int M, int rows) {
  const int mode = m->cfg.prefill_cta_pairs;  // 0 auto, 1 always, 2 never
  const int P = mode == 2 ? 0 : pair_slots(m, epi);
  PrefillChoice ch;
  ch.pair = P > 0 && (mode == 1 || groups * cdiv(M, 256) * cdiv(rows, kPrefillBN) >= P);
  const int64_t G = ch.pair ? P : m->num_sms;
  const int64_t a_tiles = cdiv(M, ch.pair ? 256 : 128);
  ch.bi = 0;
  if (m->cfg.prefill_bn) {
    ch.bi = prefill_bn_index(m->cfg.prefill_bn);
    return ch;
  }
  if (groups * a_tiles * cdiv(rows, kPrefillBNs[0]) < G) return ch;
  int64_t best_cost = INT64_MAX;
  for (int i = 0; i < kNumPrefillBN; ++i) {
    const int64_t tiles = groups * a_tiles * cdiv(rows, kPrefillBNs[i]);
    if (tiles < G) continue;
    const int64_t cost = (tiles + G - 1) / G * (kPrefillBNs[i] + 16);
    if (cost < best_cost) { best_cost = cost; ch.bi = i; }
  }
  return ch;
}

// Decode orientation: the flat (tile, K step) range is split evenly over the
// grid (stream-K): the weights are read once whatever the split.  Prefill
// orientation: whole tiles in data-parallel waves (all CTAs walk K together,
// so operand slices are shared through L2), and only the tiles of the last
// partial wave are split stream-K.
//
// Decode orientation with few output tiles: a cluster of s CTAs per tile, each
// taking 1/s of K, pieces added in K order through distributed shared memory
// (no global partials, no tail fix-up).  Used when the tiles x s CTAs cover at
// least 80% of the SMs and all those clusters can be resident at once.
// The stream-K fix-up's divisions as multiply-shifts when every flat index
// times the grid fits 31 bits (after the schedule is set).
void set_fix32(GemmArgs& a) {
  const int64_t n_tiles = (int64_t)a.n_groups * a.a_tiles * a.b_tiles;
  const int64_t K = (int64_t)a.k_slices * a.k_iters_slice;
  const int Gs = a.sk_ctas > 0 ? a.sk_ctas : a.grid;
  a.fix32 = n_tiles * K * std::max(a.grid, 1) < ((int64_t)1 << 31) ? 1 : 0;
  if (a.total_iters <= 0) a.fix32 = 0;  // no stream-K part: nothing to divide by
  if (a.fix32) {
    a.div_total = make_fastdiv(static_cast<uint32_t>(a.total_iters));
    a.div_sk = make_fastdiv(static_cast<uint32_t>(Gs));
    a.div_k = make_fastdiv(static_cast<uint32_t>(K));
    a.div_a = make_fastdiv(static_cast<uint32_t>(a.a_tiles));
    a.div_b = make_fastdiv(static_cast<uint32_t>(a.b_tiles));
  }
}

void set_schedule(GemmArgs& a, const GemmPlan& p, int num_sms, int epi) {
  const int64_t n_tiles = (int64_t)a.n_groups * a.a_tiles * a.b_tiles;
  const int64_t K = (int64_t)a.k_slices * a.k_iters_slice;
  a.cluster_split = 1;
  if (p.pair) {
    // CTA pairs: whole tiles, pair p takes tiles p, p + P, ...
    a.pair = 1;
    const int P = gemm_max_clusters(false, true, epi, 2, p.smem);
    a.grid = 2 * (int)std::min<int64_t>(std::max(P, 1), n_tiles);
    a.dp_waves = 0;
    a.total_iters = 0;
    return;
  }
  // Up to 16 tokens the pieces are small (8 KB per 128-row tile) and
  // stream-K over every SM wins (measured, same box, alternating runs:
  // Llama-8B decode layer 111.5 -> 110.7 us); at 64 tokens the cluster split
  // does (Qwen-32B layer 279.5 vs 285.3 us).
  if (p.swap && p.BN > 16) {
    // the largest cluster (8 CTAs at most, portable) whose tiles x s CTAs fill
    // at least 65% of the SMs in one wave (measured: a cluster split beats
    // stream-K's fix-up from there on); the occupancy query decides whether
    // that many clusters are co-resident on this part's GPCs
    for (int s = 8; s >= 2; --s) {
      if (n_tiles * s > num_sms || n_tiles * s * 100 < (int64_t)num_sms * 65 || K < 2 * s) continue;
      if (gemm_max_clusters(true, false, epi, s, p.smem) < n_tiles) continue;
      a.cluster_split = s;
      a.dp_waves = 0;
      a.total_iters = 0;
      a.grid = (int)(n_tiles * s);
      return;
    }
  }
  if (p.swap || n_tiles < num_sms) {
    a.dp_waves = 0;
    a.total_iters = n_tiles * K;
    a.grid = (int)std::min<int64_t>(num_sms, a.total_iters);
  } else {
    // data-parallel waves of whole tiles, the remainder as a last, partial
    // wave of whole tiles (one per CTA).  Measured against cutting the
    // remainder evenly over every CTA (stream-K): the fp32 partials of a
    // 128 x 256 tile and their reduction cost more than the idle SMs of the
    // last wave (prefill GEMMs 0.65 -> 0.73 of the sustained bf16 peak).
    a.grid = num_sms;
    a.dp_waves = (int)(n_tiles / num_sms);
    const int64_t rem = n_tiles - (int64_t)a.dp_waves * num_sms;
    a.total_iters = rem * K;
    a.sk_ctas = (int)rem;
  }
}

// Workspace regions (all offsets 256-byte aligned).
struct WsLayout {
  size_t gemm_tickets, attn_tickets, gemm_partials, attn_partials, u, q, o, act, hs, rank_partials,
      norm_sq, total;
};

// slots of per-32-feature sums of squares a row-parallel GEMM leaves for the
// next RMSNorm (decode orientation): 4 per 128-row output tile
int norm_slots(const tp_config_t& c) { return cdiv(c.hidden, 128) * 4; }

// Sums of squares a producer can leave per token: the decode GEMMs'
// norm_slots, two per output tile in the prefill orientation (at least
// ceil(H / 128) tiles), or the embedding's four.
int norm_sq_slots_max(const tp_config_t& c) {
  return std::max(norm_slots(c), (2 * cdiv(c.hidden, kPrefillBNs[kNumPrefillBN - 1]) + 3) / 4 * 4);
}

size_t max_gemm_tiles(const tp_config_t& c, int M) {
  // upper bound over every GEMM of the model for M tokens
  const int H = c.hidden, d = c.head_dim, t = c.t;
  const int nqkv = (c.q_heads_per_rank + 2 * c.kv_heads_per_rank) * d;
  const int rows[4] = {nqkv, 2 * c.inter_per_rank, H, std::max(c.vocab_per_rank, 1)};
  size_t best = 0;
  for (int r : rows) {
    // decode orientation
    best = std::max(best, (size_t)t * cdiv(r, 128));
    // prefill orientation
    best = std::max(best, (size_t)t * cdiv(M, 128) * cdiv(r, kPrefillBNs[kNumPrefillBN - 1]));
  }
  return best;
}

WsLayout ws_layout(const tp_model* m, int M) {
  const tp_config_t& c = m->cfg;
  WsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  };
  const int G = m->num_sms;
  L.gemm_tickets = take(max_gemm_tiles(c, M) * sizeof(int));
  L.attn_tickets = take((size_t)std::max(M, 1) * c.n_kv_heads * sizeof(int));
  L.gemm_partials = take((size_t)G * 2 * kPrefillBN * 128 * sizeof(float));
  L.attn_partials = take((size_t)G * 2 * attn_decode_partial_floats(c.head_dim) * sizeof(float));
  L.u = take((size_t)M * c.hidden * 2);
  L.q = take((size_t)M * c.n_heads * c.head_dim * 2);
  L.o = take((size_t)M * c.n_heads * c.head_dim * 2);
  L.act = take((size_t)M * c.intermediate * 2);
  L.hs = take((size_t)M * c.hidden * 2);
  L.rank_partials = take((size_t)c.t * M * c.hidden * sizeof(float));
  L.norm_sq = take((size_t)std::max(M, 1) * norm_sq_slots_max(c) * sizeof(float));  // [token][slot]
  L.total = off;
  return L;
}

bool ws_ok(const tp_model* m, int M, const void* ws, size_t bytes) {
  return ws != nullptr && aligned16(ws) && bytes >= ws_layout(m, M).total;
}

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

EpiArgs base_epi(const tp_model* m, int M) {
  EpiArgs e;
  memset(&e, 0, sizeof(e));
  e.M = M;
  e.head_dim = m->cfg.head_dim;
  e.q_heads_per_rank = m->cfg.q_heads_per_rank;
  e.kv_heads_per_rank = m->cfg.kv_heads_per_rank;
  e.kv_replicas = m->cfg.kv_replicas;
  e.inter_per_rank = m->cfg.inter_per_rank;
  e.vocab = m->cfg.vocab;
  e.vocab_per_rank = m->cfg.vocab_per_rank;
  return e;
}

// Column-parallel family (qkv, gate_up, LM head): each rank r produces its own
// [M, rows] output from the replicated x [M, K].  Fills the arguments and the
// schedule of one GEMM launch.
tp_status prep_column(const tp_model* m, const ShardedLinear& W, const uint16_t* x, int64_t ldx,
                      int M, int epi, const EpiArgs& e, void* ws, const WsLayout& L, GemmArgs& a,
                      GemmPlan& p) {
  const int K = W.cols;
  PrefillChoice ch{0, false};
  if (M > kSwapMaxTokens) ch = choose_prefill(m, epi, W.ranks, M, W.rows);
  p = plan_gemm(M, kPrefillBNs[ch.bi], ch.pair);
  memset(&a, 0, sizeof(a));
  bool ok;
  if (p.swap) {
    a.tmA = W.tm_a;
    ok = make_tmap(&a.tmB, x, K, M, 1, ldx * 2, (uint64_t)ldx * 2 * M, p.BN);
    a.a_tiles = cdiv(W.rows, 128);
    a.b_tiles = 1;
    a.a_slice_mode = 1;
    a.b_slice_mode = 0;
    a.a_rows_valid = W.rows;
    a.b_rows_valid = M;
    a.a_policy = 1;
    a.b_policy = 2;
  } else {
    ok = make_tmap(&a.tmA, x, K, M, 1, ldx * 2, (uint64_t)ldx * 2 * M, 128);
    a.tmB = p.pair ? W.tm_h[ch.bi] : W.tm_b[ch.bi];
    a.a_tiles = cdiv(M, p.pair ? 256 : 128);
    a.b_tiles = cdiv(W.rows, p.BN);
    a.a_slice_mode = 0;
    a.b_slice_mode = 1;
    a.a_rows_valid = M;
    a.b_rows_valid = W.rows;
  }
  if (!ok) return TP_ERR_CUDA;
  a.BN = p.BN;
  a.stages = p.stages;
  a.tmem_cols = p.tmem_cols;
  a.n_groups = W.ranks;
  a.k_slices = 1;
  a.k_iters_slice = cdiv(K, 64);
  set_schedule(a, p, m->num_sms, epi);
  set_fix32(a);
  a.partials = at<float>(ws, L.gemm_partials);
  a.tickets = at<int>(ws, L.gemm_tickets);
  a.status = m->status;
  a.e = e;
  a.e.bias = W.bias;  // rank g's rows carry their own bias entries
  a.e.bias_group_stride = W.rows;
  return TP_OK;
}

tp_status run_column(const tp_model* m, const char* name, const ShardedLinear& W,
                     const uint16_t* x, int64_t ldx, int M, int epi, const EpiArgs& e, void* ws,
                     const WsLayout& L, cudaStream_t st) {
  if (M == 0) return TP_OK;
  GemmArgs a;
  GemmPlan p;
  tp_status s = prep_column(m, W, x, ldx, M, epi, e, ws, L, a, p);
  if (s != TP_OK) return s;
  return cuda_status(launch(m, name, st, [&] { return launch_gemm(p.swap, epi, a, p.smem, st); }));
}

// Row-parallel family (o_proj, down_proj): rank r holds W_r [H, K_r] and reads
// x_r [M, K_r]; fused = sum over ranks inside the GEMM (epilogue EPI_RESID),
// otherwise per-rank fp32 partials then the ordered reduction kernel.
tp_status prep_row(const tp_model* m, const ShardedLinear& W, const uint16_t* x,
                   int64_t x_rank_stride, int64_t ldx, int M, const uint16_t* residual,
                   uint16_t* y, int fused, void* ws, const WsLayout& L, float* sq_out,
                   GemmArgs& a, GemmPlan& p, int& epi) {
  const tp_config_t& c = m->cfg;
  const int Kr = W.cols, H = W.rows, t = W.ranks;
  // fused: one output group (the ranks are summed in K); unfused: t groups
  PrefillChoice ch{0, false};
  if (M > kSwapMaxTokens)
    ch = choose_prefill(m, fused ? EPI_RESID : EPI_PARTIAL, fused ? 1 : t, M, H);
  p = plan_gemm(M, kPrefillBNs[ch.bi], ch.pair);
  memset(&a, 0, sizeof(a));
  const uint64_t xs_bytes = (uint64_t)x_rank_stride * 2;
  bool ok;
  if (p.swap) {
    a.tmA = W.tm_a;
    ok = make_tmap(&a.tmB, x, Kr, M, t, ldx * 2, xs_bytes, p.BN, &a.b_slice_mid);
    a.a_tiles = cdiv(H, 128);
    a.b_tiles = 1;
    a.a_rows_valid = H;
    a.b_rows_valid = M;
    a.a_policy = 1;
    a.b_policy = 2;
  } else {
    ok = make_tmap(&a.tmA, x, Kr, M, t, ldx * 2, xs_bytes, 128, &a.a_slice_mid);
    a.tmB = p.pair ? W.tm_h[ch.bi] : W.tm_b[ch.bi];
    a.a_tiles = cdiv(M, p.pair ? 256 : 128);
    a.b_tiles = cdiv(H, p.BN);
    a.a_rows_valid = M;
    a.b_rows_valid = H;
  }
  if (!ok) return TP_ERR_CUDA;
  a.BN = p.BN;
  a.stages = p.stages;
  a.tmem_cols = p.tmem_cols;
  a.k_iters_slice = cdiv(Kr, 64);
  a.partials = at<float>(ws, L.gemm_partials);
  a.tickets = at<int>(ws, L.gemm_tickets);
  a.status = m->status;
  a.e = base_epi(m, M);
  float* rp = at<float>(ws, L.rank_partials);
  if (fused) {
    a.n_groups = 1;
    a.k_slices = t;  // ranks folded into K, in rank order
    a.a_slice_mode = 2;
    a.b_slice_mode = 2;
    a.e.out = y;
    a.e.ld_out = H;
    a.e.residual = residual;
    a.e.ld_res = H;
    a.e.bias = W.bias;  // once: the ranks are already summed in the accumulator
    a.e.bias_group_stride = 0;
    a.e.sq_out = sq_out;  // sums of squares for the next RMSNorm
    a.e.sq_ld = p.swap ? norm_slots(c) : (2 * a.b_tiles + 3) / 4 * 4;  // a multiple of 4
    epi = a.e.sq_out ? EPI_RESID_SQ : EPI_RESID;
  } else {
    a.n_groups = t;
    a.k_slices = 1;
    a.a_slice_mode = 1;
    a.b_slice_mode = 1;
    a.e.out = rp;
    a.e.ld_out = H;
    a.e.out_group_stride = (int64_t)M * H;
    epi = EPI_PARTIAL;
  }
  set_schedule(a, p, m->num_sms, epi);
  set_fix32(a);
  return TP_OK;
}

// sq_out: where the fused reduction leaves each token's sums of squares
// for the next RMSNorm (or null); *sq_slots: how many per token it left
// (0: none).
tp_status run_row(const tp_model* m, const char* name, const ShardedLinear& W, const uint16_t* x,
                  int64_t x_rank_stride, int64_t ldx, int M, const uint16_t* residual,
                  uint16_t* y, int fused, void* ws, const WsLayout& L, cudaStream_t st,
                  float* sq_out = nullptr, int* sq_slots = nullptr) {
  if (sq_slots) *sq_slots = 0;
  if (M == 0) return TP_OK;
  const int H = W.rows, t = W.ranks;
  GemmArgs a;
  GemmPlan p;
  int epi = 0;
  tp_status s = prep_row(m, W, x, x_rank_stride, ldx, M, residual, y, fused, ws, L, sq_out, a, p, epi);
  if (s != TP_OK) return s;
  float* rp = at<float>(ws, L.rank_partials);
  TP_CHECK_CUDA(launch(m, name, st, [&] { return launch_gemm(p.swap, epi, a, p.smem, st); }));
  if (sq_slots && epi == EPI_RESID_SQ) *sq_slots = a.e.sq_ld;
  if (!fused) {
    TP_CHECK_CUDA(launch(m, "reduce_ranks", st, [&] {
      return launch_reduce_ranks(rp, (int64_t)M * H, t, M, H, W.bias, residual, y, st);
    }));
  }
  m->stats.allreduces++;
  m->stats.allreduce_payload_bytes += (int64_t)M * H * 2;
  return TP_OK;
}

// Releases one buffer obtained from dev_alloc (after the stream work that
// reads it has finished).
void dev_free(tp_model* m, void* p) {
  for (size_t i = 0; i < m->allocs.size(); ++i)
    if (m->allocs[i].first == p) {
      cudaFree(p);
      m->allocs.erase(m->allocs.begin() + i);
      return;
    }
}

bool valid_layer(const tp_model* m, int layer) {
  return m && layer >= 0 && layer < (int)m->layers.size();
}

// One sharded weight of `ranks` x [rows][cols].  The loader fills it row-major
// (copy_rows launches); reblock_linear then moves it into K blocks and encodes
// its tensor maps.
tp_status alloc_linear(tp_model* m, ShardedLinear* L, int rows, int cols, int ranks) {
  L->rows = rows;
  L->cols = cols;
  L->ranks = ranks;
  return dev_alloc(m, &L->data, (size_t)ranks * rows * cols * 2);
}

// Row-major shard -> [ranks][cols / 64][rows][64] (a new buffer; the old one
// is freed) and the tensor maps of both GEMM orientations over it.  Measured
// in isolation (8-stage TMA ring, 152 CTAs, a [28672][4096] bf16 matrix):
// 37.7 us row-major, 36.4 us in K blocks.
tp_status reblock_linear(tp_model* m, ShardedLinear* L, cudaStream_t st) {
  uint16_t* kb = nullptr;
  tp_status s = dev_alloc(m, &kb, (size_t)L->ranks * L->rows * L->cols * 2);
  if (s != TP_OK) return s;
  if (launch_reblock_k64(kb, L->data, L->ranks, L->rows, L->cols, st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess) {
    dev_free(m, kb);
    return TP_ERR_CUDA;
  }
  dev_free(m, L->data);
  L->data = kb;
  if (!make_tmap_kblocked(&L->tm_a, L->data, L->rows, L->cols, L->ranks, 128)) return TP_ERR_CUDA;
  for (int i = 0; i < kNumPrefillBN; ++i) {
    if (!make_tmap_kblocked(&L->tm_b[i], L->data, L->rows, L->cols, L->ranks, kPrefillBNs[i]) ||
        !make_tmap_kblocked(&L->tm_h[i], L->data, L->rows, L->cols, L->ranks, kPrefillBNs[i] / 2))
      return TP_ERR_CUDA;
  }
  return TP_OK;
}

struct MapUploader {
  std::vector<int32_t*> bufs;
  ~MapUploader() {
    for (auto* b : bufs) cudaFree(b);
  }
  tp_status upload(const std::vector<int32_t>& v, int32_t** out, cudaStream_t st) {
    int32_t* d = nullptr;
    cudaError_t e = cudaMalloc(&d, std::max<size_t>(v.size(), 1) * 4);
    if (e != cudaSuccess) return cuda_status(e);
    bufs.push_back(d);
    e = cudaMemcpyAsync(d, v.data(), v.size() * 4, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_status(e);
    *out = d;
    return TP_OK;
  }
};

}  // namespace

// ============================================================================
// C ABI
// ============================================================================
namespace tpk {
int gemm_max_clusters(bool swap, bool pair, int epi, int cluster_x, size_t smem) {
  // per (kernel, epilogue, cluster size, smem): the answer never changes
  static std::mutex mu;
  static std::vector<std::pair<uint64_t, int>> cache;
  const uint64_t key = ((uint64_t)smem << 16) | ((uint64_t)cluster_x << 8) | ((uint64_t)epi << 2) |
                       (pair ? 2u : 0u) | (swap ? 1u : 0u);
  std::lock_guard<std::mutex> lock(mu);
  for (auto& kv : cache)
    if (kv.first == key) return kv.second;
  int n = 0;
  switch (epi) {
    case 0: n = gemm_max_clusters_epi0(swap, pair, cluster_x, smem); break;
    case 1: n = gemm_max_clusters_epi1(swap, pair, cluster_x, smem); break;
    case 2: n = gemm_max_clusters_epi2(swap, pair, cluster_x, smem); break;
    case 3: n = gemm_max_clusters_epi3(swap, pair, cluster_x, smem); break;
    case 4: n = gemm_max_clusters_epi4(swap, pair, cluster_x, smem); break;
    case 5: n = gemm_max_clusters_epi5(swap, pair, cluster_x, smem); break;
    case 6: n = gemm_max_clusters_epi6(swap, pair, cluster_x, smem); break;
    case 7: n = gemm_max_clusters_epi7(swap, pair, cluster_x, smem); break;
  }
  cache.push_back({key, n});
  return n;
}

cudaError_t launch_gemm(bool swap, int epi, const GemmArgs& a, size_t smem, cudaStream_t st) {
  switch (epi) {
    case 0: return launch_gemm_epi0(swap, a, smem, st);
    case 1: return launch_gemm_epi1(swap, a, smem, st);
    case 2: return launch_gemm_epi2(swap, a, smem, st);
    case 3: return launch_gemm_epi3(swap, a, smem, st);
    case 4: return launch_gemm_epi4(swap, a, smem, st);
    case 5: return launch_gemm_epi5(swap, a, smem, st);
    case 6: return launch_gemm_epi6(swap, a, smem, st);
    case 7: return launch_gemm_epi7(swap, a, smem, st);
  }
  return cudaErrorInvalidValue;
}
}  // namespace tpk

extern "C" {

const char* tp_strerror(tp_status s) {
  switch (s) {
    case TP_OK: return "ok";
    case TP_ERR_ARG: return "invalid argument";
    case TP_ERR_DIVISIBILITY: return "dimension not divisible by the number of ranks";
    case TP_ERR_KV_REPLICA: return "KV heads can be neither split evenly nor replicated evenly";
    case TP_ERR_TOKEN_RANGE: return "token id outside [0, vocab)";
    case TP_ERR_OOM: return "device allocation failed";
    case TP_ERR_CUDA: return "CUDA runtime error";
    case TP_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case TP_ERR_UNSUPPORTED: return "shape outside the kernels' envelope";
    case TP_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

tp_status tp_config(tp_config_t* c) {
  if (!c) return TP_ERR_ARG;
  if (c->t < 1 || c->hidden < 1 || c->n_heads < 1 || c->n_kv_heads < 1 || c->head_dim < 1 ||
      c->intermediate < 1 || c->vocab < 0 || c->n_layers < 0 || c->max_positions < 1 ||
      !(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f))
    return TP_ERR_ARG;
  const int t = c->t;
  if (c->attn_dp < 0 || c->host_io < 0 || c->host_io > 1 || c->plain_column_shards < 0 ||
      c->plain_column_shards > 1 || (c->prefill_bn != 0 && prefill_bn_index(c->prefill_bn) < 0) ||
      c->prefill_cta_pairs < 0 || c->prefill_cta_pairs > 2)
    return TP_ERR_ARG;
  if (c->attn_dp == 0) c->attn_dp = 1;
  if (t % c->attn_dp) return TP_ERR_DIVISIBILITY;
  const int at = t / c->attn_dp;  // attention ranks per DP group
  if (c->n_heads % c->n_kv_heads) return TP_ERR_DIVISIBILITY;
  if (c->n_heads % at) return TP_ERR_DIVISIBILITY;
  if (c->intermediate % t) return TP_ERR_DIVISIBILITY;
  int kv_r, reps;
  if (c->n_kv_heads >= at) {
    if (c->n_kv_heads % at) return TP_ERR_KV_REPLICA;
    kv_r = c->n_kv_heads / at;
    reps = 1;
  } else {
    if (at % c->n_kv_heads) return TP_ERR_KV_REPLICA;
    kv_r = 1;
    reps = at / c->n_kv_heads;
  }
  const int vp = (c->vocab + t - 1) / t * t;
  c->vocab_padded = vp;
  c->vocab_per_rank = vp / t;
  c->attn_tp = at;
  c->q_heads_per_rank = c->n_heads / at;
  c->kv_heads_per_rank = kv_r;
  c->kv_replicas = reps;
  c->kv_copies = std::min(at, c->n_kv_heads);
  c->inter_per_rank = c->intermediate / t;
  // kernel envelope
  if (t > 8) return TP_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return TP_ERR_UNSUPPORTED;
  if (c->hidden % 64 || (c->q_heads_per_rank * c->head_dim) % 64 || c->inter_per_rank % 64)
    return TP_ERR_UNSUPPORTED;
  if (c->n_heads / c->n_kv_heads > 16) return TP_ERR_UNSUPPORTED;
  return TP_OK;
}

tp_status tp_model_bytes(const tp_model* m, int64_t* bytes) {
  if (!m || !bytes) return TP_ERR_ARG;
  int64_t n = 0;
  for (const auto& a : m->allocs) n += (int64_t)a.second;
  *bytes = n;
  return TP_OK;
}

tp_status tp_get_config(const tp_model* m, tp_config_t* out) {
  if (!m || !out) return TP_ERR_ARG;
  *out = m->cfg;
  return TP_OK;
}

void tp_free(tp_model* m) {
  if (!m) return;
  for (cudaEvent_t e : m->pool) cudaEventDestroy(e);
  for (auto& a : m->allocs) cudaFree(a.first);
  delete m;
}

tp_status tp_profile(tp_model* m, int32_t enable) {
  if (!m) return TP_ERR_ARG;
  m->profiling = enable != 0;
  return TP_OK;
}

tp_status tp_profile_read(tp_model* m, void* stream, tp_kernel_time_t* out, int32_t max,
                          int32_t* n) {
  if (!m || !n || (max > 0 && !out)) return TP_ERR_ARG;
  TP_CHECK_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  std::vector<tp_kernel_time_t> agg;
  for (const auto& r : m->recs) {
    float ms = 0.f;
    TP_CHECK_CUDA(cudaEventElapsedTime(&ms, r.a, r.b));
    size_t i = 0;
    while (i < agg.size() && strncmp(agg[i].name, r.name, sizeof(agg[i].name)) != 0) ++i;
    if (i == agg.size()) {
      tp_kernel_time_t k;
      memset(&k, 0, sizeof(k));
      strncpy(k.name, r.name, sizeof(k.name) - 1);
      agg.push_back(k);
    }
    agg[i].launches++;
    agg[i].total_ms += ms;
  }
  m->recs.clear();
  m->pool_used = 0;
  *n = 0;
  for (size_t i = 0; i < agg.size() && (int32_t)i < max; ++i) out[(*n)++] = agg[i];
  return TP_OK;
}

tp_status tp_load_shards(const tp_config_t* cfg_in, const tp_weights_t* w, void* stream,
                         tp_model** out) {
  if (!cfg_in || !w || !out) return TP_ERR_ARG;
  *out = nullptr;
  tp_config_t cfg = *cfg_in;
  tp_status s = tp_config(&cfg);
  if (s != TP_OK) return s;
  if (cfg.n_layers > 0 && !w->layers) return TP_ERR_ARG;
  for (int l = 0; l < cfg.n_layers; ++l) {
    const tp_layer_weights_t& L = w->layers[l];
    if (!L.attn_norm || !L.wq || !L.wk || !L.wv || !L.wo || !L.mlp_norm || !L.wg || !L.wu || !L.wd)
      return TP_ERR_ARG;
  }
  if ((w->embed || w->lm_head || w->final_norm) && cfg.vocab < 1) return TP_ERR_ARG;
  if (!get_encoder()) return TP_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  tp_model* m = new tp_model();
  m->cfg = cfg;
  memset(&m->stats, 0, sizeof(m->stats));
  auto fail = [&](tp_status e) {
    cudaStreamSynchronize(st);
    tp_free(m);
    return e;
  };
  if (cudaGetDevice(&m->device) != cudaSuccess) return fail(TP_ERR_CUDA);
  if (cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device) != cudaSuccess)
    return fail(TP_ERR_CUDA);
  {
    // a coherent host link (NVLink-C2C): native atomics over the link and
    // pageable host memory reached through the host's page tables; a PCIe
    // GPU lacks the second, and there zero-copy reads would be slow
    int atomics = 0, host_pt = 0;
    if (cudaDeviceGetAttribute(&atomics, cudaDevAttrHostNativeAtomicSupported, m->device) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&host_pt, cudaDevAttrPageableMemoryAccessUsesHostPageTables,
                               m->device) != cudaSuccess)
      return fail(TP_ERR_CUDA);
    m->host_coherent = atomics != 0 && host_pt != 0 && cfg.host_io == 0;
  }
  // the attention block is sharded over the attn_tp ranks of a DP group, the
  // MLP over all t ranks
  const int t = cfg.t, at = cfg.attn_tp, H = cfg.hidden, d = cfg.head_dim;
  const int nq = cfg.q_heads_per_rank, kvr = cfg.kv_heads_per_rank, Ipr = cfg.inter_per_rank;
  MapUploader up;
  if ((s = dev_alloc(m, &m->status, 256)) != TP_OK) return fail(s);
  if (cudaMemsetAsync(m->status, 0, 256, st) != cudaSuccess) return fail(TP_ERR_CUDA);
  if ((s = dev_alloc(m, &m->rope, (size_t)cfg.max_positions * (d / 2) * sizeof(float2))) != TP_OK)
    return fail(s);
  if (launch_rope_table(m->rope, cfg.max_positions, d, (double)cfg.rope_theta, st) != cudaSuccess)
    return fail(TP_ERR_CUDA);

  auto kv_head_of = [&](int r, int local) {
    return cfg.kv_replicas == 1 ? r * kvr + local : r / cfg.kv_replicas;
  };
  // position inside a RoPE head of shard row w: the two halves of pair j sit at 2j, 2j+1
  auto rope_src = [&](int w_) { return (w_ & 1) ? (w_ >> 1) + d / 2 : (w_ >> 1); };

  m->layers.resize(cfg.n_layers);
  for (int l = 0; l < cfg.n_layers; ++l) {
    const tp_layer_weights_t& Wl = w->layers[l];
    LayerShards& Ls = m->layers[l];
    const int nqkv = (nq + 2 * kvr) * d;
    if ((s = alloc_linear(m, &Ls.qkv, nqkv, H, at)) != TP_OK) return fail(s);
    if ((s = alloc_linear(m, &Ls.gate_up, 2 * Ipr, H, t)) != TP_OK) return fail(s);
    if ((s = alloc_linear(m, &Ls.o, H, nq * d, at)) != TP_OK) return fail(s);
    if ((s = alloc_linear(m, &Ls.down, H, Ipr, t)) != TP_OK) return fail(s);
    for (int r = 0; r < at; ++r) {
      // qkv: [its Q heads | its KV heads] with RoPE pairs adjacent; V in natural order
      std::vector<int32_t> mq(nq * d), mk(kvr * d), mv(kvr * d);
      for (int hl = 0; hl < nq; ++hl)
        for (int w_ = 0; w_ < d; ++w_) mq[hl * d + w_] = (r * nq + hl) * d + rope_src(w_);
      for (int kl = 0; kl < kvr; ++kl)
        for (int w_ = 0; w_ < d; ++w_) {
          mk[kl * d + w_] = kv_head_of(r, kl) * d + rope_src(w_);
          mv[kl * d + w_] = kv_head_of(r, kl) * d + w_;
        }
      int32_t *dq, *dk, *dv;
      if ((s = up.upload(mq, &dq, st)) != TP_OK || (s = up.upload(mk, &dk, st)) != TP_OK ||
          (s = up.upload(mv, &dv, st)) != TP_OK)
        return fail(s);
      uint16_t* base = Ls.qkv.data + (size_t)r * nqkv * H;
      if (launch_copy_rows(base, H, Wl.wq, H, dq, nq * d, H, st) != cudaSuccess ||
          launch_copy_rows(base + (size_t)nq * d * H, H, Wl.wk, H, dk, kvr * d, H, st) != cudaSuccess ||
          launch_copy_rows(base + (size_t)(nq + kvr) * d * H, H, Wl.wv, H, dv, kvr * d, H, st) !=
              cudaSuccess)
        return fail(TP_ERR_CUDA);
      // biases follow their rows (one element per row; a missing part is zero)
      if (Wl.bq || Wl.bk || Wl.bv) {
        if (!Ls.qkv.bias && (s = dev_alloc(m, &Ls.qkv.bias, (size_t)at * nqkv * 2)) != TP_OK)
          return fail(s);
        int32_t *nq_, *nk_;
        std::vector<int32_t> zq(nq * d, -1), zk(kvr * d, -1);
        if ((s = up.upload(zq, &nq_, st)) != TP_OK || (s = up.upload(zk, &nk_, st)) != TP_OK)
          return fail(s);
        uint16_t* bb = Ls.qkv.bias + (size_t)r * nqkv;
        if (launch_copy_rows(bb, 1, Wl.bq, 1, Wl.bq ? dq : nq_, nq * d, 1, st) != cudaSuccess ||
            launch_copy_rows(bb + nq * d, 1, Wl.bk, 1, Wl.bk ? dk : nk_, kvr * d, 1, st) !=
                cudaSuccess ||
            launch_copy_rows(bb + (nq + kvr) * d, 1, Wl.bv, 1, Wl.bv ? dv : nk_, kvr * d, 1, st) !=
                cudaSuccess)
          return fail(TP_ERR_CUDA);
      }
    }
    for (int r = 0; r < t; ++r) {
      // gate_up: row 2j = gate row r*Ipr + j, row 2j+1 = up row r*Ipr + j
      std::vector<int32_t> mg(Ipr);
      for (int j = 0; j < Ipr; ++j) mg[j] = r * Ipr + j;
      int32_t* dg;
      if ((s = up.upload(mg, &dg, st)) != TP_OK) return fail(s);
      uint16_t* gbase = Ls.gate_up.data + (size_t)r * 2 * Ipr * H;
      if (launch_copy_rows(gbase, 2 * H, Wl.wg, H, dg, Ipr, H, st) != cudaSuccess ||
          launch_copy_rows(gbase + H, 2 * H, Wl.wu, H, dg, Ipr, H, st) != cudaSuccess)
        return fail(TP_ERR_CUDA);
      if (Wl.bg || Wl.bu) {
        if (!Ls.gate_up.bias && (s = dev_alloc(m, &Ls.gate_up.bias, (size_t)t * 2 * Ipr * 2)) != TP_OK)
          return fail(s);
        int32_t* ng_;
        std::vector<int32_t> zg(Ipr, -1);
        if ((s = up.upload(zg, &ng_, st)) != TP_OK) return fail(s);
        uint16_t* gb = Ls.gate_up.bias + (size_t)r * 2 * Ipr;
        if (launch_copy_rows(gb, 2, Wl.bg, 1, Wl.bg ? dg : ng_, Ipr, 1, st) != cudaSuccess ||
            launch_copy_rows(gb + 1, 2, Wl.bu, 1, Wl.bu ? dg : ng_, Ipr, 1, st) != cudaSuccess)
          return fail(TP_ERR_CUDA);
      }
    }
    // row-parallel biases: whole [H] vectors, added once after the reduction
    for (auto [src, dst] : {std::make_pair(Wl.bo, &Ls.o.bias), std::make_pair(Wl.bd, &Ls.down.bias)}) {
      if (!src) continue;
      if ((s = dev_alloc(m, dst, (size_t)H * 2)) != TP_OK) return fail(s);
      if (cudaMemcpyAsync(*dst, src, (size_t)H * 2, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return fail(TP_ERR_CUDA);
    }
    // row-parallel shards: columns [r K_r, (r+1) K_r) of wo / wd
    std::vector<int32_t> ident(H);
    for (int i = 0; i < H; ++i) ident[i] = i;
    int32_t* di;
    if ((s = up.upload(ident, &di, st)) != TP_OK) return fail(s);
    for (int r = 0; r < at; ++r)
      if (launch_copy_rows(Ls.o.data + (size_t)r * H * nq * d, nq * d, Wl.wo + (size_t)r * nq * d,
                           (int64_t)cfg.n_heads * d, di, H, nq * d, st) != cudaSuccess)
        return fail(TP_ERR_CUDA);
    for (int r = 0; r < t; ++r)
      if (launch_copy_rows(Ls.down.data + (size_t)r * H * Ipr, Ipr, Wl.wd + (size_t)r * Ipr,
                           cfg.intermediate, di, H, Ipr, st) != cudaSuccess)
        return fail(TP_ERR_CUDA);
    if ((s = dev_alloc(m, &Ls.attn_norm, (size_t)H * 2)) != TP_OK ||
        (s = dev_alloc(m, &Ls.mlp_norm, (size_t)H * 2)) != TP_OK)
      return fail(s);
    if (cudaMemcpyAsync(Ls.attn_norm, Wl.attn_norm, (size_t)H * 2, cudaMemcpyDeviceToDevice, st) !=
            cudaSuccess ||
        cudaMemcpyAsync(Ls.mlp_norm, Wl.mlp_norm, (size_t)H * 2, cudaMemcpyDeviceToDevice, st) !=
            cudaSuccess)
      return fail(TP_ERR_CUDA);
    // the norms' weights folded into the column-parallel GEMMs that read them;
    // a norm weight of exactly 1 leaves the shard unchanged, and then the one
    // buffer serves the decoder layer and tp_column_linear alike
    bool shared_fold[2] = {false, false};  // the folded shard is the plain one
    for (int which = 0; which < 2; ++which) {
      ShardedLinear& plain = which == 0 ? Ls.qkv : Ls.gate_up;
      ShardedLinear& folded = which == 0 ? Ls.qkv_folded : Ls.gate_up_folded;
      const uint16_t* nw = which == 0 ? Wl.attn_norm : Wl.mlp_norm;
      std::vector<uint16_t> hw(H);
      if (cudaMemcpyAsync(hw.data(), nw, (size_t)H * 2, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
          cudaStreamSynchronize(st) != cudaSuccess)
        return fail(TP_ERR_CUDA);
      bool unit = true;
      for (uint16_t v : hw) unit = unit && v == 0x3F80;  // bf16 1.0
      if (unit) {
        shared_fold[which] = true;
        continue;
      }
      if ((s = alloc_linear(m, &folded, plain.rows, H, plain.ranks)) != TP_OK) return fail(s);
      folded.bias = plain.bias;
      if (launch_fold_cols(folded.data, plain.data, nw, (int64_t)plain.ranks * plain.rows, H, st) !=
          cudaSuccess)
        return fail(TP_ERR_CUDA);
      if (!cfg.plain_column_shards) {
        // tp_column_linear is not served for this layer: drop the unfolded copy
        if (cudaStreamSynchronize(st) != cudaSuccess) return fail(TP_ERR_CUDA);
        dev_free(m, plain.data);
        plain.data = nullptr;
      }
    }
    // every shard of the layer into K blocks
    for (ShardedLinear* Lw : {&Ls.qkv, &Ls.gate_up, &Ls.o, &Ls.down, &Ls.qkv_folded, &Ls.gate_up_folded})
      if (Lw->data && (s = reblock_linear(m, Lw, st)) != TP_OK) return fail(s);
    if (shared_fold[0]) Ls.qkv_folded = Ls.qkv;
    if (shared_fold[1]) Ls.gate_up_folded = Ls.gate_up;
  }
  {
    const std::vector<uint16_t> one(H, 0x3F80);  // bf16 1.0
    if ((s = dev_alloc(m, &m->ones, (size_t)H * 2)) != TP_OK) return fail(s);
    if (cudaMemcpyAsync(m->ones, one.data(), (size_t)H * 2, cudaMemcpyHostToDevice, st) != cudaSuccess)
      return fail(TP_ERR_CUDA);
  }
  // vocab-parallel tables: padded to Vp rows, shard r = rows [r Vp/t, (r+1) Vp/t)
  if (w->embed || w->lm_head) {
    std::vector<int32_t> mv(cfg.vocab_padded);
    for (int v = 0; v < cfg.vocab_padded; ++v) mv[v] = v < cfg.vocab ? v : -1;
    int32_t* dmv;
    if ((s = up.upload(mv, &dmv, st)) != TP_OK) return fail(s);
    if (w->embed) {
      if ((s = dev_alloc(m, &m->embed, (size_t)cfg.vocab_padded * H * 2)) != TP_OK) return fail(s);
      if (launch_copy_rows(m->embed, H, w->embed, H, dmv, cfg.vocab_padded, H, st) != cudaSuccess)
        return fail(TP_ERR_CUDA);
    }
    if (w->lm_head) {
      if ((s = alloc_linear(m, &m->lm, cfg.vocab_per_rank, H, t)) != TP_OK) return fail(s);
      if (launch_copy_rows(m->lm.data, H, w->lm_head, H, dmv, cfg.vocab_padded, H, st) != cudaSuccess)
        return fail(TP_ERR_CUDA);
      if ((s = reblock_linear(m, &m->lm, st)) != TP_OK) return fail(s);
    }
  }
  if (w->final_norm) {
    if ((s = dev_alloc(m, &m->final_norm, (size_t)H * 2)) != TP_OK) return fail(s);
    if (cudaMemcpyAsync(m->final_norm, w->final_norm, (size_t)H * 2, cudaMemcpyDeviceToDevice, st) !=
        cudaSuccess)
      return fail(TP_ERR_CUDA);
  }
  if (cudaStreamSynchronize(st) != cudaSuccess) return fail(TP_ERR_CUDA);
  *out = m;
  return TP_OK;
}

size_t tp_workspace_bytes(const tp_model* m, int32_t max_tokens) {
  if (!m || max_tokens < 0) return 0;
  return ws_layout(m, std::max(max_tokens, 1)).total;
}

tp_status tp_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws) return TP_ERR_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

tp_status tp_column_linear(const tp_model* m, int32_t layer, int32_t which, const tp_bf16* x,
                           int32_t M, tp_bf16* y, int64_t y_rank_stride, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!valid_layer(m, layer) || (which != TP_QKV && which != TP_GATE_UP) || M < 0) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if (!x || !y || !aligned16(x) || !aligned16(y) || y_rank_stride % 8) return TP_ERR_ARG;
  const ShardedLinear& W = which == TP_QKV ? m->layers[layer].qkv : m->layers[layer].gate_up;
  if (!W.data) return TP_ERR_UNSUPPORTED;  // only the norm-folded shards were kept
  if (y_rank_stride < (int64_t)M * W.rows) return TP_ERR_ARG;
  if (!ws_ok(m, M, ws, ws_bytes)) return TP_ERR_WORKSPACE;
  EpiArgs e = base_epi(m, M);
  e.out = y;
  e.ld_out = W.rows;
  e.out_group_stride = y_rank_stride;
  e.which = which == TP_QKV ? 0 : 1;
  return run_column(m, "gemm_column", W, x, m->cfg.hidden, M, EPI_PLAIN, e, ws, ws_layout(m, M),
                    static_cast<cudaStream_t>(stream));
}

tp_status tp_row_linear_reduce(const tp_model* m, int32_t layer, int32_t which,
                               const tp_bf16* x, int64_t x_rank_stride, int64_t ldx, int32_t M,
                               const tp_bf16* residual, tp_bf16* y, int32_t fused, void* ws,
                               size_t ws_bytes, void* stream) {
  if (!valid_layer(m, layer) || (which != TP_O && which != TP_DOWN) || M < 0) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  const ShardedLinear& W = which == TP_O ? m->layers[layer].o : m->layers[layer].down;
  if (!x || !y || !aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)) ||
      x_rank_stride % 8 || ldx % 8 || ldx < W.cols)
    return TP_ERR_ARG;
  if (!ws_ok(m, M, ws, ws_bytes)) return TP_ERR_WORKSPACE;
  return run_row(m, "gemm_row", W, x, x_rank_stride, ldx, M, residual, y, fused, ws, ws_layout(m, M),
                 static_cast<cudaStream_t>(stream));
}

// The vocab-parallel lookup (counted as its all-reduce); sq (or null): each
// row's sum of squares in the [token][4 slots] form for the next RMSNorm.
static tp_status embed_rows(const tp_model* m, const int32_t* ids, int M, uint16_t* h, float* sq,
                            cudaStream_t st) {
  m->stats.allreduces++;
  m->stats.allreduce_payload_bytes += (int64_t)M * m->cfg.hidden * 2;
  return cuda_status(launch(m, "vocab_embed", st, [&] {
    return launch_embed(m->embed, m->cfg.vocab, m->cfg.vocab_per_rank, m->cfg.t, ids, M,
                        m->cfg.hidden, h, sq, m->status, st);
  }));
}

tp_status tp_vocab_embed(const tp_model* m, const int32_t* ids, int32_t M, tp_bf16* h,
                         void* stream) {
  if (!m || M < 0) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if (!m->embed || !ids || !h || !aligned16(h)) return TP_ERR_ARG;
  return embed_rows(m, ids, M, h, nullptr, static_cast<cudaStream_t>(stream));
}

static void count_gather(const tp_model* m, int S) {
  m->stats.allgathers++;
  const tp_config_t& c = m->cfg;
  m->stats.allgather_recv_bytes_per_rank +=
      (int64_t)S * ((int64_t)(c.t - 1) * c.vocab * 2 / c.t);
}

tp_status tp_lm_head_gather(const tp_model* m, const tp_bf16* x, int32_t S, tp_bf16* logits,
                            int64_t ld_logits, void* ws, size_t ws_bytes, void* stream) {
  if (!m || S < 0) return TP_ERR_ARG;
  if (S == 0) return TP_OK;
  if (!m->lm.data || !x || !logits || !aligned16(x) || ld_logits < m->cfg.vocab) return TP_ERR_ARG;
  if (!ws_ok(m, S, ws, ws_bytes)) return TP_ERR_WORKSPACE;
  EpiArgs e = base_epi(m, S);
  e.out = logits;
  e.ld_out = ld_logits;
  count_gather(m, S);
  return run_column(m, "gemm_lm_head", m->lm, x, m->cfg.hidden, S, EPI_LOGITS, e, ws, ws_layout(m, S),
                    static_cast<cudaStream_t>(stream));
}

tp_status tp_rmsnorm(const tp_model* m, const tp_bf16* x, const tp_bf16* w, int32_t M,
                     tp_bf16* y, void* stream) {
  if (!m || M < 0) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if (!x || !w || !y || !aligned16(x) || !aligned16(w) || !aligned16(y)) return TP_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_status(launch(m, "rmsnorm", st, [&] {
    return launch_rmsnorm(x, m->cfg.hidden, nullptr, w, M, m->cfg.hidden, m->cfg.rms_eps, y,
                          m->cfg.hidden, st, false);
  }));
}

static tp_status check_batch(const tp_model* m, const tp_batch_t* b) {
  if (!b || b->n_seqs < 1 || b->n_tokens < 1 || !b->positions || !b->token_seq || !b->k_cache ||
      !b->v_cache || b->l_max < 1 || b->max_ctx < 1 || b->max_ctx > b->l_max ||
      b->max_ctx > m->cfg.max_positions || b->l_max > m->cfg.max_positions)
    return TP_ERR_ARG;
  if (b->mode == TP_DECODE) {
    if (b->n_tokens != b->n_seqs) return TP_ERR_ARG;
  } else if (b->mode == TP_PREFILL) {
    if (!b->seq_start || b->max_q_per_seq < 1) return TP_ERR_ARG;
  } else {
    return TP_ERR_ARG;
  }
  return TP_OK;
}

// Arguments of the decode / prefill attention over the batch's caches; the
// decode grid is chosen for num_ctas SMs.
static tp_status prep_attention(const tp_model* m, const tp_batch_t* b, uint16_t* kc, uint16_t* vc,
                                const uint16_t* q, uint16_t* o, void* ws, const WsLayout& L,
                                int num_ctas, AttnArgs& a) {
  const tp_config_t& c = m->cfg;
  const int d = c.head_dim, nhd = c.n_heads * d;
  memset(&a, 0, sizeof(a));
  const uint64_t slices = (uint64_t)c.kv_copies * b->n_seqs * c.kv_heads_per_rank;
  if (!make_tmap(&a.tmK, kc, d, b->l_max, slices, (uint64_t)d * 2, (uint64_t)b->l_max * d * 2, 64) ||
      !make_tmap(&a.tmV, vc, d, b->l_max, slices, (uint64_t)d * 2, (uint64_t)b->l_max * d * 2, 64))
    return TP_ERR_CUDA;
  a.q = q;
  a.ld_q = nhd;
  a.o = o;
  a.ld_o = nhd;
  a.k_cache = kc;  // also the decode kernel's L2 prefetch of cache tiles
  a.v_cache = vc;
  a.positions = b->positions;
  a.seq_start = b->seq_start;
  a.n_seqs = b->n_seqs;
  a.n_heads = c.n_heads;
  a.n_kv = c.n_kv_heads;
  a.head_dim = d;
  a.kv_r = c.kv_heads_per_rank;
  a.group = c.n_heads / c.n_kv_heads;
  a.l_max = b->l_max;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)d));
  a.status = m->status;
  if (b->mode == TP_DECODE) {
    a.tiles_per_bg = cdiv(b->max_ctx, 64);
    a.total_units = (int64_t)b->n_seqs * c.n_kv_heads * a.tiles_per_bg;
    // Whole (sequence, KV head) pairs per CTA when they can be dealt out
    // evenly to at least 80% of the SMs and a CTA's share stays within
    // kAttnWholeMaxTiles key tiles: no pair is then split and no partial
    // result needs combining.  Otherwise split the flat range evenly over the
    // SMs (measured: whole pairs win by 8.5 us at 16 tiles per CTA and by
    // 4.5 us at 64, tie at 128, and lose by 4 us at 256, where the longer
    // streams amortise the combine).
    const int64_t n_bg = (int64_t)b->n_seqs * c.n_kv_heads;
    int grid = (int)std::min<int64_t>(num_ctas, a.total_units);
    for (int64_t dd = 1; dd <= n_bg; ++dd) {
      if (n_bg % dd) continue;
      const int64_t g = n_bg / dd;
      if (g <= num_ctas) {
        if (g * 5 >= (int64_t)num_ctas * 4 && dd * a.tiles_per_bg <= kAttnWholeMaxTiles)
          grid = (int)g;
        break;
      }
    }
    a.grid = grid;
    a.idx32 = a.total_units * grid < ((int64_t)1 << 31) ? 1 : 0;
    if (a.idx32) {
      a.div_units = make_fastdiv(static_cast<uint32_t>(a.total_units));
      a.div_grid = make_fastdiv(static_cast<uint32_t>(grid));
      a.div_tb = make_fastdiv(static_cast<uint32_t>(a.tiles_per_bg));
      a.div_kv = make_fastdiv(static_cast<uint32_t>(c.n_kv_heads));
    }
    a.stages = attn_decode_stages(d, a.group);
    if (a.stages < 2) return TP_ERR_UNSUPPORTED;
    a.partials = at<float>(ws, L.attn_partials);
    a.tickets = at<int>(ws, L.attn_tickets);
  }
  return TP_OK;
}

// The epilogue arguments of the qkv projection: RoPE, q into its buffer, the
// new K/V rows into the rank caches.
static EpiArgs qkv_epi(const tp_model* m, const tp_batch_t* b, int M, uint16_t* q, uint16_t* kc,
                       uint16_t* vc) {
  const tp_config_t& c = m->cfg;
  EpiArgs e = base_epi(m, M);
  e.out = q;
  e.ld_out = c.n_heads * c.head_dim;
  e.k_cache = kc;
  e.v_cache = vc;
  e.kv_copy_stride = (int64_t)b->n_seqs * c.kv_heads_per_rank * b->l_max * c.head_dim;
  e.n_seqs = b->n_seqs;
  e.l_max = b->l_max;
  e.positions = b->positions;
  e.token_seq = b->token_seq;
  e.rope = m->rope;
  return e;
}

// h_sq: on entry, how many partial sums of squares per token of h's rows sit
// in the workspace (left by the previous layer's down_proj or by the
// embedding; 0: none); on exit, how many this layer's down_proj left for the
// next.
static tp_status layer_forward(const tp_model* m, int layer, const tp_batch_t* b, uint16_t* h,
                               int fused, void* ws, const WsLayout& L, cudaStream_t st,
                               int* h_sq) {
  const tp_config_t& c = m->cfg;
  const LayerShards& Ls = m->layers[layer];
  const int M = b->n_tokens, H = c.hidden, d = c.head_dim;
  const int nhd = c.n_heads * d;
  uint16_t* u = at<uint16_t>(ws, L.u);
  uint16_t* q = at<uint16_t>(ws, L.q);
  uint16_t* o = at<uint16_t>(ws, L.o);
  uint16_t* act = at<uint16_t>(ws, L.act);
  uint16_t* kc = b->k_cache[layer];
  uint16_t* vc = b->v_cache[layer];
  if (!kc || !vc || !aligned16(kc) || !aligned16(vc)) return TP_ERR_ARG;
  tp_status s;
  // Each RMSNorm's weight is folded into the GEMM after it (qkv_folded,
  // gate_up_folded).  That GEMM reads h itself and scales each token's
  // outputs by its 1/rms, which its epilogue gets
  //  - in the decode orientation up to kNormInGemmTokens tokens by reading
  //    h's rows while the weights stream (every CTA reads all M rows from L2);
  //  - otherwise from the partial sums of squares that the fused row-parallel
  //    GEMM (or the embedding) that wrote h left in the workspace (decode
  //    orientation measured: a ~1 us loss at 16 tokens from the extra epilogue
  //    work in o_proj / down_proj, a gain at 64; prefill orientation: two norm
  //    kernels of ~10 us each fewer per layer);
  //  - where neither applies (the layer's first norm without such sums, the
  //    unfused reduction) u = h / rms(h) runs first.
  const bool swap = plan_gemm(M).swap;
  const bool leaves_sq = fused != 0 && (!swap || M > kNormInGemmTokens);  // o_proj, down_proj
  float* sq = at<float>(ws, L.norm_sq);
  auto norm_in = [&](EpiArgs& e_, int have_sq, const uint16_t** xin) -> tp_status {
    e_.norm_src = h;
    e_.norm_ld = H;
    e_.norm_width = H;
    e_.norm_eps = c.rms_eps;
    e_.norm_partials = sq;
    e_.norm_slots = have_sq;
    *xin = h;
    if (swap && M <= kNormInGemmTokens) { e_.norm_mode = 1; return TP_OK; }
    if (have_sq > 0) { e_.norm_mode = 2; return TP_OK; }
    e_.norm_mode = 0;
    *xin = u;
    return cuda_status(launch(m, "rmsnorm", st, [&] {
      return launch_rmsnorm(h, H, nullptr, m->ones, M, H, c.rms_eps, u, H, st, true);
    }));
  };
  const uint16_t* xin = nullptr;
  // qkv (column-parallel) + RoPE + K/V into the rank caches
  EpiArgs e = qkv_epi(m, b, M, q, kc, vc);
  if ((s = norm_in(e, *h_sq, &xin)) != TP_OK) return s;
  AttnArgs a;
  if ((s = prep_attention(m, b, kc, vc, q, o, ws, L, m->num_sms, a)) != TP_OK) return s;
  if (b->mode == TP_DECODE && swap) {
    // Decode: the qkv GEMM only leaves its stream-K pieces (no arrival
    // tickets, no fix-up at its end); each attention CTA sums the pieces of
    // its own sequence and KV head and finishes the qkv epilogue (norm, bias,
    // RoPE, new K/V cache row) while its cache tiles stream in.
    GemmArgs g;
    GemmPlan p;
    if ((s = prep_column(m, Ls.qkv_folded, xin, H, M, EPI_QKV_PIECES, e, ws, L, g, p)) != TP_OK)
      return s;
    const int64_t n_tiles = (int64_t)g.n_groups * g.a_tiles * g.b_tiles;
    g.cluster_split = 1;
    g.dp_waves = 0;
    g.sk_ctas = 0;
    g.total_iters = n_tiles * g.k_slices * g.k_iters_slice;
    g.grid = (int)std::min<int64_t>(m->num_sms, g.total_iters);
    set_fix32(g);
    // every CTA's range spans at most two tiles when there are no more tiles
    // than CTAs; the attention kernel locates pieces in 32-bit arithmetic
    if (n_tiles <= g.grid && g.total_iters * g.grid < (int64_t)1 << 31) {
      TP_CHECK_CUDA(launch(m, "gemm_qkv", st, [&] {
        return launch_gemm(true, EPI_QKV_PIECES, g, p.smem, st);
      }));
      a.qkv_pieces = 1;
      a.pc = g.partials;
      a.pc_total = g.total_iters;
      a.pc_grid = g.grid;
      a.pc_k = g.k_slices * g.k_iters_slice;
      a.pc_div_total = make_fastdiv(static_cast<uint32_t>(a.pc_total));
      a.pc_div_grid = make_fastdiv(static_cast<uint32_t>(a.pc_grid));
      a.pc_div_q = make_fastdiv(static_cast<uint32_t>(c.q_heads_per_rank));
      a.pc_bn = g.BN;
      a.pc_a_tiles = g.a_tiles;
      a.nqkv_r = Ls.qkv_folded.rows;
      a.q_per_rank = c.q_heads_per_rank;
      a.kv_replicas = c.kv_replicas;
      a.qkv_bias = Ls.qkv_folded.bias;
      a.rope = m->rope;
      a.k_cache = kc;
      a.v_cache = vc;
      a.kv_copy_stride = e.kv_copy_stride;
      a.norm_mode = e.norm_mode;
      a.norm_src = e.norm_src;
      a.norm_ld = e.norm_ld;
      a.norm_width = e.norm_width;
      a.norm_eps = e.norm_eps;
      a.norm_partials = e.norm_partials;
      a.norm_slots = e.norm_slots;
    }
  }
  if (!a.qkv_pieces &&
      (s = run_column(m, "gemm_qkv", Ls.qkv_folded, xin, H, M, EPI_QKV, e, ws, L, st)) != TP_OK)
    return s;
  // attention
  if (b->mode == TP_DECODE) {
    TP_CHECK_CUDA(launch(m, "attn_decode", st, [&] { return launch_attn_decode(a, st); }));
  } else {
    const int nqb = cdiv(b->max_q_per_seq, 64);
    TP_CHECK_CUDA(launch(m, "attn_prefill", st, [&] { return launch_attn_prefill(a, nqb, st); }));
  }
  // o_proj (row-parallel) + reduction ① + residual
  int o_sq = 0;
  if ((s = run_row(m, "gemm_o", Ls.o, o, c.q_heads_per_rank * d, nhd, M, h, h, fused, ws, L, st,
                   leaves_sq ? sq : nullptr, &o_sq)) != TP_OK)
    return s;
  // DP attention: every group's hidden rows are gathered for the MLP (one
  // buffer here; counted as each rank receiving the other groups' rows)
  if (c.attn_dp > 1) {
    m->stats.dp_gathers++;
    m->stats.dp_gather_recv_bytes_per_rank += (int64_t)(c.attn_dp - 1) * M * H * 2 / c.attn_dp;
  }
  // RMSNorm(h) folded as above; gate_up (column-parallel) + SiLU(gate) * up
  EpiArgs e2 = base_epi(m, M);
  if ((s = norm_in(e2, o_sq, &xin)) != TP_OK) return s;
  e2.out = act;
  e2.ld_out = c.intermediate;
  if ((s = run_column(m, "gemm_gate_up", Ls.gate_up_folded, xin, H, M, EPI_SILU, e2, ws, L, st)) !=
      TP_OK)
    return s;
  // down_proj (row-parallel) + reduction ② + residual
  return run_row(m, "gemm_down", Ls.down, act, c.inter_per_rank, c.intermediate, M, h, h, fused, ws,
                 L, st, leaves_sq ? sq : nullptr, h_sq);
}

tp_status tp_layer_forward(const tp_model* m, int32_t layer, const tp_batch_t* b,
                           tp_bf16* h_inout, int32_t fused, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!valid_layer(m, layer) || !h_inout || !aligned16(h_inout)) return TP_ERR_ARG;
  tp_status s = check_batch(m, b);
  if (s != TP_OK) return s;
  if (!ws_ok(m, b->n_tokens, ws, ws_bytes)) return TP_ERR_WORKSPACE;
  int h_sq = 0;  // the caller's h comes without sums of squares
  return layer_forward(m, layer, b, h_inout, fused, ws, ws_layout(m, b->n_tokens),
                       static_cast<cudaStream_t>(stream), &h_sq);
}

// The device address of pinned (page-locked) host memory, or false for any
// other pointer.
static bool pinned_device_ptr(const void* p, void** out) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return false;
  *out = at.devicePointer;
  return true;
}

tp_status tp_layer_forward_host(const tp_model* m, int32_t layer, const tp_batch_t* b,
                                const tp_bf16* h_in_host, tp_bf16* h_out_host, tp_bf16* h_dev,
                                int32_t fused, void* ws, size_t ws_bytes, void* stream) {
  if (!valid_layer(m, layer) || !h_in_host || !h_out_host || !h_dev || !aligned16(h_dev) ||
      !aligned16(h_in_host) || !aligned16(h_out_host))
    return TP_ERR_ARG;
  tp_status s = check_batch(m, b);
  if (s != TP_OK) return s;
  if (!ws_ok(m, b->n_tokens, ws, ws_bytes)) return TP_ERR_WORKSPACE;
  void *din = nullptr, *dout = nullptr;
  if (!pinned_device_ptr(h_in_host, &din) || !pinned_device_ptr(h_out_host, &dout))
    return TP_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)b->n_tokens * m->cfg.hidden * 2;  // H % 64 == 0: a multiple of 16
  if (m->host_coherent) {
    TP_CHECK_CUDA(launch(m, "host_in", st, [&] { return launch_host_copy(din, h_dev, bytes, false, st); }));
  } else {
    TP_CHECK_CUDA(cudaMemcpyAsync(h_dev, h_in_host, bytes, cudaMemcpyHostToDevice, st));
  }
  int h_sq = 0;
  if ((s = layer_forward(m, layer, b, h_dev, fused, ws, ws_layout(m, b->n_tokens), st, &h_sq)) !=
      TP_OK)
    return s;
  if (m->host_coherent)
    return cuda_status(
        launch(m, "host_out", st, [&] { return launch_host_copy(h_dev, dout, bytes, true, st); }));
  return cuda_status(cudaMemcpyAsync(h_out_host, h_dev, bytes, cudaMemcpyDeviceToHost, st));
}

// Layers [first, first + n) on h; the embedding first when ids is set, the
// final norm and the LM head after when logits is set.  tp_forward is the
// single stage covering every layer.
static tp_status stage_forward(const tp_model* m, int first, int n, const int32_t* ids,
                               const tp_batch_t* b, tp_bf16* h, tp_bf16* logits,
                               int64_t ld_logits, int32_t fused, void* ws, size_t ws_bytes,
                               void* stream) {
  if (!m || !h || !aligned16(h) || first < 0 || n < 0 || first + n > m->cfg.n_layers)
    return TP_ERR_ARG;
  if (ids && (first != 0 || !m->embed)) return TP_ERR_ARG;
  if (logits && (first + n != m->cfg.n_layers || !m->lm.data || !m->final_norm)) return TP_ERR_ARG;
  tp_status s = check_batch(m, b);
  if (s != TP_OK) return s;
  if (logits && (!b->sample_rows || b->n_samples < 1 || ld_logits < m->cfg.vocab)) return TP_ERR_ARG;
  const int M = b->n_tokens;
  const int rows = logits ? std::max(M, b->n_samples) : M;
  if (!ws_ok(m, rows, ws, ws_bytes)) return TP_ERR_WORKSPACE;
  const WsLayout L = ws_layout(m, rows);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the embedding leaves each row's sum of squares for the first layer's
  // RMSNorm (four slots per token); a stage's input h comes without them
  int h_sq = 0;
  if (ids) {
    if ((s = embed_rows(m, ids, M, h, at<float>(ws, L.norm_sq), st)) != TP_OK) return s;
    h_sq = 4;
  }
  for (int l = first; l < first + n; ++l)
    if ((s = layer_forward(m, l, b, h, fused, ws, L, st, &h_sq)) != TP_OK) return s;
  if (!logits) return TP_OK;
  uint16_t* hs = at<uint16_t>(ws, L.hs);
  TP_CHECK_CUDA(launch(m, "rmsnorm_final", st, [&] {
    return launch_rmsnorm(h, m->cfg.hidden, b->sample_rows, m->final_norm, b->n_samples,
                          m->cfg.hidden, m->cfg.rms_eps, hs, m->cfg.hidden, st, true);
  }));
  EpiArgs e = base_epi(m, b->n_samples);
  e.out = logits;
  e.ld_out = ld_logits;
  count_gather(m, b->n_samples);
  return run_column(m, "gemm_lm_head", m->lm, hs, m->cfg.hidden, b->n_samples, EPI_LOGITS, e, ws, L, st);
}

tp_status tp_forward(const tp_model* m, const int32_t* ids, const tp_batch_t* b, tp_bf16* h,
                     tp_bf16* logits, int64_t ld_logits, int32_t fused, void* ws,
                     size_t ws_bytes, void* stream) {
  if (!m || !ids || !logits) return TP_ERR_ARG;
  return stage_forward(m, 0, m->cfg.n_layers, ids, b, h, logits, ld_logits, fused, ws, ws_bytes,
                       stream);
}

tp_status tp_stage_forward(const tp_model* m, int32_t first_layer, int32_t n_layers,
                           const int32_t* ids, const tp_batch_t* b, tp_bf16* h,
                           tp_bf16* logits, int64_t ld_logits, int32_t fused, void* ws,
                           size_t ws_bytes, void* stream) {
  return stage_forward(m, first_layer, n_layers, ids, b, h, logits, ld_logits, fused, ws,
                       ws_bytes, stream);
}

tp_status tp_stage_send(const tp_model* m, const tp_bf16* src, tp_bf16* dst, int32_t M,
                        void* stream) {
  if (!m || M < 0) return TP_ERR_ARG;
  const int H = m->cfg.hidden, t = m->cfg.t;
  if ((H / t) % 8 || H % t) return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  if (!src || !dst || !aligned16(src) || !aligned16(dst)) return TP_ERR_ARG;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(src), b0 = reinterpret_cast<uintptr_t>(dst);
  const uintptr_t bytes = (uintptr_t)M * H * 2;
  if (a0 < b0 + bytes && b0 < a0 + bytes) return TP_ERR_ARG;
  m->stats.stage_sends++;
  m->stats.stage_send_bytes += (int64_t)bytes;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_status(launch(m, "stage_send", st, [&] {
    return launch_stage_send(src, dst, M, H, t, st);
  }));
}

}  // extern "C"

struct tp_graph {
  const tp_model* m = nullptr;
  cudaGraphExec_t exec = nullptr;
  tp_stats_t delta;  // counters of the captured call, added on each replay
};

namespace {
template <class F>
tp_status capture_graph(const tp_model* m, void* stream, tp_graph** out, F&& body) {
  if (!m || !out || !stream || m->profiling) return TP_ERR_ARG;
  *out = nullptr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const tp_stats_t before = m->stats;
  TP_CHECK_CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeRelaxed));
  const tp_status s = body();
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(st, &graph);
  const tp_stats_t after = m->stats;
  m->stats = before;  // nothing ran yet
  if (s != TP_OK || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return s != TP_OK ? s : cuda_status(e);
  }
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ei = cudaGraphInstantiate(&exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess) return cuda_status(ei);
  tp_graph* g = new tp_graph;
  g->m = m;
  g->exec = exec;
  g->delta.allreduces = after.allreduces - before.allreduces;
  g->delta.allreduce_payload_bytes = after.allreduce_payload_bytes - before.allreduce_payload_bytes;
  g->delta.allgathers = after.allgathers - before.allgathers;
  g->delta.allgather_recv_bytes_per_rank =
      after.allgather_recv_bytes_per_rank - before.allgather_recv_bytes_per_rank;
  g->delta.kernel_launches = after.kernel_launches - before.kernel_launches;
  g->delta.stage_sends = after.stage_sends - before.stage_sends;
  g->delta.stage_send_bytes = after.stage_send_bytes - before.stage_send_bytes;
  g->delta.dp_gathers = after.dp_gathers - before.dp_gathers;
  g->delta.dp_gather_recv_bytes_per_rank =
      after.dp_gather_recv_bytes_per_rank - before.dp_gather_recv_bytes_per_rank;
  *out = g;
  return TP_OK;
}
}  // namespace

extern "C" {

tp_status tp_graph_capture_forward(const tp_model* m, const int32_t* ids, const tp_batch_t* b,
                                   tp_bf16* h, tp_bf16* logits, int64_t ld_logits,
                                   int32_t fused, void* ws, size_t ws_bytes, void* stream,
                                   tp_graph** out) {
  return capture_graph(m, stream, out, [&] {
    return tp_forward(m, ids, b, h, logits, ld_logits, fused, ws, ws_bytes, stream);
  });
}

tp_status tp_graph_capture_layer(const tp_model* m, int32_t layer, const tp_batch_t* b,
                                 tp_bf16* h_inout, int32_t fused, void* ws, size_t ws_bytes,
                                 void* stream, tp_graph** out) {
  return capture_graph(m, stream, out, [&] {
    return tp_layer_forward(m, layer, b, h_inout, fused, ws, ws_bytes, stream);
  });
}

tp_status tp_graph_launch(tp_graph* g, void* stream) {
  if (!g || !g->exec) return TP_ERR_ARG;
  TP_CHECK_CUDA(cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)));
  tp_stats_t& s = g->m->stats;
  s.allreduces += g->delta.allreduces;
  s.allreduce_payload_bytes += g->delta.allreduce_payload_bytes;
  s.allgathers += g->delta.allgathers;
  s.allgather_recv_bytes_per_rank += g->delta.allgather_recv_bytes_per_rank;
  s.kernel_launches += g->delta.kernel_launches;
  s.stage_sends += g->delta.stage_sends;
  s.stage_send_bytes += g->delta.stage_send_bytes;
  s.dp_gathers += g->delta.dp_gathers;
  s.dp_gather_recv_bytes_per_rank += g->delta.dp_gather_recv_bytes_per_rank;
  return TP_OK;
}

void tp_graph_free(tp_graph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  delete g;
}

tp_status tp_get_stats(const tp_model* m, tp_stats_t* out) {
  if (!m || !out) return TP_ERR_ARG;
  *out = m->stats;
  return TP_OK;
}

void tp_reset_stats(tp_model* m) {
  if (m) memset(&m->stats, 0, sizeof(m->stats));
}

tp_status tp_selftest_wait_timeout(tp_model* m, int32_t milliseconds, void* stream) {
  if (!m || milliseconds < 1 || milliseconds > 5000) return TP_ERR_ARG;
  int dev = 0, khz = 0;
  TP_CHECK_CUDA(cudaGetDevice(&dev));
  TP_CHECK_CUDA(cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev));
  const long long cycles = (long long)milliseconds * (khz > 0 ? khz : 2000000);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return cuda_status(launch(m, "wait_timeout", st, [&] {
    return launch_wait_timeout(m->status, cycles, st);
  }));
}

tp_status tp_check_device(tp_model* m, void* stream) {
  if (!m) return TP_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TP_CHECK_CUDA(cudaStreamSynchronize(st));
  int v = 0;
  TP_CHECK_CUDA(cudaMemcpy(&v, m->status, sizeof(int), cudaMemcpyDeviceToHost));
  TP_CHECK_CUDA(cudaMemset(m->status, 0, sizeof(int)));
  return static_cast<tp_status>(v);
}

}  // extern "C"

// ============================================================================
// Fused row-parallel reduction whose stream-K partials and tickets live in a
// fixed scratch region the caller already owns (the no-allocation entry point
// in no_alloc.cu passes its static device array).  Layout of the region:
// [tickets: ticket_bytes][partials: partial_bytes].  The tickets are cleared
// on `st` before the launch.
// ============================================================================
namespace tpk {
// Whether one fused row-parallel call of M tokens over out_rows output
// features on a GPU of num_sms SMs fits a fixed scratch of ticket_bytes +
// partial_bytes: the decode orientation only (M <= max_tokens <=
// kSwapMaxTokens), one ticket per 128-row output tile, and two fp32 partial
// tiles of [BN][128] per CTA of the stream-K grid (at most one CTA per SM).
bool noalloc_fits(int M, int out_rows, int num_sms, size_t ticket_bytes, size_t partial_bytes,
                  int max_tokens) {
  if (M < 0 || out_rows < 1 || num_sms < 1 || M > max_tokens || M > kSwapMaxTokens) return false;
  const GemmPlan p = plan_gemm(std::max(M, 1));
  if (!p.swap) return false;
  const size_t tiles = (size_t)cdiv(out_rows, 128);
  const size_t partials = (size_t)num_sms * 2 * p.BN * 128 * sizeof(float);
  return tiles * sizeof(int) <= ticket_bytes && partials <= partial_bytes;
}

tp_status row_reduce_in_scratch(const tp_model* m, int32_t layer, int32_t which, const tp_bf16* x,
                                int64_t x_rank_stride, int64_t ldx, int32_t M,
                                const tp_bf16* residual, tp_bf16* y, void* scratch,
                                size_t ticket_bytes, size_t partial_bytes, int32_t max_tokens,
                                cudaStream_t st) {
  if (!valid_layer(m, layer) || (which != TP_O && which != TP_DOWN) || M < 0 || !scratch)
    return TP_ERR_ARG;
  if (M == 0) return TP_OK;
  const ShardedLinear& W = which == TP_O ? m->layers[layer].o : m->layers[layer].down;
  if (!x || !y || !aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)) ||
      x_rank_stride % 8 || ldx % 8 || ldx < W.cols)
    return TP_ERR_ARG;
  if (!noalloc_fits(M, W.rows, m->num_sms, ticket_bytes, partial_bytes, max_tokens))
    return TP_ERR_WORKSPACE;
  const size_t tiles = (size_t)cdiv(W.rows, 128);
  TP_CHECK_CUDA(cudaMemsetAsync(scratch, 0, tiles * sizeof(int), st));
  WsLayout L;
  memset(&L, 0, sizeof(L));
  L.gemm_tickets = 0;
  L.gemm_partials = ticket_bytes;
  return run_row(m, "gemm_row_noalloc", W, x, x_rank_stride, ldx, M, residual, y, 1, scratch, L,
                 st);
}
}  // namespace tpk
