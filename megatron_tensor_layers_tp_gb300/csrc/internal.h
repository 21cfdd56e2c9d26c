// Declarations shared by the translation units of the library: kernel
// argument blocks and host-side launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tpk {

// Decode orientation (tokens on the MMA N side) for at most this many tokens;
// the GEMM keeps their positions and sequences in shared memory.
constexpr int kSwapMaxTokens = 64;

enum Epi : int {
  EPI_PLAIN = 0,    // column-parallel output, standard per-rank order
  EPI_QKV = 1,      // RoPE on q,k; q -> q buffer, k,v -> rank cache
  EPI_SILU = 2,     // SiLU(gate) * up
  EPI_RESID = 3,    // fused row-parallel: y = residual + sum of rank partials
  EPI_PARTIAL = 4,  // unfused row-parallel: fp32 partial of each rank
  EPI_LOGITS = 5,   // LM head: logits placed in the rank's vocab slot
  EPI_RESID_SQ = 6, // EPI_RESID that also leaves the next RMSNorm's partial
                    // sums of squares (EpiArgs::sq_out; both orientations)
  EPI_QKV_PIECES = 7,  // qkv in the decode orientation, stream-K: every CTA only
                       // stores its fp32 pieces; the decode attention kernel sums
                       // them and finishes the qkv epilogue (norm, bias, RoPE, cache)
};

// Unsigned division by an invariant divisor d (1 <= d < 2^31) as a multiply-
// high, a subtract and two shifts: the round-up method of Granlund and
// Montgomery, "Division by invariant integers using multiplication" (1994),
// in the form that is exact for every 32-bit dividend.  With l = ceil(log2 d),
// m = floor(2^32 (2^l - d) / d) + 1; then n / d = (((n - q) >> s1) + q) >> s2
// with q = mulhi(m, n), s1 = min(l, 1), s2 = max(l - 1, 0).
struct FastDiv {
  uint32_t m, s1, s2;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  FastDiv f;
  f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l > 0 ? l - 1 : 0;
  return f;
}
__host__ __device__ inline uint32_t fast_div(uint32_t n, const FastDiv& f) {
#ifdef __CUDA_ARCH__
  const uint32_t q = __umulhi(f.m, n);
#else
  const uint32_t q = static_cast<uint32_t>((static_cast<uint64_t>(f.m) * n) >> 32);
#endif
  return (((n - q) >> f.s1) + q) >> f.s2;
}

struct EpiArgs {
  int M;                    // tokens
  void* out;                // bf16 (or fp32 for EPI_PARTIAL)
  int64_t ld_out;           // row stride of out (elements)
  int64_t out_group_stride; // elements between ranks' outputs (PLAIN, PARTIAL)
  const uint16_t* residual; // EPI_RESID, may be null
  int64_t ld_res;
  int which;                // EPI_PLAIN: 0 = qkv layout, 1 = gate_up layout
  int head_dim;
  int q_heads_per_rank;
  int kv_heads_per_rank;
  int kv_replicas;
  int inter_per_rank;
  // EPI_QKV
  uint16_t* k_cache;
  uint16_t* v_cache;
  int64_t kv_copy_stride;   // elements per rank copy
  int n_seqs;
  int l_max;
  const int32_t* positions;
  const int32_t* token_seq;
  const float2* rope;       // [max_positions][head_dim/2] (cos, sin)
  // EPI_LOGITS
  int vocab;
  int vocab_per_rank;
  // optional bias over the output features (PLAIN, QKV, SILU, RESID): the
  // value of output row f of rank g is bias[g * bias_group_stride + f]
  const uint16_t* bias;
  int64_t bias_group_stride;
  // RMSNorm folded into the GEMM (QKV and SILU; norm_mode 1 only in the
  // decode orientation): the
  // weights already carry the norm weight w (W[n][k] * w[k], rounded to bf16
  // at load) and the GEMM reads the raw hidden state, so every output of
  // token m is scaled by 1 / sqrt(ss_m / norm_width + norm_eps) before bias,
  // RoPE and SiLU, where ss_m = sum_k h[m][k]^2 comes from
  //   norm_mode 1: the rows of norm_src (read by the epilogue warps),
  //   norm_mode 2: sum over i < norm_slots of norm_partials[m * norm_slots + i],
  //                left by the kernel that wrote h (sq_out below);
  //   norm_mode 0: no scaling.
  int norm_mode;
  const uint16_t* norm_src;
  int64_t norm_ld;          // row stride of norm_src (elements)
  int norm_width;           // k extent (H), a multiple of 8
  float norm_eps;
  const float* norm_partials;  // 16-byte aligned
  int norm_slots;               // a multiple of 4
  // EPI_RESID_SQ: sums of squares of the stored (bf16) outputs for the next
  // RMSNorm, token-major with sq_ld slots per token.  Decode orientation: the
  // warp holding output features [32 i, 32 i + 32) for token m writes slot i.
  // Prefill orientation: the epilogue thread of token m writes, for output
  // tile ib, slot 2 ib + (its half of the tile's 16-column units; slot
  // 2 ib + 1 is zero when one thread covers the whole tile), so
  // sq_ld = 2 x the tiles across the output features.
  float* sq_out;
  int sq_ld;
};

struct GemmArgs {
  CUtensorMap tmA;          // (K, rows, slices), box (64, 128, 1)
  CUtensorMap tmB;          // (K, rows, slices), box (64, BN, 1)
  int BN;                   // N tile: multiple of 16, <= 256
  int stages;
  int tmem_cols;            // power of two >= 2*BN
  int n_groups;             // output groups (ranks) on the tile axis
  int a_tiles, b_tiles;     // tiles per group along A rows / B rows
  int k_slices;             // rank slices folded into K (fused row-parallel)
  int k_iters_slice;        // 64-wide K steps per slice
  int a_slice_mode;         // 0: slice 0; 1: slice = group; 2: slice = K slice
  int b_slice_mode;
  int a_rows_valid;         // A rows per group that exist
  int b_rows_valid;         // B rows per group that exist
  int a_policy, b_policy;   // L2 policy: 0 normal, 1 evict_first, 2 evict_last
  int a_slice_mid, b_slice_mid;  // 1: tensor map dims are (K, slice, rows)
  int grid;                 // G
  int dp_waves;             // W: tiles [0, W*G) are whole-tile, data-parallel
  int cluster_split;        // s > 1: cluster of s CTAs per tile, K split s ways (DSMEM sum)
  int64_t total_iters;      // (n_tiles - W*G) * k_slices * k_iters_slice (stream-K part)
  int pair;                 // 1: prefill orientation on CTA pairs (gemm_pair_kernel): a_tiles
                            // counts 256-row tiles, tmB has a box of BN/2 rows, grid = 2 x pairs
  int fix32;                // 1: every flat index x grid < 2^31: the index divisions after
                            // the dependency wait are multiply-shifts
  FastDiv div_total, div_sk, div_k;  // by total_iters, the stream-K CTA count, K steps per tile
  FastDiv div_a, div_b;              // by a_tiles, b_tiles
  int sk_ctas;              // CTAs 0..sk_ctas-1 share the stream-K part (0: all G); with
                            // sk_ctas = n_tiles - W*G each of them takes one whole tile
  float* partials;          // [G][2][BN][128]
  int* tickets;             // [n_tiles], zero on entry and exit
  int* status;              // device status word
  EpiArgs e;
};

struct AttnArgs {
  CUtensorMap tmK;            // (d, l_max, copies*n_seqs*kv_r), box (64, 64, 1)
  CUtensorMap tmV;
  const uint16_t* q;          // [M, n_heads*d]
  int64_t ld_q;
  uint16_t* o;                // [M, n_heads*d]
  int64_t ld_o;
  const int32_t* positions;
  const int32_t* seq_start;   // prefill
  int n_seqs, n_heads, n_kv, head_dim, kv_r, group;
  int l_max;                  // cache capacity per sequence
  float scale_log2;           // log2(e) / sqrt(d)
  // decode: even split of (sequence, KV head, key tile) units over the grid
  int tiles_per_bg;
  int64_t total_units;
  int grid;
  // total_units * grid < 2^31: the schedule's divisions by total_units, grid,
  // tiles_per_bg and n_kv are multiply-shifts (else 64-bit divisions)
  int idx32;
  FastDiv div_units, div_grid, div_tb, div_kv;
  int stages;                 // K/V stages in shared memory (even)
  float* partials;            // [grid][2][16][d+2]
  int* tickets;               // [n_seqs*n_kv]
  int* status;
  // decode, qkv reduction deferred to this kernel (the qkv GEMM ran with
  // EPI_QKV_PIECES): each CTA sums the GEMM's fp32 pieces of its sequence's q,
  // k and v rows in K order, scales them by the token's 1/rms, adds the bias,
  // applies RoPE, writes the new K/V cache row and merges the new key into the
  // softmax itself; cached keys at the new position are not read
  int qkv_pieces;
  const float* pc;            // pieces [pc_grid][2][pc_bn][128] fp32 (stream-K slots)
  int64_t pc_total;           // the GEMM's stream-K K steps
  int pc_grid, pc_k, pc_bn;   // its grid, K steps per tile, token tile width
  FastDiv pc_div_total, pc_div_grid, pc_div_q;  // by pc_total, pc_grid, q_per_rank
  int pc_a_tiles;             // 128-row tiles per rank
  int nqkv_r;                 // qkv shard rows per rank
  int q_per_rank, kv_replicas;
  const uint16_t* qkv_bias;   // [ranks][nqkv_r] or null
  const float2* rope;         // [max_positions][d/2]
  uint16_t* k_cache;          // [copies][n_seqs][kv_r][l_max][d]
  uint16_t* v_cache;
  int64_t kv_copy_stride;
  int norm_mode;              // 1/rms of the token as EpiArgs: 0 none, 1 rows, 2 partial sums
  const uint16_t* norm_src;
  int64_t norm_ld;
  int norm_width;
  float norm_eps;
  const float* norm_partials;
  int norm_slots;
};

// Every kernel on the forward path is launched with programmatic stream
// serialisation: it may begin (set-up, weight prefetch) while its predecessor
// on the stream finishes, and waits (griddepcontrol.wait) before touching data
// a predecessor wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kc(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  if (cluster_x > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attr;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args... args) {
  return launch_kc(kernel, grid, block, smem, st, 1, args...);
}

// gemm.cu / gemm_epi*.cu
cudaError_t launch_gemm(bool swap, int epi, const GemmArgs& a, size_t smem, cudaStream_t st);
// co-resident clusters of cluster_x CTAs of the GEMM kernel (pair: the CTA-pair
// kernel, cluster_x = 2) with `smem` bytes each
int gemm_max_clusters(bool swap, bool pair, int epi, int cluster_x, size_t smem);
#define TPK_DECLARE_EPI(E)                                                                   \
  cudaError_t launch_gemm_epi##E(bool swap, const GemmArgs& a, size_t smem, cudaStream_t st); \
  int gemm_max_clusters_epi##E(bool swap, bool pair, int cluster_x, size_t smem);
TPK_DECLARE_EPI(0)
TPK_DECLARE_EPI(1)
TPK_DECLARE_EPI(2)
TPK_DECLARE_EPI(3)
TPK_DECLARE_EPI(4)
TPK_DECLARE_EPI(5)
TPK_DECLARE_EPI(6)
TPK_DECLARE_EPI(7)

// attention.cu
cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t st);
cudaError_t launch_attn_prefill(const AttnArgs& a, int n_qb, cudaStream_t st);
size_t attn_decode_partial_floats(int head_dim);
// the decode kernel's K/V stage count for `rows` query rows per KV head
int attn_decode_stages(int head_dim, int rows);

// small.cu
// sq (may be null): each row's sum of squares at sq[row * 4], zeros at
// sq[row * 4 + 1..3] (the [token][slot] form the GEMMs' folded RMSNorm reads)
cudaError_t launch_embed(const uint16_t* table, int vocab, int vocab_per_rank, int t,
                         const int32_t* ids, int M, int H, uint16_t* h, float* sq, int* status,
                         cudaStream_t st);
// w_loaded: w is a model weight written at load time (read before the
// dependency wait); otherwise it is read after it
cudaError_t launch_rmsnorm(const uint16_t* x, int64_t ldx, const int32_t* rows, const uint16_t* w,
                           int M, int H, float eps, uint16_t* y, int64_t ldy, cudaStream_t st,
                           bool w_loaded);
cudaError_t launch_reduce_ranks(const float* partials, int64_t rank_stride, int t, int M, int H,
                                const uint16_t* bias, const uint16_t* residual, uint16_t* y,
                                cudaStream_t st);
cudaError_t launch_rope_table(float2* table, int max_pos, int head_dim, double theta,
                              cudaStream_t st);
// dst[i][k] = bf16(src[i][k] * w[k]) for n_rows rows of cols elements (RNE;
// the fp32 product of two bf16 values is exact).  Folds an RMSNorm weight into
// the weight rows that consume its output.
cudaError_t launch_fold_cols(uint16_t* dst, const uint16_t* src, const uint16_t* w, int64_t n_rows,
                             int cols, cudaStream_t st);
// bytes (a multiple of 16, 16-byte aligned ends) from src to dst by a kernel;
// to_host: src on the device, dst pinned host memory (its device address);
// else the other way round.  Waits for the preceding kernel first.
cudaError_t launch_host_copy(const void* src, void* dst, size_t bytes, bool to_host,
                             cudaStream_t st);
cudaError_t launch_reblock_k64(uint16_t* dst, const uint16_t* src, int ranks, int rows, int cols,
                               cudaStream_t st);
cudaError_t launch_copy_rows(uint16_t* dst, int64_t dst_ld, const uint16_t* src, int64_t src_ld,
                             const int32_t* row_map, int n_rows, int n_cols, cudaStream_t st);
cudaError_t launch_stage_send(const uint16_t* src, uint16_t* dst, int M, int H, int t,
                              cudaStream_t st);
cudaError_t launch_wait_timeout(int* status, long long limit, cudaStream_t st);

}  // namespace tpk
