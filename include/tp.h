/*
 * tp.h — C ABI of the tensor-parallel (TP) Llama decoder forward, with the t
 * ranks of a TP group emulated as shard buffers on one GPU.
 *
 * What the calls compute follows three pages on Megatron-style tensor
 * parallelism in LLM inference engines:
 *   [P1] "第 9 章 多进程与张量并行" (zero-to-sglang), §3.1 通信, §3.2 切分
 *   [P2] "Tensor Parallelism 执行路径" (sglang-internals), 前向执行的实际流程,
 *        KV Cache 在 TP 下怎样分布
 *   [P3] "张量、流水线与数据并行" (inference/05-parallel/tensor-parallel),
 *        线性层怎么切, 每 token 的通信量（估算）
 *
 * Conventions for every call
 *   - Pointers named in the signatures are DEVICE pointers unless stated
 *     otherwise.  bf16 values travel as raw 16-bit patterns (tp_bf16).
 *   - Matrices are row-major.  Weights use the [out, in] layout.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     is asynchronous on it, except tp_load_shards and tp_check_device, which
 *     synchronise it.  Nothing on the forward path allocates device memory or
 *     synchronises.
 *   - Ownership: the caller owns every activation, id, logits, KV cache and
 *     workspace buffer.  The model (tp_model) owns only the weight shards, a
 *     RoPE table and a small device status word, all freed by tp_free.
 *   - Errors: argument and rule violations are returned before anything is
 *     launched.  Errors found on the device (a token id >= vocab, a pipeline
 *     wait that ran out) set the model's device status word; tp_check_device
 *     reads and clears it.  No call aborts the process or throws.
 *   - Workspace: calls that take (ws, ws_bytes) need at least
 *     tp_workspace_bytes(model, M) bytes, zero-filled before the first use
 *     (tp_workspace_init).  The kernels leave the counters in it at zero when
 *     they finish; after a device error, zero it again.  Calls that use the
 *     same workspace must not overlap on the device.
 */
#ifndef TP_GB300_H
#define TP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t tp_bf16; /* bit pattern of one bfloat16 value */

typedef enum {
  TP_OK = 0,
  TP_ERR_ARG = 1,            /* null pointer, bad index, size out of range */
  TP_ERR_DIVISIBILITY = 2,   /* n_heads % t, intermediate % t, n_heads % n_kv_heads */
  TP_ERR_KV_REPLICA = 3,     /* n_kv >= t with n_kv % t != 0, or n_kv < t with t % n_kv != 0 */
  TP_ERR_TOKEN_RANGE = 4,    /* (device) a token id outside [0, vocab) */
  TP_ERR_OOM = 5,            /* device allocation failed in tp_load_shards */
  TP_ERR_CUDA = 6,           /* a CUDA runtime call failed */
  TP_ERR_DEVICE_TIMEOUT = 7, /* (device) a bounded pipeline wait ran out */
  TP_ERR_UNSUPPORTED = 8,    /* shape outside the kernels' envelope (see tp_config) */
  TP_ERR_WORKSPACE = 9       /* workspace missing or smaller than tp_workspace_bytes */
} tp_status;

/* Model shape.  The caller fills the first block; tp_config validates it and
 * fills the derived block.
 *
 * Rules (P1 §3.2 切分): Q heads split by head, so n_heads % t == 0.  KV heads
 * split n_kv/t per rank when n_kv >= t (n_kv % t == 0); when n_kv < t each KV
 * head is replicated on t/n_kv ranks that share one cache copy
 * (t % n_kv == 0), and rank r reads KV head r / (t/n_kv).  The vocabulary is
 * padded to a multiple of t with zero rows and split evenly.  The
 * intermediate size splits evenly (intermediate % t == 0).
 *
 * DP attention (P3 SGLang 的 DP attention): attn_dp > 1 splits the t ranks
 * into attn_dp attention groups of attn_tp = t / attn_dp ranks.  Each group
 * batches its own sequences (contiguous blocks of the batch) and keeps their
 * KV; the attention block (qkv_proj, attention, o_proj and its reduction) is
 * tensor-parallel over the group's attn_tp ranks, while the MLP stays
 * tensor-parallel over all t ranks, after the groups' hidden rows are
 * gathered.  The head and KV rules above then apply with attn_tp in place of
 * t, and the per-rank head fields below describe the attention ranks.
 * attn_dp = 0 is read as 1 (plain tensor parallelism); t % attn_dp != 0 is
 * TP_ERR_DIVISIBILITY.
 *
 * Kernel envelope (TP_ERR_UNSUPPORTED otherwise): head_dim in {64, 128};
 * hidden, n_heads*head_dim/attn_tp and intermediate/t multiples of 64;
 * 1 <= t <= 8; max_positions >= 1. */
typedef struct {
  int32_t hidden;
  int32_t n_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t intermediate;
  int32_t vocab;
  int32_t n_layers;
  int32_t t;             /* emulated TP ranks */
  float rms_eps;         /* RMSNorm epsilon */
  float rope_theta;      /* RoPE base */
  int32_t max_positions; /* RoPE table length: every position must be < this */
  int32_t attn_dp;       /* attention data-parallel groups (0 or 1: none) */
  int32_t host_io;       /* tp_layer_forward_host transfers: 0 = chosen from the
                            device (kernels over a coherent host link, else the
                            copy engine), 1 = always cudaMemcpyAsync */
  int32_t plain_column_shards; /* 1: keep an unfolded copy of every qkv / gate_up
                            shard for tp_column_linear (see tp_load_shards) */
  int32_t prefill_bn;    /* output-feature tile width of the GEMMs above 64
                            tokens: 0 = chosen per GEMM (the width among 256,
                            224, 192, 160, 128 whose whole-tile waves over the
                            SMs take least time, 256 when that GEMM has fewer
                            tiles than SMs); else one of those five, used by
                            every such GEMM (any other value: TP_ERR_ARG) */
  int32_t prefill_cta_pairs; /* GEMMs above 64 tokens on pairs of SMs
                            (tcgen05 cta_group::2, 256 token rows per tile):
                            0 = when the GEMM has at least one wave of such
                            tiles, 1 = always, 2 = never (single-CTA kernel);
                            any other value: TP_ERR_ARG */
  /* derived, written by tp_config */
  int32_t vocab_padded;
  int32_t vocab_per_rank;
  int32_t q_heads_per_rank;
  int32_t kv_heads_per_rank; /* KV heads in one rank's cache (1 when replicated) */
  int32_t kv_replicas;       /* ranks sharing one KV head (1 when split) */
  int32_t kv_copies;         /* distinct per-rank caches = min(attn_tp, n_kv_heads) */
  int32_t inter_per_rank;
  int32_t attn_tp;           /* attention ranks per DP group = t / attn_dp */
} tp_config_t;

/* Validates the shape and fills the derived fields. */
tp_status tp_config(tp_config_t* c);

/* Unsharded weights of one decoder layer (device pointers, bf16).
 * attn_norm, mlp_norm [H]; wq [n_heads*d, H]; wk, wv [n_kv*d, H];
 * wo [H, n_heads*d]; wg, wu [I, H]; wd [H, I].
 * Optional biases over each projection's output features (NULL = none;
 * Qwen2.5-style models carry bq, bk, bv): bq [n_heads*d]; bk, bv [n_kv*d];
 * bo [H]; bg, bu [I]; bd [H].  A column-parallel bias is cut with its weight
 * rows (P1 §3.2 切分: weights and their biases split along the output
 * dimension), so rank r adds the entries of its own rows; the bias of a
 * row-parallel output (bo, bd) belongs to the whole reduced output and is
 * added once, after the reduction, before the residual. */
typedef struct {
  const tp_bf16 *attn_norm, *wq, *wk, *wv, *wo, *mlp_norm, *wg, *wu, *wd;
  const tp_bf16 *bq, *bk, *bv, *bo, *bg, *bu, *bd;
} tp_layer_weights_t;

/* embed, lm_head [vocab, H]; final_norm [H]: may all be NULL for a model used
 * layer by layer.  `layers` is a HOST array of n_layers entries. */
typedef struct {
  const tp_bf16* embed;
  const tp_bf16* final_norm;
  const tp_bf16* lm_head;
  const tp_layer_weights_t* layers;
} tp_weights_t;

typedef struct tp_model tp_model; /* opaque: owns the shard buffers */

/* Builds the t per-rank shards (P1 §3.2 切分; P3 线性层怎么切) on the device of
 * the current CUDA context and returns the model.  The unsharded weights are
 * only read; the caller may free them afterwards.  Synchronises `stream`.
 *   qkv shard r    : rows of rank r's Q heads, then of its KV heads (copies
 *                    when replicated) — column-parallel
 *   gate_up shard r: rows [r I/t, (r+1) I/t) of the gate and of the up weight
 *                    — column-parallel
 *   o / down shard r: columns [r K/t, (r+1) K/t) of wo / wd — row-parallel
 *   embed / lm_head shard r: vocab rows [r Vp/t, (r+1) Vp/t), zero padded
 * Within a shard, rows are stored in the order the fused epilogues want (the
 * two halves of each RoPE pair, and each gate row with its up row, sit next
 * to each other); every output of the API is in the standard order.
 * The decoder layer reads qkv and gate_up shards with the preceding RMSNorm's
 * weight folded into their columns (W[n][k] * w[k], rounded to bf16):
 * (x / rms(x) * w) . W[n] equals (x . (W[n] * w)) / rms(x).  tp_column_linear
 * computes with the unfolded weights.  When a layer's norm weight is exactly
 * 1 everywhere the folded and unfolded shards are the same bytes and one
 * buffer serves both; otherwise the unfolded copy (2 bytes per qkv and
 * gate_up weight, 285 MB per Llama-3.1-8B layer) is kept only when
 * cfg->plain_column_shards = 1, and tp_column_linear on a layer without it
 * returns TP_ERR_UNSUPPORTED. */
tp_status tp_load_shards(const tp_config_t* cfg, const tp_weights_t* w, void* stream,
                         tp_model** out);
void tp_free(tp_model* m);
tp_status tp_get_config(const tp_model* m, tp_config_t* out);
/* Device memory the model owns (every shard, the RoPE table, the status
 * word), in bytes, in *bytes. */
tp_status tp_model_bytes(const tp_model* m, int64_t* bytes);

/* Workspace bytes needed by any call on up to max_tokens rows. */
size_t tp_workspace_bytes(const tp_model* m, int32_t max_tokens);
/* Zero-fills a workspace (async on stream). */
tp_status tp_workspace_init(void* ws, size_t ws_bytes, void* stream);

enum { TP_QKV = 0, TP_GATE_UP = 1, TP_O = 2, TP_DOWN = 3 };

/* Column-parallel linear, all t ranks in one launch (P3 线性层怎么切: the
 * weight A is split along the output dimension, rank i computes
 * Y_i = X A_i from the full replicated X, and the outputs stay sharded —
 * no communication, gather_output = false).
 *   which : TP_QKV or TP_GATE_UP
 *   x     : [M, H] bf16
 *   y     : rank r's output at y + r*y_rank_stride (elements), [M, N_r]
 *           row-major with N_r = (q_heads_per_rank + 2 kv_heads_per_rank)*d
 *           for TP_QKV (its Q heads, then K heads, then V heads) and
 *           N_r = 2 I/t for TP_GATE_UP (gate slice, then up slice).
 *           y_rank_stride >= M*N_r.
 * Plain GEMM output plus the rank's slice of the layer's bias when the model
 * has one (bq/bk/bv or bg/bu): no RoPE, no activation.  TP_ERR_UNSUPPORTED
 * when the model keeps no unfolded copy of this layer's shards (see
 * tp_load_shards). */
tp_status tp_column_linear(const tp_model* m, int32_t layer, int32_t which, const tp_bf16* x,
                           int32_t M, tp_bf16* y, int64_t y_rank_stride, void* ws,
                           size_t ws_bytes, void* stream);

/* Row-parallel linear plus the all-reduce of its t partial sums
 * (P1 §3.1: Y = Y_0 + Y_1 + ... + Y_{t-1}; P3 线性层怎么切).
 *   which    : TP_O or TP_DOWN
 *   x        : rank r's input shard at x + r*x_rank_stride, [M, K_r] with row
 *              stride ldx (K_r = n_heads*d/t for TP_O, I/t for TP_DOWN)
 *   residual : [M, H] or NULL; added once, in fp32, before the rounding
 *   bias     : the layer's bo / bd, when the model has one, is added once to
 *              the reduced sum (not per rank), in fp32, before the residual
 *   y        : [M, H] bf16; may alias `residual`
 *   fused    : 1 = one kernel; the t partials are accumulated in fp32 in
 *              rank order 0..t-1 and rounded once to bf16 in its epilogue.
 *              0 = each rank's fp32 partial is written to the workspace, then
 *              a separate kernel sums them in rank order (same rounding).
 * The reduction order is fixed, so results are deterministic. */
tp_status tp_row_linear_reduce(const tp_model* m, int32_t layer, int32_t which,
                               const tp_bf16* x, int64_t x_rank_stride, int64_t ldx, int32_t M,
                               const tp_bf16* residual, tp_bf16* y, int32_t fused, void* ws,
                               size_t ws_bytes, void* stream);

/* Vocab-parallel embedding (P1 §3.2 Vocab Parallel; P3 词嵌入): rank r looks
 * up only ids in [r Vp/t, (r+1) Vp/t) and contributes -0.0 elsewhere; the t
 * contributions are summed in rank order, which reproduces E[id] bit for bit.
 *   ids : [M] int32;  h : [M, H] bf16.
 * An id outside [0, vocab) writes a zero row and sets TP_ERR_TOKEN_RANGE in
 * the device status word. */
tp_status tp_vocab_embed(const tp_model* m, const int32_t* ids, int32_t M, tp_bf16* h,
                         void* stream);

/* Vocab-parallel LM head with the logits all-gather (P1 §3.1 All-Gather:
 * Y = cat(Y_0, ..., Y_{t-1}); P3 输出层).  Rank r computes logits of its
 * Vp/t vocab rows and writes them straight into columns [r Vp/t, (r+1) Vp/t)
 * of the output; columns >= vocab (padding) are not written.
 *   x      : [S, H] bf16 (already normalised)
 *   logits : [S, vocab] bf16 with row stride ld_logits >= vocab */
tp_status tp_lm_head_gather(const tp_model* m, const tp_bf16* x, int32_t S, tp_bf16* logits,
                            int64_t ld_logits, void* ws, size_t ws_bytes, void* stream);

enum { TP_DECODE = 0, TP_PREFILL = 1 };

/* One forward step's batch.
 * Tokens are grouped by sequence: sequence b owns tokens
 * [seq_start[b], seq_start[b+1]).  Token i sits at position positions[i] of
 * its sequence and attends to cache positions 0..positions[i] of that
 * sequence (causal).  In DECODE mode token b is the single token of sequence
 * b (seq_start may be NULL).
 * KV cache (per layer, caller-owned, bf16): rank copy c of sequence b, KV head
 * g (local to the copy), position p, element e lives at
 *   base[(((c*n_seqs + b)*kv_heads_per_rank + g)*l_max + p)*head_dim + e]
 * Replica ranks (n_kv < t) share copy c = r / kv_replicas.  The layer writes
 * each token's K and V at its position before attention reads them; the rows
 * below a token's position must already hold their values when the call is
 * enqueued (written earlier in stream order), since decode attention may start
 * reading them while the kernels before it are still running. */
typedef struct {
  int32_t mode;                /* TP_DECODE or TP_PREFILL */
  int32_t n_seqs;
  int32_t n_tokens;            /* M */
  int32_t max_q_per_seq;       /* host: max tokens of one sequence in this batch */
  int32_t max_ctx;             /* host: max over tokens of positions[i] + 1 */
  int32_t l_max;               /* cache capacity per sequence (positions < l_max) */
  const int32_t* seq_start;    /* device [n_seqs + 1] (PREFILL) */
  const int32_t* positions;    /* device [n_tokens] */
  const int32_t* token_seq;    /* device [n_tokens]: sequence of each token */
  tp_bf16* const* k_cache;     /* HOST array [n_layers] of device base pointers */
  tp_bf16* const* v_cache;     /* HOST array [n_layers] of device base pointers */
  const int32_t* sample_rows;  /* device [n_samples]: token rows that produce logits */
  int32_t n_samples;
} tp_batch_t;

/* One decoder layer, all t ranks (P3 线性层怎么切 flowchart; P2 前向执行的实际流程):
 *   u = RMSNorm(h)                        replicated
 *   q,k,v = column-parallel qkv_proj(u), RoPE on q and k, k/v -> rank caches
 *   o = per-rank GQA attention over the rank's own heads and cache
 *   h = h + all_reduce(row-parallel o_proj(o))           reduction ①
 *   u = RMSNorm(h)
 *   a = SiLU(gate) * up from column-parallel gate_up_proj(u)
 *   h = h + all_reduce(row-parallel down_proj(a))        reduction ②
 * h_inout [n_tokens, H] bf16 is read and overwritten.  fused selects the
 * row-parallel reduction variant (see tp_row_linear_reduce).
 * Each RMSNorm's weight is folded into the GEMM after it (tp_load_shards):
 * that GEMM reads h and scales token m's outputs by 1/sqrt(mean(h_m^2) +
 * eps) in fp32.  Up to 32 tokens it computes mean(h_m^2) from h's rows (five
 * kernels per layer).  Above that, with the fused reduction, the second norm
 * takes partial sums of squares that o_proj leaves, and in tp_forward /
 * tp_stage_forward so does every later layer's first norm (from down_proj)
 * and the first layer's (from the embedding); the first norm of a
 * tp_layer_forward call, and every norm with the unfused reduction, runs as a
 * kernel.  The sums are added in a fixed order: the result is deterministic. */
tp_status tp_layer_forward(const tp_model* m, int32_t layer, const tp_batch_t* b,
                           tp_bf16* h_inout, int32_t fused, void* ws, size_t ws_bytes,
                           void* stream);

/* tp_layer_forward on host-resident hidden rows (no counterpart on the
 * pages; the call a host program makes when its hidden states live in host
 * memory).  h_in_host [n_tokens, H] bf16 is brought to the caller's device
 * buffer h_dev [n_tokens, H] (overwritten), the layer runs there, and the
 * result is written to h_out_host [n_tokens, H].  Both host buffers must be
 * pinned (cudaHostAlloc / cudaHostRegister; otherwise TP_ERR_ARG) and 16-byte
 * aligned; they may be the same buffer, also across consecutive calls.  On a
 * GPU that reaches host memory coherently (NVLink-C2C: GB300 with its Grace
 * host) the two transfers are kernels that read and write the pinned memory
 * directly and join the layer's chain of dependent launches; elsewhere, or
 * when the model was configured with host_io = 1, they are cudaMemcpyAsync on
 * `stream`.  The GPU counts as coherent with its host when it reports both
 * native atomics over the host link and access to pageable host memory
 * through the host's page tables (true of NVLink-C2C, false of PCIe).
 * Asynchronous: h_out_host is valid once `stream` has reached this point. */
tp_status tp_layer_forward_host(const tp_model* m, int32_t layer, const tp_batch_t* b,
                                const tp_bf16* h_in_host, tp_bf16* h_out_host, tp_bf16* h_dev,
                                int32_t fused, void* ws, size_t ws_bytes, void* stream);

/* Full forward: vocab-parallel embedding of ids [n_tokens] into h, every
 * layer, final RMSNorm of the sampled rows, vocab-parallel LM head gathered
 * into logits [n_samples, vocab] (row stride ld_logits).
 *   h : [n_tokens, H] bf16 scratch that ends holding the last hidden state. */
tp_status tp_forward(const tp_model* m, const int32_t* ids, const tp_batch_t* b, tp_bf16* h,
                     tp_bf16* logits, int64_t ld_logits, int32_t fused, void* ws,
                     size_t ws_bytes, void* stream);

/* One pipeline stage (P3 流水线并行: the layers are cut into consecutive groups,
 * each stage builds only its own layers, and a non-final stage hands its
 * running hidden state to the next).  Runs layers
 * [first_layer, first_layer + n_layers) on h in place.
 *   ids    : non-NULL on the first stage only: h = vocab-parallel embedding of
 *            ids [n_tokens] before the layers (first_layer must then be 0).
 *   logits : non-NULL on the last stage only: final RMSNorm of the sampled rows
 *            and the vocab-parallel LM head with the logits gather, as
 *            tp_forward (first_layer + n_layers must then be n_layers of the
 *            model; ld_logits >= vocab).
 * Stages covering layers 0..n_layers-1 in order, joined by tp_stage_send,
 * launch the same kernels in the same order as tp_forward and return its
 * logits bit for bit.  Errors: TP_ERR_ARG for a layer range outside the model
 * or the conditions above; otherwise as tp_forward. */
tp_status tp_stage_forward(const tp_model* m, int32_t first_layer, int32_t n_layers,
                           const int32_t* ids, const tp_batch_t* b, tp_bf16* h,
                           tp_bf16* logits, int64_t ld_logits, int32_t fused, void* ws,
                           size_t ws_bytes, void* stream);

/* Stage-boundary hand-off (P3 流水线并行).  Copies the running hidden state
 * [M, H] bf16 from one stage's buffer (src) to the next stage's (dst).  With
 * tensor parallelism inside each stage, rank r sends only its slice of
 * columns [r H/t, (r+1) H/t) and the receiving stage all-gathers the slices
 * inside its TP group; here one kernel moves the t slices and they land side
 * by side in dst, which is that all-gather's result.
 * Counters: stage_sends += 1, stage_send_bytes += M*H*2 (M*H*2/t per rank).
 * The pages estimate 2 x H x 2 bytes per token because their engines hand
 * over the hidden state and the residual as two tensors; this library adds
 * the residual inside the row-parallel epilogues, so one tensor of H x 2
 * bytes per token carries both.
 * Requires (H / t) % 8 == 0, 16-byte aligned src and dst that do not overlap;
 * TP_ERR_ARG otherwise. */
tp_status tp_stage_send(const tp_model* m, const tp_bf16* src, tp_bf16* dst, int32_t M,
                        void* stream);

/* CUDA-graph capture of one decode step (P3 每 token 的通信量 读法: a fixed cost
 * per synchronisation that "custom all-reduce and CUDA graph" address; P1
 * names CUDA graph among the engines' decode optimisations).
 * tp_graph_capture_forward / tp_graph_capture_layer record the kernels that
 * tp_forward / tp_layer_forward would launch with these arguments, on
 * `stream` (a stream the caller created, not the legacy default stream), into
 * an executable graph; nothing runs during the capture.  tp_graph_launch
 * replays it on any stream.  A replay reads the current contents of every
 * buffer the captured call named (ids, positions, caches, h, workspace), so
 * the caller refreshes their contents between replays but keeps their
 * addresses, the batch shape and the workspace alive and unshared while the
 * graph exists.  Each replay adds the captured call's counters to the model's
 * (tp_get_stats).  Errors: TP_ERR_ARG for a NULL stream or output pointer or
 * while tp_profile is enabled; the captured call's own argument errors;
 * TP_ERR_CUDA if capture or instantiation fails (the stream is left out of
 * capture mode). */
typedef struct tp_graph tp_graph;
tp_status tp_graph_capture_forward(const tp_model* m, const int32_t* ids, const tp_batch_t* b,
                                   tp_bf16* h, tp_bf16* logits, int64_t ld_logits,
                                   int32_t fused, void* ws, size_t ws_bytes, void* stream,
                                   tp_graph** out);
tp_status tp_graph_capture_layer(const tp_model* m, int32_t layer, const tp_batch_t* b,
                                 tp_bf16* h_inout, int32_t fused, void* ws, size_t ws_bytes,
                                 void* stream, tp_graph** out);
tp_status tp_graph_launch(tp_graph* g, void* stream);
void tp_graph_free(tp_graph* g);

/* tp_row_linear_reduce with fused = 1, for callers that cannot allocate
 * device memory — for example a plug-in that its host framework hands only
 * input and output tensors, or a latency-critical loop that cannot afford
 * cudaMalloc's implicit device-wide synchronisation.  The pages have no
 * counterpart: this is a packaging of the same computation, which it returns
 * bit for bit as tp_row_linear_reduce (fused) does.
 *   Arguments: as tp_row_linear_reduce, minus the workspace.
 *   Scratch: the GEMM's split partials and arrival tickets live in one
 *     library-owned array in device memory of 10 MiB + 16 KiB (allocated when
 *     the library is loaded, on every GPU that loads it, held until the
 *     process exits).  It limits M to 64 tokens and the GPU to 160 SMs; larger
 *     requests return TP_ERR_WORKSPACE.  The tickets are cleared on `stream`
 *     before each launch.
 *   Set-up: the first call on each device resolves the array's device address
 *     (cudaGetSymbolAddress) with that device current and keeps it for the
 *     life of the process; make that first call before any stream capture,
 *     and do not call the entry point on a device after cudaDeviceReset
 *     (the address belonged to the destroyed context).
 *   Concurrency: every call shares the one array, so calls that may overlap
 *     on the GPU (different streams, or different host threads) race; order
 *     them on one stream.
 *   Allocation: the call makes no cudaMalloc/cudaFree and calls no allocating
 *     library routine. */
tp_status tp_row_linear_reduce_noalloc(const tp_model* m, int32_t layer, int32_t which,
                                       const tp_bf16* x, int64_t x_rank_stride, int64_t ldx,
                                       int32_t M, const tp_bf16* residual, tp_bf16* y,
                                       void* stream);

/* Whether tp_row_linear_reduce_noalloc's fixed scratch can hold a call of M
 * tokens with `hidden` output features on a GPU with num_sms SMs (1) or the
 * call would return TP_ERR_WORKSPACE (0).  Pure host arithmetic: no CUDA
 * call, usable without a GPU. */
int32_t tp_row_linear_reduce_noalloc_fits(int32_t M, int32_t hidden, int32_t num_sms);

/* Replicated RMSNorm (P1 §3.2: small layers stay whole on every rank):
 * y = x / sqrt(mean(x^2) + eps) * w, fp32 arithmetic, bf16 in and out.
 *   x, y : [M, H] (may alias); w : [H] — any device vector. */
tp_status tp_rmsnorm(const tp_model* m, const tp_bf16* x, const tp_bf16* w, int32_t M,
                     tp_bf16* y, void* stream);

/* Counters of the emulated collectives, accumulated by the host over every
 * launch since the model was created (or tp_reset_stats).  The payload is the
 * bf16 result each all-reduce delivers (M*H*2 bytes) and, for the gather, the
 * bytes of the concatenated logits each rank receives from the others
 * ((t-1)/t * vocab * 2 bytes per sampled row) (P3 每 token 的通信量). */
typedef struct {
  int64_t allreduces;          /* row-parallel reductions + embedding reductions */
  int64_t allreduce_payload_bytes;
  int64_t allgathers;          /* logits gathers */
  int64_t allgather_recv_bytes_per_rank;
  int64_t kernel_launches;     /* kernels launched by the library */
  int64_t stage_sends;         /* pipeline-stage boundaries crossed (tp_stage_send) */
  int64_t stage_send_bytes;    /* bytes handed across them, all ranks together */
  int64_t dp_gathers;          /* DP attention: token gathers before the MLP (1 per layer) */
  int64_t dp_gather_recv_bytes_per_rank; /* (attn_dp-1)/attn_dp * M*H*2 per gather */
} tp_stats_t;

tp_status tp_get_stats(const tp_model* m, tp_stats_t* out);
void tp_reset_stats(tp_model* m);

/* Per-kernel timing.  While enabled, every launch the library makes is
 * bracketed by two CUDA events recorded on the launch stream (at most 16384
 * launches are recorded between two reads).  tp_profile_read synchronises
 * `stream`, sums the elapsed times per kernel name into `out` (up to `max`
 * entries, count in *n) and clears the records. */
typedef struct {
  char name[24];
  int64_t launches;
  double total_ms;
} tp_kernel_time_t;

tp_status tp_profile(tp_model* m, int32_t enable);
tp_status tp_profile_read(tp_model* m, void* stream, tp_kernel_time_t* out, int32_t max,
                          int32_t* n);

/* Synchronises `stream`, returns the device status word (TP_OK,
 * TP_ERR_TOKEN_RANGE or TP_ERR_DEVICE_TIMEOUT) and clears it. */
tp_status tp_check_device(tp_model* m, void* stream);

/* Failure-detection self-test (no counterpart on the pages): launches one
 * warp that waits on an mbarrier phase nothing ever completes, through the
 * same bounded wait every kernel of the library uses, with its limit set to
 * about `milliseconds` (1..5000) of SM clock.  The wait gives up, records
 * TP_ERR_DEVICE_TIMEOUT in the model's status word and the kernel returns;
 * nothing faults and the context stays usable.  tp_check_device reports and
 * clears the status. */
tp_status tp_selftest_wait_timeout(tp_model* m, int32_t milliseconds, void* stream);

const char* tp_strerror(tp_status s);

#ifdef __cplusplus
}
#endif
#endif /* TP_GB300_H */
