"""CPU oracle for the tensor-parallel Llama decoder forward.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
baseline leg of the benchmark may import this module.  The product path never
calls it and shares no code with it.

Plain, slow, obviously-correct float64 numpy.  Two parts:

1. The *unsharded* decoder math (embedding, RMSNorm, Y = X W^T, RoPE, GQA
   softmax attention, SiLU gate, LM head).  Tensor parallelism is an exact
   re-association of this math, so this is the definition the sharded path
   must reproduce ("第 9 章 多进程与张量并行", §3 通信与切分: the local results
   must reconstruct the original model's computation).
2. A plain *sharded emulation* that follows the pages step by step: column
   shards computed per rank without communication, row shards producing
   partials that an all-reduce sums, vocab shards with a masked lookup plus
   sum, and LM-head shards whose logits an all-gather concatenates
   ("张量、流水线与数据并行", §线性层怎么切; "第 9 章", §3.1 and §3.2).

Storage rounding: values that the CUDA path stores as bf16 are rounded here
too, by ``round_bf16`` (round to nearest, ties to even, straight from float64),
at the same points: after each norm, q/k/v after RoPE, the attention output,
each residual sum (rounded once after the reduction), SiLU(gate)*up and the
logits.  Every function takes ``rb`` so a test can switch rounding off and
check exact re-association.

Readings where the pages are silent (each listed in the design notes):
pre-norm residual blocks with a final RMSNorm; rotate-half RoPE with
inv_freq_j = theta^(-2j/d); Q head j reads KV head j // (n_h / n_kv); rank r
owns Q heads [r n_h/t, (r+1) n_h/t); when n_kv < t rank r reads KV head
r // (t / n_kv) and the replica ranks share one cache copy; vocab padded to
ceil(V/t)*t with zero rows.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable, List, Optional, Sequence

import numpy as np

Array = np.ndarray


# ---------------------------------------------------------------------------
# bf16 rounding (the oracle's own; float64 -> nearest bf16, ties to even)
# ---------------------------------------------------------------------------
def round_bf16(x) -> Array:
    """Round float64 values to the nearest bf16 value (ties to even).

    bf16 keeps 8 significant bits and the float32 exponent range; below
    2^-126 the spacing is fixed at 2^-133 (subnormals).  Values whose rounding
    reaches 2^128 become infinities.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                      # |x| in [2^(e-1), 2^e)
    q = np.maximum(e - 8, -133)             # spacing exponent of 8-bit significands
    r = np.rint(np.ldexp(x, -q))            # exact scaling, then ties-to-even
    y = np.ldexp(r, q)
    y = np.where(np.abs(y) >= 2.0 ** 128, np.copysign(np.inf, x), y)
    return y


def no_round(x) -> Array:
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# configuration rules ("第 9 章 多进程与张量并行", §3.2 切分)
# ---------------------------------------------------------------------------
class RuleError(ValueError):
    pass


@dataclass(frozen=True)
class Plan:
    t: int
    q_heads_per_rank: int
    kv_heads_per_rank: int     # KV heads in one rank's cache (1 when replicated)
    kv_replicas: int           # ranks that share one KV head (1 when split)
    kv_copies: int             # distinct per-rank caches: min(t, n_kv)
    vocab_padded: int
    vocab_per_rank: int
    inter_per_rank: int


def plan(n_heads: int, n_kv_heads: int, intermediate: int, vocab: int, t: int) -> Plan:
    """Shard plan for t ranks.

    Q heads split by head: n_heads % t == 0.  KV heads: split evenly when
    n_kv >= t (n_kv % t == 0), otherwise each KV head is replicated on
    t / n_kv ranks that share one copy (t % n_kv == 0).  The intermediate
    dimension splits evenly (I % t == 0).  The vocabulary is padded up to a
    multiple of t and split evenly.
    """
    if t < 1 or n_heads < 1 or n_kv_heads < 1:
        raise RuleError("t, n_heads and n_kv_heads must be positive")
    if n_heads % n_kv_heads:
        raise RuleError("n_heads must be a multiple of n_kv_heads (GQA groups)")
    if n_heads % t:
        raise RuleError("n_heads % t != 0")
    if intermediate % t:
        raise RuleError("intermediate % t != 0")
    if n_kv_heads >= t:
        if n_kv_heads % t:
            raise RuleError("n_kv_heads >= t but n_kv_heads % t != 0")
        kv_r, reps = n_kv_heads // t, 1
    else:
        if t % n_kv_heads:
            raise RuleError("n_kv_heads < t but t % n_kv_heads != 0")
        kv_r, reps = 1, t // n_kv_heads
    vp = -(-vocab // t) * t
    return Plan(t, n_heads // t, kv_r, reps, min(t, n_kv_heads), vp, vp // t, intermediate // t)


def kv_heads_of_rank(p: Plan, n_kv_heads: int, r: int) -> List[int]:
    if p.kv_replicas == 1:
        return list(range(r * p.kv_heads_per_rank, (r + 1) * p.kv_heads_per_rank))
    return [r // p.kv_replicas]


def kv_copy_of_rank(p: Plan, r: int) -> int:
    return r // p.kv_replicas


def q_heads_of_rank(p: Plan, r: int) -> List[int]:
    return list(range(r * p.q_heads_per_rank, (r + 1) * p.q_heads_per_rank))


# ---------------------------------------------------------------------------
# communication counts ("张量、流水线与数据并行", §每 token 的通信量（估算）)
# ---------------------------------------------------------------------------
def allreduces_per_forward(n_layers: int) -> int:
    """Two row-parallel all-reduces per layer plus one for the embedding."""
    return 2 * n_layers + 1


def allreduce_payload_bytes_per_token(hidden: int, elem_bytes: int = 2) -> int:
    return hidden * elem_bytes


def ring_bytes_sent_per_rank(payload: int, t: int) -> float:
    return 2.0 * (t - 1) / t * payload


def logits_gather_received_per_rank(vocab: int, t: int, elem_bytes: int = 2) -> float:
    return (t - 1) / t * vocab * elem_bytes


def kv_bytes_per_token_per_rank(n_layers: int, n_kv_heads: int, head_dim: int, t: int,
                                elem_bytes: int = 2) -> int:
    kv_r = n_kv_heads // t if n_kv_heads >= t else 1
    return n_layers * kv_r * head_dim * 2 * elem_bytes


# ---------------------------------------------------------------------------
# unsharded layer math
# ---------------------------------------------------------------------------
def linear(x: Array, w: Array, b: Optional[Array] = None) -> Array:
    """Y = X W^T (+ b) for a weight stored [out, in] (the pages' Y = XW) and
    an optional bias over the output features."""
    y = x @ w.T
    return y if b is None else y + b


def rmsnorm(x: Array, w: Array, eps: float) -> Array:
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * w


def rope_inv_freq(head_dim: int, theta: float) -> Array:
    j = np.arange(head_dim // 2, dtype=np.float64)
    return theta ** (-(2.0 * j) / head_dim)


def rope(x: Array, pos: Array, theta: float) -> Array:
    """Rotate-half RoPE.  x: [T, n, d]; pos: [T].  Pair (j, j + d/2) turns by
    pos * theta^(-2j/d)."""
    d = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[:, None] * rope_inv_freq(d, theta)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: Array) -> Array:
    return x / (1.0 + np.exp(-x))


def softmax(s: Array) -> Array:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def attend(q: Array, k: Array, v: Array) -> Array:
    """One head: q [d]; k, v [S, d] (the visible positions) -> [d]."""
    s = (k @ q) / np.sqrt(q.shape[-1])
    return softmax(s) @ v


def gqa_attend_token(q: Array, kc: Array, vc: Array, pos: int) -> Array:
    """All heads of one token: q [n_h, d]; kc, vc [n_kv, L_max, d] of its
    sequence; positions 0..pos are visible.  Q head j reads KV head
    j // (n_h / n_kv)."""
    nh, nkv = q.shape[0], kc.shape[0]
    group = nh // nkv
    return np.stack([attend(q[j], kc[j // group, : pos + 1], vc[j // group, : pos + 1])
                     for j in range(nh)])


# ---------------------------------------------------------------------------
# batch description
# ---------------------------------------------------------------------------
@dataclass
class Batch:
    """Token t belongs to sequence seq[t] at position pos[t]; it sees cache
    positions 0..pos[t] of its own sequence."""
    seq: Array
    pos: Array

    @staticmethod
    def decode(n_seqs: int, ctx: int) -> "Batch":
        return Batch(np.arange(n_seqs), np.full(n_seqs, ctx - 1))

    @staticmethod
    def prefill(n_seqs: int, seq_len: int) -> "Batch":
        return Batch(np.repeat(np.arange(n_seqs), seq_len), np.tile(np.arange(seq_len), n_seqs))

    def sample_rows(self) -> Array:
        """Rows whose logits are computed: the last token of each sequence."""
        last = {}
        for i, b in enumerate(self.seq):
            last[int(b)] = i
        return np.array([last[b] for b in sorted(last)], dtype=np.int64)


@dataclass
class LayerWeights:
    attn_norm: Array
    wq: Array
    wk: Array
    wv: Array
    wo: Array
    mlp_norm: Array
    wg: Array
    wu: Array
    wd: Array
    # optional biases over each projection's output features (Qwen2.5-style
    # models carry bq, bk, bv); None = no bias
    bq: Optional[Array] = None
    bk: Optional[Array] = None
    bv: Optional[Array] = None
    bo: Optional[Array] = None
    bg: Optional[Array] = None
    bu: Optional[Array] = None
    bd: Optional[Array] = None


@dataclass
class Dims:
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0


# ---------------------------------------------------------------------------
# unsharded decoder layer / forward
# ---------------------------------------------------------------------------
def layer_forward(h: Array, W: LayerWeights, kcache: dict, vcache: dict, batch: Batch,
                  dims: Dims, rb: Callable = round_bf16) -> Array:
    """One pre-norm Llama decoder layer over the batch.

    kcache[b], vcache[b]: [n_kv, L_max, d] arrays of sequence b, updated in
    place at each token's position.  Returns the new hidden [T, H].
    """
    T = h.shape[0]
    nh, nkv, d = dims.n_heads, dims.n_kv_heads, dims.head_dim
    u = rb(rmsnorm(h, W.attn_norm, dims.rms_eps))
    q = linear(u, W.wq, W.bq).reshape(T, nh, d)
    k = linear(u, W.wk, W.bk).reshape(T, nkv, d)
    v = linear(u, W.wv, W.bv).reshape(T, nkv, d)
    q = rb(rope(q, batch.pos, dims.rope_theta))
    k = rb(rope(k, batch.pos, dims.rope_theta))
    v = rb(v)
    for i in range(T):
        b, p = int(batch.seq[i]), int(batch.pos[i])
        kcache[b][:, p, :] = k[i]
        vcache[b][:, p, :] = v[i]
    o = np.empty((T, nh, d))
    for i in range(T):
        b, p = int(batch.seq[i]), int(batch.pos[i])
        o[i] = gqa_attend_token(q[i], kcache[b], vcache[b], p)
    o = rb(o.reshape(T, nh * d))
    h = rb(h + linear(o, W.wo, W.bo))
    u2 = rb(rmsnorm(h, W.mlp_norm, dims.rms_eps))
    a = rb(silu(linear(u2, W.wg, W.bg)) * linear(u2, W.wu, W.bu))
    return rb(h + linear(a, W.wd, W.bd))


def embed(E: Array, ids: Array) -> Array:
    return E[np.asarray(ids)]


def lm_head(h_rows: Array, final_norm: Array, W_lm: Array, dims: Dims,
            rb: Callable = round_bf16) -> Array:
    x = rb(rmsnorm(h_rows, final_norm, dims.rms_eps))
    return rb(linear(x, W_lm))


def forward(ids: Array, E: Array, layers, final_norm: Array, W_lm: Array, batch: Batch,
            dims: Dims, rb: Callable = round_bf16, rows: Optional[Array] = None) -> Array:
    """The whole decoder forward in the order the pages draw it
    ("张量、流水线与数据并行", §线性层怎么切 flowchart and §输出层): the embedding
    lookup, then every layer in turn (attention block, then MLP), then the
    final RMSNorm and the LM head on the sampled rows.

    layers: iterable of (LayerWeights, kcache, vcache) in layer order (a
    generator may build each layer's weights on demand); rows: the token rows
    whose logits are returned (default: the last token of each sequence)."""
    h = embed(E, ids)
    for W, kc, vc in layers:
        h = layer_forward(h, W, kc, vc, batch, dims, rb)
    sel = batch.sample_rows() if rows is None else np.asarray(rows)
    return lm_head(h[sel], final_norm, W_lm, dims, rb)


# ---------------------------------------------------------------------------
# sharded emulation (t ranks, in order 0..t-1)
# ---------------------------------------------------------------------------
def shard_qkv(W: LayerWeights, dims: Dims, p: Plan) -> List[Array]:
    """Column-parallel qkv_proj: rank r holds the rows of its own Q heads and
    of its KV head(s) (copies of the KV rows when they are replicated)."""
    d = dims.head_dim
    out = []
    for r in range(p.t):
        qrows = np.concatenate([W.wq[j * d:(j + 1) * d] for j in q_heads_of_rank(p, r)])
        kvh = kv_heads_of_rank(p, dims.n_kv_heads, r)
        krows = np.concatenate([W.wk[g * d:(g + 1) * d] for g in kvh])
        vrows = np.concatenate([W.wv[g * d:(g + 1) * d] for g in kvh])
        out.append(np.concatenate([qrows, krows, vrows]))
    return out


def shard_qkv_bias(W: LayerWeights, dims: Dims, p: Plan) -> List[Array]:
    """Column-parallel bias: split with its weight along the output features
    ("第 9 章", §3.2: weights and their biases are cut along the output
    dimension), so rank r holds the bias entries of exactly its own q/k/v
    rows (copies for replicated KV heads)."""
    d = dims.head_dim
    zq = np.zeros(dims.n_heads * d) if W.bq is None else W.bq
    zk = np.zeros(dims.n_kv_heads * d) if W.bk is None else W.bk
    zv = np.zeros(dims.n_kv_heads * d) if W.bv is None else W.bv
    out = []
    for r in range(p.t):
        kvh = kv_heads_of_rank(p, dims.n_kv_heads, r)
        out.append(np.concatenate([zq[j * d:(j + 1) * d] for j in q_heads_of_rank(p, r)] +
                                  [zk[g * d:(g + 1) * d] for g in kvh] +
                                  [zv[g * d:(g + 1) * d] for g in kvh]))
    return out


def shard_gate_up_bias(W: LayerWeights, p: Plan) -> List[Array]:
    """The gate and up biases cut like their rows."""
    n = p.inter_per_rank
    I = p.inter_per_rank * p.t
    zg = np.zeros(I) if W.bg is None else W.bg
    zu = np.zeros(I) if W.bu is None else W.bu
    return [np.concatenate([zg[r * n:(r + 1) * n], zu[r * n:(r + 1) * n]]) for r in range(p.t)]


def shard_gate_up(W: LayerWeights, p: Plan) -> List[Array]:
    """Column-parallel gate_up_proj: rank r holds the matching slices of the
    gate and of the up rows, so SiLU(gate) * up needs no communication."""
    n = p.inter_per_rank
    return [np.concatenate([W.wg[r * n:(r + 1) * n], W.wu[r * n:(r + 1) * n]]) for r in range(p.t)]


def shard_rows_by_input(w: Array, t: int) -> List[Array]:
    """Row-parallel weight: split along the input dimension (columns of an
    [out, in] weight)."""
    k = w.shape[1] // t
    return [w[:, r * k:(r + 1) * k] for r in range(t)]


def shard_vocab(E: Array, p: Plan) -> List[Array]:
    """Vocab-parallel table: pad the vocabulary to a multiple of t with zero
    rows and give rank r rows [r Vp/t, (r+1) Vp/t)."""
    V, H = E.shape
    padded = np.zeros((p.vocab_padded, H))
    padded[:V] = E
    n = p.vocab_per_rank
    return [padded[r * n:(r + 1) * n] for r in range(p.t)]


def all_reduce_sum(partials: Sequence[Array]) -> Array:
    """Y = Y_0 + Y_1 + ... + Y_{t-1}, summed in rank order."""
    acc = partials[0].copy()
    for y in partials[1:]:
        acc = acc + y
    return acc


def all_gather_cat(parts: Sequence[Array]) -> Array:
    """Y = cat(Y_0, ..., Y_{t-1}) along the last (vocab) dimension."""
    return np.concatenate(list(parts), axis=-1)


def sharded_embed(E_shards: List[Array], ids: Array, p: Plan, fill: float = -0.0) -> Array:
    """Each rank looks up only the ids in its vocab range and contributes
    ``fill`` elsewhere; an all-reduce sums the t contributions.  With fill
    -0.0 the sum reproduces E[id] bit for bit (x + (-0.0) == x for every x)."""
    n = p.vocab_per_rank
    H = E_shards[0].shape[1]
    parts = []
    for r in range(p.t):
        local = np.asarray(ids) - r * n
        mine = (local >= 0) & (local < n)
        y = np.full((len(ids), H), fill)
        y[mine] = E_shards[r][local[mine]]
        parts.append(y)
    return all_reduce_sum(parts)


def sharded_lm_head(x: Array, L_shards: List[Array], vocab: int, rb: Callable = round_bf16) -> Array:
    """Each rank computes its V/t logits; the all-gather concatenates them in
    vocab order; the padding columns are dropped."""
    return all_gather_cat([rb(linear(x, Lr)) for Lr in L_shards])[:, :vocab]


def sharded_layer_forward(h: Array, W: LayerWeights, kcopies: List[dict], vcopies: List[dict],
                          batch: Batch, dims: Dims, p: Plan, rb: Callable = round_bf16,
                          skip_allreduce: bool = False, bias_on_every_rank: bool = False) -> Array:
    """The same layer computed as t ranks: column shards with no
    communication, per-rank attention over the rank's own heads and cache,
    row-parallel partials summed by an all-reduce (① after o_proj, ② after
    down_proj).  kcopies[c][b]: cache copy c of sequence b, [kv_r, L_max, d].

    ``skip_allreduce`` keeps only rank 0's partial (the "missing collective"
    fault of the pages' debugging checklist).  A row-parallel bias belongs to
    the whole output, so it is added once, after the all-reduce;
    ``bias_on_every_rank`` instead adds it to every rank's partial (the t-fold
    bias a misplaced add would produce), for the tests."""
    T = h.shape[0]
    d = dims.head_dim
    nq = p.q_heads_per_rank
    group = dims.n_heads // dims.n_kv_heads
    reduce = (lambda parts: parts[0]) if skip_allreduce else all_reduce_sum

    def row_bias(partials, b):
        if b is None:
            return reduce(partials)
        if bias_on_every_rank:
            return reduce([y + b for y in partials])
        return reduce(partials) + b

    u = rb(rmsnorm(h, W.attn_norm, dims.rms_eps))       # replicated on every rank
    qkv_sh = shard_qkv(W, dims, p)
    qkv_b = shard_qkv_bias(W, dims, p)
    o_parts = []
    for r in range(p.t):
        y = linear(u, qkv_sh[r], qkv_b[r])                # Y_r = X A_r + b_r
        kvh = kv_heads_of_rank(p, dims.n_kv_heads, r)
        nkv = len(kvh)
        q = rb(rope(y[:, : nq * d].reshape(T, nq, d), batch.pos, dims.rope_theta))
        k = rb(rope(y[:, nq * d:(nq + nkv) * d].reshape(T, nkv, d), batch.pos, dims.rope_theta))
        v = rb(y[:, (nq + nkv) * d:].reshape(T, nkv, d))
        c = kv_copy_of_rank(p, r)
        for i in range(T):
            b, pos = int(batch.seq[i]), int(batch.pos[i])
            kcopies[c][b][:, pos, :] = k[i]
            vcopies[c][b][:, pos, :] = v[i]
        o_parts.append((q, kvh, c))
    Wo_sh = shard_rows_by_input(W.wo, p.t)
    partials = []
    for r, (q, kvh, c) in enumerate(o_parts):
        o = np.empty((T, nq, d))
        for i in range(T):
            b, pos = int(batch.seq[i]), int(batch.pos[i])
            for jl, j in enumerate(q_heads_of_rank(p, r)):
                gl = kvh.index(j // group)
                o[i, jl] = attend(q[i, jl], kcopies[c][b][gl, : pos + 1], vcopies[c][b][gl, : pos + 1])
        partials.append(linear(rb(o.reshape(T, nq * d)), Wo_sh[r]))
    h = rb(h + row_bias(partials, W.bo))

    u2 = rb(rmsnorm(h, W.mlp_norm, dims.rms_eps))
    gu_sh = shard_gate_up(W, p)
    gu_b = shard_gate_up_bias(W, p)
    Wd_sh = shard_rows_by_input(W.wd, p.t)
    n = p.inter_per_rank
    partials = []
    for r in range(p.t):
        y = linear(u2, gu_sh[r], gu_b[r])
        a = rb(silu(y[:, :n]) * y[:, n:])
        partials.append(linear(a, Wd_sh[r]))
    return rb(h + row_bias(partials, W.bd))


def split_cache_copies(kcache: dict, dims: Dims, p: Plan) -> List[dict]:
    """Per-rank cache copies viewing the logical cache: copy c holds the KV
    heads of its owner rank(s)."""
    out = []
    for c in range(p.kv_copies):
        if p.kv_replicas == 1:
            heads = slice(c * p.kv_heads_per_rank, (c + 1) * p.kv_heads_per_rank)
        else:
            heads = slice(c, c + 1)
        out.append({b: arr[heads] for b, arr in kcache.items()})
    return out


# ---------------------------------------------------------------------------
# DP attention ("张量、流水线与数据并行", SGLang 的 DP attention): the t ranks of
# a TP group split into attn_dp attention groups.  Each group batches its own
# sequences and keeps their KV, with the attention part tensor-parallel over
# attn_tp = t / attn_dp ranks; the FFN stays tensor-parallel over all t
# ranks, so the tokens of every group are gathered before it and each group
# keeps its own rows after it.
# Readings: sequences are dealt to the groups in contiguous blocks
# (group k gets sequences [k*ceil(B/attn_dp), ...)); the gather before the FFN
# is an all-gather of the groups' hidden rows; the FFN's own reduction is the
# usual all-reduce over t ranks, after which each group takes its rows back
# (no further traffic).
# ---------------------------------------------------------------------------
def attn_tp_size(t: int, attn_dp: int) -> int:
    """The attention TP width left inside one DP group."""
    if attn_dp < 1 or t % attn_dp:
        raise RuleError("attn_dp must divide t")
    return t // attn_dp


def dp_group_of_seq(n_seqs: int, attn_dp: int, b: int) -> int:
    per = -(-n_seqs // attn_dp)
    return b // per


def kv_bytes_per_rank(n_seqs: int, n_kv_heads: int, head_dim: int, ctx: int, t: int,
                      attn_dp: int = 1, elem_bytes: int = 2) -> int:
    """K and V bytes one rank keeps for one layer: its attention group's
    sequences (all of them under plain TP), and its KV heads among the
    group's attn_tp ranks (one replicated head when n_kv < attn_tp)."""
    atp = attn_tp_size(t, attn_dp)
    heads = n_kv_heads // atp if n_kv_heads >= atp else 1
    seqs = -(-n_seqs // attn_dp)
    return seqs * heads * ctx * head_dim * 2 * elem_bytes


def dp_gather_received_per_rank(tokens_per_group: Sequence[int], hidden: int,
                                elem_bytes: int = 2) -> List[int]:
    """Hidden-row bytes each group's ranks receive from the other groups when
    the tokens are gathered for the FFN."""
    total = sum(tokens_per_group)
    return [(total - n) * hidden * elem_bytes for n in tokens_per_group]


def dp_attention_layer_forward(h: Array, W: LayerWeights, kcopies: List[dict],
                               vcopies: List[dict], batch: Batch, dims: Dims, t: int,
                               attn_dp: int, rb: Callable = round_bf16) -> Array:
    """One layer with DP attention.  kcopies / vcopies: the cache copies of
    the attention plan (attn_tp ranks), indexed [copy][sequence]; a group's
    ranks touch only its own sequences."""
    atp = attn_tp_size(t, attn_dp)
    pa = plan(dims.n_heads, dims.n_kv_heads, dims.intermediate, dims.vocab, atp)
    pf = plan(dims.n_heads, dims.n_kv_heads, dims.intermediate, dims.vocab, t)
    n_seqs = int(np.max(batch.seq)) + 1 if len(batch.seq) else 0
    T = h.shape[0]
    d = dims.head_dim
    nq = pa.q_heads_per_rank
    group = dims.n_heads // dims.n_kv_heads
    qkv_sh = shard_qkv(W, dims, pa)
    qkv_b = shard_qkv_bias(W, dims, pa)
    Wo_sh = shard_rows_by_input(W.wo, atp)
    h_after = np.empty_like(h)
    for k in range(attn_dp):
        rows = np.array([i for i in range(T) if dp_group_of_seq(n_seqs, attn_dp, int(batch.seq[i])) == k],
                        dtype=np.int64)
        if len(rows) == 0:
            continue
        hk = h[rows]
        u = rb(rmsnorm(hk, W.attn_norm, dims.rms_eps))
        parts = []
        for r in range(atp):                                  # the group's attention ranks
            y = linear(u, qkv_sh[r], qkv_b[r])
            kvh = kv_heads_of_rank(pa, dims.n_kv_heads, r)
            nkv = len(kvh)
            pos = batch.pos[rows]
            q = rb(rope(y[:, : nq * d].reshape(len(rows), nq, d), pos, dims.rope_theta))
            kk = rb(rope(y[:, nq * d:(nq + nkv) * d].reshape(len(rows), nkv, d), pos, dims.rope_theta))
            v = rb(y[:, (nq + nkv) * d:].reshape(len(rows), nkv, d))
            c = kv_copy_of_rank(pa, r)
            for i, row in enumerate(rows):
                b, p = int(batch.seq[row]), int(batch.pos[row])
                kcopies[c][b][:, p, :] = kk[i]
                vcopies[c][b][:, p, :] = v[i]
            parts.append((q, kvh, c))
        partials = []
        for r, (q, kvh, c) in enumerate(parts):
            o = np.empty((len(rows), nq, d))
            for i, row in enumerate(rows):
                b, p = int(batch.seq[row]), int(batch.pos[row])
                for jl, j in enumerate(q_heads_of_rank(pa, r)):
                    gl = kvh.index(j // group)
                    o[i, jl] = attend(q[i, jl], kcopies[c][b][gl, : p + 1], vcopies[c][b][gl, : p + 1])
            partials.append(linear(rb(o.reshape(len(rows), nq * d)), Wo_sh[r]))
        red = all_reduce_sum(partials)                          # inside the attention group
        h_after[rows] = rb(hk + (red if W.bo is None else red + W.bo))
    # gather every group's rows, FFN over all t ranks, each group keeps its rows
    u2 = rb(rmsnorm(h_after, W.mlp_norm, dims.rms_eps))
    gu_sh = shard_gate_up(W, pf)
    gu_b = shard_gate_up_bias(W, pf)
    Wd_sh = shard_rows_by_input(W.wd, t)
    n = pf.inter_per_rank
    partials = []
    for r in range(t):
        y = linear(u2, gu_sh[r], gu_b[r])
        a = rb(silu(y[:, :n]) * y[:, n:])
        partials.append(linear(a, Wd_sh[r]))
    red = all_reduce_sum(partials)
    return rb(h_after + (red if W.bd is None else red + W.bd))
