"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test ties an oracle function to something other than itself: a value the
pages print, a closed form, an invariant, a library routine, or the exact
equality that tensor parallelism is a re-association of the unsharded math.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------
def test_round_bf16_matches_torch_on_float32_inputs():
    # torch's float32 -> bf16 conversion rounds to nearest even: a library routine
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    bits[:1000] = (bits[:1000] & 0xFFFF0000) | 0x8000          # exact ties
    bits[1000:2000] = bits[1000:2000] & 0x807FFFFF              # float32 subnormals
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    f = f[np.abs(f) < 3.0e38]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    got = O.round_bf16(f.astype(np.float64))
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_round_bf16_ties_and_direct_rounding():
    one = 1.0
    assert O.round_bf16(one + 2.0**-8) == 1.0                      # tie -> even
    assert O.round_bf16(one + 3 * 2.0**-8) == one + 2.0**-6        # tie -> even (up)
    # just above a tie: a float64 -> float32 -> bf16 double rounding would give 1.0
    assert O.round_bf16(one + 2.0**-8 + 2.0**-40) == one + 2.0**-7
    assert np.signbit(O.round_bf16(-0.0))
    assert O.round_bf16(3.5e38) == np.inf and O.round_bf16(-3.5e38) == -np.inf
    assert O.round_bf16(2.0**-133) == 2.0**-133                    # smallest subnormal
    assert O.round_bf16(2.0**-135) == 0.0


def test_round_bf16_agrees_with_the_generator_conversion():
    # two independent implementations (numpy frexp/rint vs the generator's C)
    x = synth.normal_f64(7, 99, (100_000,), 0.02)
    assert np.array_equal(O.round_bf16(x), x)                     # already bf16 values


# ---------------------------------------------------------------------------
# linear / RMSNorm / SiLU / softmax
# ---------------------------------------------------------------------------
def test_linear_orientation():
    # W stored [out, in]; y_o = sum_i x_i W[o, i]; a transposed operand fails
    W = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, 7.0]])
    x = np.array([[10.0, 100.0]])
    assert np.array_equal(O.linear(x, W), np.array([[210.0, 430.0, 750.0]]))


def test_rmsnorm_closed_forms():
    H, eps = 64, 1e-5
    w = 1.0 + rng.standard_normal(H) * 0.1
    c = -0.37
    y = O.rmsnorm(np.full((1, H), c), w, eps)
    assert np.allclose(y, w * c / math.sqrt(c * c + eps), rtol=1e-14)
    a = 5.0
    x = np.zeros((1, H)); x[0, 3] = a
    y = O.rmsnorm(x, w, eps)
    assert np.isclose(y[0, 3], a / math.sqrt(a * a / H + eps) * w[3], rtol=1e-14)
    assert np.count_nonzero(y) == 1
    # mean of squares of the output (w = 1) is 1 up to eps
    z = rng.standard_normal((3, H)) * 4
    out = O.rmsnorm(z, np.ones(H), 0.0)
    assert np.allclose(np.mean(out * out, axis=-1), 1.0, rtol=1e-13)


def test_rmsnorm_weight_folds_into_the_next_linear():
    # the reading behind the CUDA path's decode layer: a norm's weight can be
    # multiplied into the columns of the linear that reads its output, and the
    # per-token 1/rms applied to that linear's output instead
    H, N, M, eps = 96, 40, 5, 1e-5
    w = 1.0 + rng.standard_normal(H) * 0.3
    W = rng.standard_normal((N, H)) * 0.02
    b = rng.standard_normal(N)
    x = rng.standard_normal((M, H)) * 3
    ref = O.linear(O.rmsnorm(x, w, eps), W, b)
    rstd = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    folded = O.linear(x, W * w[None, :]) * rstd + b
    assert np.allclose(folded, ref, rtol=1e-12, atol=1e-14)
    # scaling the output rows by 1/rms of the wrong token, or folding w into
    # the rows (output features) instead of the columns, is caught
    assert not np.allclose(O.linear(x, W * w[None, :]) * rstd[::-1] + b, ref, rtol=1e-3)
    Wr = W * w[:N, None]
    assert not np.allclose(O.linear(x, Wr) * rstd + b, ref, rtol=1e-3)


def test_silu_against_expit():
    x = np.linspace(-30, 30, 1001)
    assert np.allclose(O.silu(x), x * scipy.special.expit(x), rtol=1e-13, atol=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(O.silu(x) - O.silu(-x), x, rtol=1e-12, atol=1e-12)


def test_softmax_and_attention_special_cases():
    s = rng.standard_normal((5, 17)) * 3
    assert np.allclose(O.softmax(s), scipy.special.softmax(s, axis=-1), rtol=1e-13)
    d = 16
    v1 = rng.standard_normal((1, d)); k1 = rng.standard_normal((1, d))
    assert np.allclose(O.attend(rng.standard_normal(d), k1, v1), v1[0])          # L = 1
    k = rng.standard_normal((9, d)); v = rng.standard_normal((9, d))
    assert np.allclose(O.attend(np.zeros(d), k, v), v.mean(axis=0))             # q = 0
    kk = np.zeros((9, d)); kk[4, 0] = 1.0
    q = np.zeros(d); q[0] = 4000.0
    assert np.allclose(O.attend(q, kk, v), v[4])                                # one-hot
    # scores are scaled by 1/sqrt(d): two keys whose dot products differ by sqrt(d)*ln 3
    k2 = np.zeros((2, d)); k2[0, 0] = math.sqrt(d) * math.log(3.0)
    q2 = np.zeros(d); q2[0] = 1.0
    v2 = np.array([np.ones(d), np.zeros(d)])
    assert np.allclose(O.attend(q2, k2, v2), 0.75 * np.ones(d))


def test_gqa_head_to_kv_head_map():
    nh, nkv, L, d = 8, 2, 3, 4
    kc = np.zeros((nkv, L, d))
    vc = np.stack([np.full((L, d), float(g)) for g in range(nkv)])
    q = rng.standard_normal((nh, d))
    o = O.gqa_attend_token(q, kc, vc, L - 1)
    assert np.array_equal(o[:, 0], np.array([0, 0, 0, 0, 1, 1, 1, 1], dtype=float))


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------
def test_rope_convention_and_invariants():
    d, theta = 8, 10000.0
    assert np.allclose(O.rope_inv_freq(4, theta), [1.0, 0.01])
    x = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    p = 2.5
    assert np.allclose(O.rope(x, np.array([p]), theta), [[[math.cos(p), 0, math.sin(p), 0]]])
    X = rng.standard_normal((6, 3, d))
    assert np.array_equal(O.rope(X, np.zeros(6), theta), X)                       # p = 0
    pos = rng.integers(0, 5000, 6).astype(float)
    Y = O.rope(X, pos, theta)
    # complex multiplication of the (j, j + d/2) pairs by exp(i p theta_j)
    z = X[..., : d // 2] + 1j * X[..., d // 2:]
    zr = z * np.exp(1j * pos[:, None, None] * O.rope_inv_freq(d, theta)[None, None, :])
    assert np.allclose(Y[..., : d // 2], zr.real, atol=1e-12)
    assert np.allclose(Y[..., d // 2:], zr.imag, atol=1e-12)
    assert np.allclose(np.linalg.norm(Y, axis=-1), np.linalg.norm(X, axis=-1))
    # relative position: <rope(q, m), rope(k, n)> depends on m - n only
    q = rng.standard_normal((1, 1, d)); k = rng.standard_normal((1, 1, d))
    a = np.sum(O.rope(q, [7.0], theta) * O.rope(k, [3.0], theta))
    b = np.sum(O.rope(q, [107.0], theta) * O.rope(k, [103.0], theta))
    assert np.isclose(a, b, rtol=1e-10)


# ---------------------------------------------------------------------------
# rules and counts printed on the pages
# ---------------------------------------------------------------------------
def test_sharding_rules_golden():
    g = json.load(open(os.path.join(GOLDEN, "sharding_rules.json")))
    for c in g["cases"]:
        p = O.plan(c["n_heads"], c["n_kv_heads"], c["intermediate"], c["vocab"], c["t"])
        assert (p.q_heads_per_rank, p.kv_heads_per_rank, p.kv_replicas, p.vocab_padded) == \
            (c["q_per_rank"], c["kv_per_rank"], c["replicas"], c["vocab_padded"]), c
        assert p.vocab_padded % c["t"] == 0 and p.vocab_padded >= c["vocab"]
        assert p.vocab_padded - c["vocab"] < c["t"]
    for c in g["invalid"]:
        with pytest.raises(O.RuleError):
            O.plan(c["n_heads"], c["n_kv_heads"], c["intermediate"], c["vocab"], c["t"])


def test_kv_replica_assignment_matches_q_heads():
    # 40 Q heads, 4 KV heads, t = 8: rank r's Q heads 5r..5r+4 all read KV head r // 2
    p = O.plan(40, 4, 27648, 152064, 8)
    for r in range(8):
        assert O.kv_heads_of_rank(p, 4, r) == [r // 2]
        assert {j // 10 for j in O.q_heads_of_rank(p, r)} == {r // 2}
    p = O.plan(40, 8, 27648, 152064, 8)
    for r in range(8):
        assert {j // 5 for j in O.q_heads_of_rank(p, r)} == set(O.kv_heads_of_rank(p, 8, r))


def test_payload_counts_golden():
    g = json.load(open(os.path.join(GOLDEN, "payload_counts.json")))
    m = g["model"]
    assert O.allreduces_per_forward(m["n_layers"]) == g["allreduces_per_forward"]
    per_tok = O.allreduce_payload_bytes_per_token(m["hidden"], m["elem_bytes"])
    assert per_tok == g["allreduce_payload_bytes_per_token"]
    total = per_tok * O.allreduces_per_forward(m["n_layers"])
    assert total == g["allreduce_payload_kib_per_token_total"] * 1024
    for t, kib in g["ring_bytes_sent_per_rank_per_token_kib"].items():
        assert O.ring_bytes_sent_per_rank(total, int(t)) == kib * 1024
        assert 2 * (int(t) - 1) / int(t) == g["ring_factor"][t]
    for t, kib in g["logits_allgather_received_per_rank_kib_rounded"].items():
        assert round(O.logits_gather_received_per_rank(m["vocab"], int(t)) / 1024) == kib
    for s in g["step_payloads"]:
        assert s["tokens"] * per_tok == s["per_allreduce_kib"] * 1024
        mib = s["tokens"] * total / 2**20
        assert f"{mib:.1f}" == s["total_mib_printed"]
    for t, kib in g["kv_per_token_per_rank_kib"].items():
        assert O.kv_bytes_per_token_per_rank(m["n_layers"], m["n_kv_heads"], m["head_dim"], int(t)) \
            == kib * 1024


# ---------------------------------------------------------------------------
# embedding / LM head sharding
# ---------------------------------------------------------------------------
def test_sharded_embedding_is_bit_exact_with_negative_zero_fill():
    V, H = 1001, 32
    E = synth.normal_f64(3, 1, (V, H), 0.02)
    E[5, :4] = -0.0
    ids = np.concatenate([rng.integers(0, V, 200), [0, V - 1, 5, 500, 501]])
    ref = O.embed(E, ids)
    for t in (1, 2, 4, 7, 8):
        p = O.plan(8, 8, 8 * 7, V, t) if t in (1, 2, 4, 8) else O.Plan(t, 1, 1, 1, 1, -(-V // t) * t,
                                                                       -(-V // t), 1)
        got = O.sharded_embed(O.shard_vocab(E, p), ids, p)
        assert np.array_equal(got.view(np.uint64), ref.view(np.uint64)), t
    # the reading matters: a +0.0 fill turns -0.0 entries into +0.0
    p = O.plan(8, 8, 56, V, 2)
    plus = O.sharded_embed(O.shard_vocab(E, p), np.array([5]), p, fill=0.0)
    assert not np.array_equal(plus.view(np.uint64), O.embed(E, [5]).view(np.uint64))


def test_sharded_lm_head_equals_unsharded_and_drops_padding():
    V, H = 1001, 48
    W = synth.normal_f64(3, 2, (V, H), 0.02)
    x = synth.normal_f64(3, 3, (3, H), 1.0)
    ref = O.round_bf16(O.linear(x, W))
    for t in (1, 2, 4, 8):
        p = O.plan(8, 8, 56, V, t)
        got = O.sharded_lm_head(x, O.shard_vocab(W, p), V)
        assert got.shape == (3, V)
        assert np.array_equal(got, ref)        # vocab sharding never splits K


# ---------------------------------------------------------------------------
# the sharded layer equals the unsharded layer (exact re-association)
# ---------------------------------------------------------------------------
def _tiny(n_heads, n_kv, d=16, H=64, I=96, seed=5):
    dims = O.Dims(H, n_heads, n_kv, d, I, 1000)
    W = O.LayerWeights(
        attn_norm=1.0 + synth.normal_f64(seed, 1, (H,), 0.1),
        wq=synth.normal_f64(seed, 2, (n_heads * d, H), 0.1),
        wk=synth.normal_f64(seed, 3, (n_kv * d, H), 0.1),
        wv=synth.normal_f64(seed, 4, (n_kv * d, H), 0.1),
        wo=synth.normal_f64(seed, 5, (H, n_heads * d), 0.1),
        mlp_norm=1.0 + synth.normal_f64(seed, 6, (H,), 0.1),
        wg=synth.normal_f64(seed, 7, (I, H), 0.1),
        wu=synth.normal_f64(seed, 8, (I, H), 0.1),
        wd=synth.normal_f64(seed, 9, (H, I), 0.1))
    return dims, W


def _caches(n_seqs, n_kv, L, d, seed=11):
    kc = {b: synth.normal_f64(seed, 100 + b, (n_kv, L, d), 1.0) for b in range(n_seqs)}
    vc = {b: synth.normal_f64(seed, 200 + b, (n_kv, L, d), 1.0) for b in range(n_seqs)}
    return kc, vc


def _copy(c):
    return {b: a.copy() for b, a in c.items()}


@pytest.mark.parametrize("n_heads,n_kv,t", [
    (4, 4, 1), (4, 4, 2), (4, 4, 4), (4, 2, 2), (4, 2, 4), (4, 1, 2), (4, 1, 4),
    (8, 2, 8), (8, 4, 2), (6, 3, 3), (6, 2, 6), (6, 3, 6)])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_sharded_layer_equals_unsharded(n_heads, n_kv, t, mode):
    dims, W = _tiny(n_heads, n_kv)
    if mode == "decode":
        n_seqs, L = 3, 7
        batch = O.Batch.decode(n_seqs, L)
    else:
        n_seqs, L = 2, 5
        batch = O.Batch.prefill(n_seqs, L)
    T = len(batch.seq)
    h = synth.normal_f64(9, 9, (T, dims.hidden), 1.0)
    kc, vc = _caches(n_seqs, n_kv, L, dims.head_dim)
    p = O.plan(n_heads, n_kv, dims.intermediate, dims.vocab, t)
    for rb, tol in ((O.no_round, 1e-12), (O.round_bf16, 1e-2)):
        k1, v1 = _copy(kc), _copy(vc)
        ref = O.layer_forward(h, W, k1, v1, batch, dims, rb=rb)
        k2, v2 = _copy(kc), _copy(vc)
        got = O.sharded_layer_forward(h, W, O.split_cache_copies(k2, dims, p),
                                      O.split_cache_copies(v2, dims, p), batch, dims, p, rb=rb)
        err = np.max(np.abs(got - ref)) / (np.max(np.abs(ref)) + 1e-6)
        assert err <= tol, (rb, err)
        for b in k1:
            assert np.allclose(k1[b], k2[b], rtol=tol, atol=tol) and np.allclose(v1[b], v2[b], rtol=tol, atol=tol)


def test_missing_allreduce_is_wrong():
    dims, W = _tiny(4, 2)
    batch = O.Batch.decode(2, 5)
    h = synth.normal_f64(9, 9, (2, dims.hidden), 1.0)
    kc, vc = _caches(2, 2, 5, dims.head_dim)
    p = O.plan(4, 2, dims.intermediate, dims.vocab, 2)
    ref = O.layer_forward(h, W, _copy(kc), _copy(vc), batch, dims)
    bad = O.sharded_layer_forward(h, W, O.split_cache_copies(_copy(kc), dims, p),
                                  O.split_cache_copies(_copy(vc), dims, p), batch, dims, p,
                                  skip_allreduce=True)
    assert np.max(np.abs(bad - ref)) / np.max(np.abs(ref)) > 0.05


def test_naive_cut_of_concatenated_gate_up_is_wrong():
    dims, W = _tiny(4, 2)
    p = O.plan(4, 2, dims.intermediate, dims.vocab, 2)
    u = synth.normal_f64(9, 10, (3, dims.hidden), 1.0)
    n = p.inter_per_rank
    ref = O.silu(O.linear(u, W.wg)) * O.linear(u, W.wu)
    good = np.concatenate([
        O.silu(O.linear(u, s)[:, :n]) * O.linear(u, s)[:, n:] for s in O.shard_gate_up(W, p)], axis=1)
    assert np.allclose(good, ref, rtol=1e-12, atol=1e-14)
    cat = np.concatenate([W.wg, W.wu])
    naive = [cat[r * 2 * n:(r + 1) * 2 * n] for r in range(p.t)]
    bad = np.concatenate([O.silu(O.linear(u, s)[:, :n]) * O.linear(u, s)[:, n:] for s in naive], axis=1)
    assert not np.allclose(bad, ref, rtol=1e-2)


def test_zero_projections_leave_the_residual_stream_unchanged():
    dims, W = _tiny(4, 2)
    W.wo[:] = 0.0
    W.wd[:] = 0.0
    batch = O.Batch.prefill(1, 4)
    h = O.round_bf16(synth.normal_f64(9, 12, (4, dims.hidden), 1.0))
    kc, vc = _caches(1, 2, 4, dims.head_dim)
    assert np.array_equal(O.layer_forward(h, W, kc, vc, batch, dims), h)


def test_decode_step_equals_last_prefill_row_and_causality():
    dims, W = _tiny(4, 2)
    L = 6
    h = synth.normal_f64(9, 13, (L, dims.hidden), 1.0)
    kc, vc = _caches(1, 2, L, dims.head_dim)
    kp, vp = _copy(kc), _copy(vc)
    pre = O.layer_forward(h, W, kp, vp, O.Batch.prefill(1, L), dims, rb=O.no_round)
    # decode the last token against a cache holding the prefill's K/V for 0..L-2
    kd, vd = _copy(kp), _copy(vp)
    kd[0][:, L - 1] = 123.0
    dec = O.layer_forward(h[L - 1:], W, kd, vd, O.Batch.decode(1, L), dims, rb=O.no_round)
    assert np.allclose(dec[0], pre[L - 1], rtol=1e-12, atol=1e-12)
    # causal: changing a later token does not change earlier rows
    h2 = h.copy(); h2[L - 1] += 1.0
    pre2 = O.layer_forward(h2, W, _copy(kc), _copy(vc), O.Batch.prefill(1, L), dims, rb=O.no_round)
    assert np.array_equal(pre2[: L - 1], pre[: L - 1])
    # first position attends only to itself: its attention output is v_0
    assert not np.array_equal(pre2[L - 1], pre[L - 1])


def test_prefill_sequences_do_not_see_each_other():
    dims, W = _tiny(4, 2)
    L = 4
    h = synth.normal_f64(9, 14, (2 * L, dims.hidden), 1.0)
    kc, vc = _caches(2, 2, L, dims.head_dim)
    both = O.layer_forward(h, W, _copy(kc), _copy(vc), O.Batch.prefill(2, L), dims, rb=O.no_round)
    kc1 = {0: kc[1].copy()}; vc1 = {0: vc[1].copy()}
    alone = O.layer_forward(h[L:], W, kc1, vc1, O.Batch.prefill(1, L), dims, rb=O.no_round)
    assert np.allclose(both[L:], alone, rtol=1e-12, atol=1e-12)


def test_batch_sample_rows_are_last_tokens():
    b = O.Batch.prefill(3, 4)
    assert list(b.sample_rows()) == [3, 7, 11]
    assert list(O.Batch.decode(5, 9).sample_rows()) == [0, 1, 2, 3, 4]


# ---------------------------------------------------------------------------
# projection biases ("第 9 章", §3.2: a weight and its bias are cut along the
# output dimension; the bias of a row-parallel output is added once)
# ---------------------------------------------------------------------------
def _with_biases(dims, W, seed=21, sigma=0.5):
    d, H, I = dims.head_dim, dims.hidden, dims.intermediate
    W.bq = synth.normal_f64(seed, 1, (dims.n_heads * d,), sigma)
    W.bk = synth.normal_f64(seed, 2, (dims.n_kv_heads * d,), sigma)
    W.bv = synth.normal_f64(seed, 3, (dims.n_kv_heads * d,), sigma)
    W.bo = synth.normal_f64(seed, 4, (H,), sigma)
    W.bg = synth.normal_f64(seed, 5, (I,), sigma)
    W.bu = synth.normal_f64(seed, 6, (I,), sigma)
    W.bd = synth.normal_f64(seed, 7, (H,), sigma)
    return W


def test_linear_bias_closed_forms():
    x = np.array([[1.0, 2.0], [3.0, -1.0]])
    w = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0]])
    b = np.array([0.5, -0.25, 10.0])
    assert np.array_equal(O.linear(x, w, b), np.array([[1.5, 1.75, 13.0], [3.5, -1.25, 12.0]]))
    assert np.array_equal(O.linear(x, np.zeros((3, 2)), b), np.tile(b, (2, 1)))


def test_row_parallel_biases_enter_once():
    # with o_proj and down_proj weights zero the layer reduces to
    # h -> round(round(h + bo) + bd), whatever the attention and MLP compute
    dims, W = _tiny(4, 2)
    W = _with_biases(dims, W)
    W.wo[:] = 0.0
    W.wd[:] = 0.0
    batch = O.Batch.decode(2, 5)
    h = O.round_bf16(synth.normal_f64(9, 13, (2, dims.hidden), 1.0))
    kc, vc = _caches(2, 2, 5, dims.head_dim)
    want = O.round_bf16(O.round_bf16(h + W.bo) + W.bd)
    assert np.array_equal(O.layer_forward(h, W, _copy(kc), _copy(vc), batch, dims), want)
    for t in (2, 4):
        p = O.plan(4, 2, dims.intermediate, dims.vocab, t)
        got = O.sharded_layer_forward(h, W, O.split_cache_copies(_copy(kc), dims, p),
                                      O.split_cache_copies(_copy(vc), dims, p), batch, dims, p)
        assert np.array_equal(got, want)
        bad = O.sharded_layer_forward(h, W, O.split_cache_copies(_copy(kc), dims, p),
                                      O.split_cache_copies(_copy(vc), dims, p), batch, dims, p,
                                      rb=O.no_round, bias_on_every_rank=True)
        assert np.allclose(bad - h, t * (W.bo + W.bd), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n_heads,n_kv,t", [(4, 4, 2), (4, 2, 4), (4, 1, 2), (8, 2, 8), (6, 3, 3)])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_sharded_layer_with_biases_equals_unsharded(n_heads, n_kv, t, mode):
    dims, W = _tiny(n_heads, n_kv)
    W = _with_biases(dims, W)
    batch = O.Batch.decode(3, 7) if mode == "decode" else O.Batch.prefill(2, 5)
    n_seqs = 3 if mode == "decode" else 2
    L = 7 if mode == "decode" else 5
    T = len(batch.seq)
    h = synth.normal_f64(9, 9, (T, dims.hidden), 1.0)
    kc, vc = _caches(n_seqs, n_kv, L, dims.head_dim)
    p = O.plan(n_heads, n_kv, dims.intermediate, dims.vocab, t)
    ref = O.layer_forward(h, W, _copy(kc), _copy(vc), batch, dims, rb=O.no_round)
    got = O.sharded_layer_forward(h, W, O.split_cache_copies(_copy(kc), dims, p),
                                  O.split_cache_copies(_copy(vc), dims, p), batch, dims, p,
                                  rb=O.no_round)
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= 1e-12
    # and the biases matter at this scale
    W0 = _tiny(n_heads, n_kv)[1]
    nob = O.layer_forward(h, W0, _copy(kc), _copy(vc), batch, dims, rb=O.no_round)
    assert np.max(np.abs(nob - ref)) / np.max(np.abs(ref)) > 0.05


def test_qk_bias_is_added_before_rope():
    # head_dim 2 (one rotation pair, angle = position x 1 rad), one head, one
    # KV head, zero q/k weights: q = R(1) bq and k_new = R(1) bk at position 1,
    # against a cached key k0 at position 0.  Attention weights of the two
    # keys are softmax([q.k0, q.k_new] / sqrt(2)); with bq = (1, 0), bk = (0, 0),
    # k0 = (1, 0): q.k0 = cos 1 (bias rotated) rather than 1 (bias added after
    # the rotation); the output is the weighted mix of v0 and v_new = bv.
    H = 4
    dims = O.Dims(H, 1, 1, 2, 4, 10)
    z = lambda *s: np.zeros(s)
    W = O.LayerWeights(attn_norm=np.ones(H), wq=z(2, H), wk=z(2, H), wv=z(2, H),
                       wo=np.eye(H, 2), mlp_norm=np.ones(H), wg=z(4, H), wu=z(4, H), wd=z(H, 4),
                       bq=np.array([1.0, 0.0]), bk=np.zeros(2), bv=np.array([0.0, 3.0]))
    batch = O.Batch.decode(1, 2)               # the new token sits at position 1
    kc = {0: np.array([[[1.0, 0.0], [0.0, 0.0]]])}
    vc = {0: np.array([[[2.0, 0.0], [0.0, 0.0]]])}
    h = np.zeros((1, H))
    out = O.layer_forward(h, W, kc, vc, batch, dims, rb=O.no_round)
    s0, s1 = np.cos(1.0) / np.sqrt(2.0), 0.0
    a0 = np.exp(s0) / (np.exp(s0) + np.exp(s1))
    want = np.array([2.0 * a0, 3.0 * (1 - a0), 0.0, 0.0])
    assert np.allclose(out[0], want, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# DP attention ("张量、流水线与数据并行", SGLang 的 DP attention)
# ---------------------------------------------------------------------------
def test_attn_tp_width_rule():
    assert O.attn_tp_size(8, 1) == 8 and O.attn_tp_size(8, 2) == 4 and O.attn_tp_size(8, 8) == 1
    with pytest.raises(O.RuleError):
        O.attn_tp_size(8, 3)


def test_dp_attention_removes_kv_duplication_for_few_kv_heads():
    # one KV "head" (the latent head of an MLA-style model): plain TP keeps a
    # full copy of every sequence's KV on each rank, DP attention splits the
    # sequences instead
    B, d, L, t = 64, 512, 1024, 8
    full = B * 1 * L * d * 2 * 2
    assert O.kv_bytes_per_rank(B, 1, d, L, t) == full
    assert O.kv_bytes_per_rank(B, 1, d, L, t, attn_dp=8) == full // 8
    # 8 KV heads at TP <= 8: nothing is duplicated, so DP attention buys nothing
    per_rank_tp = O.kv_bytes_per_rank(B, 8, 128, L, 8)
    assert per_rank_tp * 8 == B * 8 * L * 128 * 2 * 2
    assert O.kv_bytes_per_rank(B, 8, 128, L, 8, attn_dp=2) == per_rank_tp


def test_dp_gather_counts():
    assert O.dp_gather_received_per_rank([16, 16], 4096) == [16 * 4096 * 2] * 2
    assert O.dp_gather_received_per_rank([3, 5, 0], 64) == [5 * 128, 3 * 128, 8 * 128]


@pytest.mark.parametrize("n_heads,n_kv,t,attn_dp", [(4, 2, 4, 2), (4, 1, 4, 4), (8, 2, 8, 2),
                                                     (8, 8, 8, 4), (4, 4, 2, 2)])
@pytest.mark.parametrize("mode", ["decode", "prefill"])
@pytest.mark.parametrize("bias", [False, True])
def test_dp_attention_layer_equals_unsharded(n_heads, n_kv, t, attn_dp, mode, bias):
    dims, W = _tiny(n_heads, n_kv)
    if bias:
        W = _with_biases(dims, W)
    batch = O.Batch.decode(5, 7) if mode == "decode" else O.Batch.prefill(3, 5)
    n_seqs = 5 if mode == "decode" else 3
    L = 7 if mode == "decode" else 5
    T = len(batch.seq)
    h = synth.normal_f64(9, 19, (T, dims.hidden), 1.0)
    kc, vc = _caches(n_seqs, n_kv, L, dims.head_dim)
    pa = O.plan(n_heads, n_kv, dims.intermediate, dims.vocab, O.attn_tp_size(t, attn_dp))
    for rb, tol in ((O.no_round, 1e-12), (O.round_bf16, 1e-2)):
        k1, v1 = _copy(kc), _copy(vc)
        ref = O.layer_forward(h, W, k1, v1, batch, dims, rb=rb)
        k2, v2 = _copy(kc), _copy(vc)
        got = O.dp_attention_layer_forward(h, W, O.split_cache_copies(k2, dims, pa),
                                           O.split_cache_copies(v2, dims, pa), batch, dims, t,
                                           attn_dp, rb=rb)
        assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= tol, (rb, attn_dp)
        for b in k1:
            assert np.allclose(k1[b], k2[b], rtol=tol, atol=tol)
