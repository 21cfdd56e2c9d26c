"""Pins of the oracle's whole decoder layer and whole forward against
evaluations that share none of its code.

- A one-token layer small enough to work out by hand, with every projection
  and both norm weights non-trivial, so the MLP half is exercised: which h the
  MLP norm reads, SiLU on the gate (not on up), down_proj on SiLU(gate) * up,
  and the residual that the MLP output is added to.
- A scalar-loop evaluation written straight from the definitions the pages
  use (embedding lookup, pre-norm RMSNorm, Y = X W^T, rotate-half RoPE, GQA
  softmax attention, SiLU(gate) * up, final norm, LM head), with plain Python
  floats and the math module only: no numpy arithmetic and no oracle
  function.  It runs config 1 (H256, 4 Q / 2 KV heads, 16 prefill tokens,
  embedding + layer + LM head) and a small decode case over a cache with
  biases and non-unit norm weights, and must agree with ``O.forward`` to
  1e-12 with the storage rounding switched off.

Pages: "张量、流水线与数据并行", §线性层怎么切 (the flowchart: qkv_proj ->
attention -> o_proj -> all-reduce ① -> gate_up -> SiLU x up -> down_proj ->
all-reduce ② -> next layer), §词嵌入 / §输出层; "第 9 章 多进程与张量并行", §3.2
切分 (the sharded computation must reconstruct the original model's math).
"""
import math

import numpy as np
import pytest

import oracle as O
import synth


# ---------------------------------------------------------------------------
# a layer worked out by hand
# ---------------------------------------------------------------------------
def _hand_layer():
    # H = 2, one head of width 2 (one RoPE pair), one KV head, I = 1; the token
    # sits at position 0 (RoPE is the identity there) and attends to itself
    # alone, so the attention output is its own v.
    dims = O.Dims(hidden=2, n_heads=1, n_kv_heads=1, head_dim=2, intermediate=1, vocab=4,
                  rms_eps=0.0)
    W = O.LayerWeights(
        attn_norm=np.array([2.0, 1.0]),
        wq=np.array([[0.3, -0.7], [1.1, 0.2]]),
        wk=np.array([[-0.4, 0.9], [0.5, 0.6]]),
        wv=np.eye(2),
        wo=np.array([[1.0, 0.0], [0.0, 3.0]]),
        mlp_norm=np.array([1.0, 3.0]),
        wg=np.array([[1.0, 0.0]]),
        wu=np.array([[0.0, -1.0]]),
        wd=np.array([[1.0], [2.0]]))
    return dims, W


def test_layer_with_nonzero_mlp_matches_hand_computation():
    dims, W = _hand_layer()
    h = np.array([[1.0, -1.0]])
    kc = {0: np.zeros((1, 1, 2))}
    vc = {0: np.zeros((1, 1, 2))}
    got = O.layer_forward(h, W, kc, vc, O.Batch.decode(1, 1), dims, rb=O.no_round)
    # attention block: mean square of h is 1, so u = h * attn_norm = (2, -1);
    # v = u; o_proj: (2*1, -1*3) = (2, -3); h1 = h + (2, -3) = (3, -4)
    # MLP block: mean square of h1 is 12.5, u2 = h1 / sqrt(12.5) * (1, 3);
    # gate = u2[0] = 3r, up = -u2[1] = 12r with r = 1 / sqrt(12.5)
    r = 1.0 / math.sqrt(12.5)
    gate, up = 3.0 * r, 12.0 * r
    a = gate / (1.0 + math.exp(-gate)) * up
    want = np.array([3.0 + a, -4.0 + 2.0 * a])
    assert np.allclose(got[0], want, rtol=1e-14, atol=1e-14)
    # the cache slot of position 0 holds the token's k and v
    assert np.allclose(vc[0][0, 0], [2.0, -1.0], rtol=0, atol=1e-15)
    assert np.allclose(kc[0][0, 0], W.wk @ np.array([2.0, -1.0]), rtol=0, atol=1e-15)


def test_hand_layer_rejects_plausible_mistakes():
    # each plausible slip in the MLP half gives a value the test above rejects
    r = 1.0 / math.sqrt(12.5)
    silu = lambda x: x / (1.0 + math.exp(-x))
    right = np.array([3.0 + silu(3 * r) * 12 * r, -4.0 + 2 * silu(3 * r) * 12 * r])
    wrong = {
        # the MLP norm reads the pre-attention h = (1, -1)
        "mlp_norm_on_old_h": np.array([3.0 + silu(1.0) * 3.0, -4.0 + 2 * silu(1.0) * 3.0]),
        # SiLU applied to up instead of the gate
        "silu_on_up": np.array([3.0 + silu(12 * r) * 3 * r, -4.0 + 2 * silu(12 * r) * 3 * r]),
        # the residual stream skips the MLP
        "mlp_dropped": np.array([3.0, -4.0]),
        # the MLP output added to the pre-attention h
        "mlp_on_old_residual": np.array([1.0 + silu(3 * r) * 12 * r, -1.0 + 2 * silu(3 * r) * 12 * r]),
    }
    for name, v in wrong.items():
        assert not np.allclose(v, right, rtol=1e-6), name


# ---------------------------------------------------------------------------
# scalar-loop evaluation from the definitions
# ---------------------------------------------------------------------------
def _dot(a, b):
    s = 0.0
    for x, y in zip(a, b):
        s += x * y
    return s


def _rmsnorm(x, w, eps):
    ms = 0.0
    for v in x:
        ms += v * v
    r = 1.0 / math.sqrt(ms / len(x) + eps)
    return [x[i] * r * w[i] for i in range(len(x))]


def _rope_head(vec, pos, theta):
    d = len(vec)
    half = d // 2
    out = [0.0] * d
    for i in range(half):
        ang = pos * theta ** (-(2.0 * i) / d)
        c, s = math.cos(ang), math.sin(ang)
        x1, x2 = vec[i], vec[i + half]
        out[i] = x1 * c - x2 * s
        out[i + half] = x2 * c + x1 * s
    return out


def _proj(u, rows, bias):
    return [_dot(u, rows[o]) + (bias[o] if bias is not None else 0.0) for o in range(len(rows))]


def _bruteforce_forward(ids, E, layers, final_norm, lm, seqs, poss, dims, sample_rows):
    """Token m of sequence seqs[m] at position poss[m]; layers: list of
    (weights as nested lists, per-sequence cache dict {b: [n_kv][L][d] lists})."""
    H, nh, nkv, d = dims.hidden, dims.n_heads, dims.n_kv_heads, dims.head_dim
    group = nh // nkv
    T = len(ids)
    h = [list(E[i]) for i in ids]
    for Wl, kc, vc in layers:
        # attention block
        qs = []
        for m in range(T):
            u = _rmsnorm(h[m], Wl["attn_norm"], dims.rms_eps)
            q = _proj(u, Wl["wq"], Wl.get("bq"))
            k = _proj(u, Wl["wk"], Wl.get("bk"))
            v = _proj(u, Wl["wv"], Wl.get("bv"))
            p = poss[m]
            q = sum((_rope_head(q[j * d:(j + 1) * d], p, dims.rope_theta) for j in range(nh)), [])
            k = sum((_rope_head(k[g * d:(g + 1) * d], p, dims.rope_theta) for g in range(nkv)), [])
            b = seqs[m]
            for g in range(nkv):
                kc[b][g][p] = k[g * d:(g + 1) * d]
                vc[b][g][p] = v[g * d:(g + 1) * d]
            qs.append(q)
        h_new = []
        for m in range(T):
            b, p = seqs[m], poss[m]
            o = []
            for j in range(nh):
                g = j // group
                qj = qs[m][j * d:(j + 1) * d]
                sc = [_dot(qj, kc[b][g][s]) / math.sqrt(d) for s in range(p + 1)]
                mx = max(sc)
                ex = [math.exp(x - mx) for x in sc]
                den = sum(ex)
                for f in range(d):
                    acc = 0.0
                    for s in range(p + 1):
                        acc += ex[s] / den * vc[b][g][s][f]
                    o.append(acc)
            y = _proj(o, Wl["wo"], Wl.get("bo"))
            h_new.append([h[m][i] + y[i] for i in range(H)])
        h = h_new
        # MLP block
        h_new = []
        for m in range(T):
            u2 = _rmsnorm(h[m], Wl["mlp_norm"], dims.rms_eps)
            gate = _proj(u2, Wl["wg"], Wl.get("bg"))
            up = _proj(u2, Wl["wu"], Wl.get("bu"))
            a = [gate[i] / (1.0 + math.exp(-gate[i])) * up[i] for i in range(len(gate))]
            y = _proj(a, Wl["wd"], Wl.get("bd"))
            h_new.append([h[m][i] + y[i] for i in range(H)])
        h = h_new
    out = []
    for m in sample_rows:
        x = _rmsnorm(h[m], final_norm, dims.rms_eps)
        out.append([_dot(x, row) for row in lm])
    return np.array(out)


def _as_lists(W: O.LayerWeights):
    out = {}
    for k, v in W.__dict__.items():
        if v is not None:
            out[k] = v.tolist()
    return out


def _cache_lists(c):
    return {b: a.tolist() for b, a in c.items()}


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / (np.max(np.abs(b)) + 1e-300))


def test_bruteforce_config1_forward_equals_oracle():
    w = synth.WORKLOADS["tiny"]
    dims = O.Dims(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab,
                  w.rms_eps, w.rope_theta)
    shapes = synth.weight_shapes(w, 0)
    W = O.LayerWeights(**{k: synth.host_weight(w, k, 0, shapes[k]) for k in shapes})
    E = synth.host_weight(w, "embed", 0, (w.vocab, w.hidden))
    lm = synth.host_weight(w, "lm_head", 0, (w.vocab, w.hidden))
    fn = synth.host_weight(w, "final_norm", 0, (w.hidden,))
    ids = synth.token_ids(w)
    batch = O.Batch.prefill(w.n_seqs, w.seq_len)
    kc = {b: synth.host_kv(w, "k_cache", 0, b) for b in range(w.n_seqs)}
    vc = {b: synth.host_kv(w, "v_cache", 0, b) for b in range(w.n_seqs)}
    rows = batch.sample_rows()
    got = O.forward(ids, E, [(W, {b: a.copy() for b, a in kc.items()},
                              {b: a.copy() for b, a in vc.items()})],
                    fn, lm, batch, dims, rb=O.no_round)
    ref = _bruteforce_forward(ids.tolist(), E.tolist(), [(_as_lists(W), _cache_lists(kc),
                                                          _cache_lists(vc))],
                              fn.tolist(), lm.tolist(), batch.seq.tolist(), batch.pos.tolist(),
                              dims, rows.tolist())
    assert got.shape == (1, w.vocab)
    assert _rel(got, ref) <= 1e-12


def test_bruteforce_decode_over_cache_with_biases_equals_oracle():
    # two layers, 3 sequences decoding at context 5 (4 cached positions and
    # the new token), 4 Q heads over 2 KV heads, biases on every projection,
    # non-unit norm weights
    H, nh, nkv, d, I, V = 32, 4, 2, 8, 48, 40
    dims = O.Dims(H, nh, nkv, d, I, V, 1e-5, 10000.0)
    rng_seed = 77
    layers_o, layers_b = [], []
    for l in range(2):
        s = rng_seed + 20 * l
        W = O.LayerWeights(
            attn_norm=1.0 + synth.normal_f64(s, 1, (H,), 0.2),
            wq=synth.normal_f64(s, 2, (nh * d, H), 0.2),
            wk=synth.normal_f64(s, 3, (nkv * d, H), 0.2),
            wv=synth.normal_f64(s, 4, (nkv * d, H), 0.2),
            wo=synth.normal_f64(s, 5, (H, nh * d), 0.2),
            mlp_norm=1.0 + synth.normal_f64(s, 6, (H,), 0.2),
            wg=synth.normal_f64(s, 7, (I, H), 0.2),
            wu=synth.normal_f64(s, 8, (I, H), 0.2),
            wd=synth.normal_f64(s, 9, (H, I), 0.2),
            bq=synth.normal_f64(s, 10, (nh * d,), 0.3),
            bk=synth.normal_f64(s, 11, (nkv * d,), 0.3),
            bv=synth.normal_f64(s, 12, (nkv * d,), 0.3),
            bo=synth.normal_f64(s, 13, (H,), 0.3),
            bg=synth.normal_f64(s, 14, (I,), 0.3),
            bu=synth.normal_f64(s, 15, (I,), 0.3),
            bd=synth.normal_f64(s, 16, (H,), 0.3))
        kc = {b: synth.normal_f64(s, 30 + b, (nkv, 5, d), 1.0) for b in range(3)}
        vc = {b: synth.normal_f64(s, 40 + b, (nkv, 5, d), 1.0) for b in range(3)}
        layers_o.append((W, {b: a.copy() for b, a in kc.items()}, {b: a.copy() for b, a in vc.items()}))
        layers_b.append((_as_lists(W), _cache_lists(kc), _cache_lists(vc)))
    E = synth.normal_f64(rng_seed, 90, (V, H), 1.0)
    lm = synth.normal_f64(rng_seed, 91, (V, H), 0.2)
    fn = 1.0 + synth.normal_f64(rng_seed, 92, (H,), 0.2)
    ids = np.array([3, 17, 39])
    batch = O.Batch.decode(3, 5)
    got = O.forward(ids, E, layers_o, fn, lm, batch, dims, rb=O.no_round)
    ref = _bruteforce_forward(ids.tolist(), E.tolist(), layers_b, fn.tolist(), lm.tolist(),
                              batch.seq.tolist(), batch.pos.tolist(), dims, [0, 1, 2])
    assert got.shape == (3, V)
    assert _rel(got, ref) <= 1e-12
    # and the cached positions take part: perturbing an old key changes the result
    layers_o2 = [(W, {b: a.copy() for b, a in kc.items()}, {b: a.copy() for b, a in vc.items()})
                 for W, kc, vc in layers_o]
    layers_o2[0][1][1][0, 2] += 1.0
    got2 = O.forward(ids, E, layers_o2, fn, lm, batch, dims, rb=O.no_round)
    assert _rel(got2[1], ref[1]) > 1e-6 and _rel(got2[0], ref[0]) <= 1e-12


def test_forward_composition_rejects_a_skipped_final_norm():
    # the final RMSNorm (non-unit weight) changes the logits: an evaluation that
    # skipped it would not meet the 1e-12 bar above
    w = synth.WORKLOADS["tiny"]
    dims = O.Dims(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab,
                  w.rms_eps, w.rope_theta)
    x = synth.normal_f64(5, 5, (1, w.hidden), 3.0)
    lm = synth.normal_f64(5, 6, (w.vocab, w.hidden), 0.02)
    fn = 1.0 + synth.normal_f64(5, 7, (w.hidden,), 0.2)
    with_norm = O.lm_head(x, fn, lm, dims, rb=O.no_round)
    without = O.linear(x, lm)
    assert _rel(without, with_norm) > 0.1
