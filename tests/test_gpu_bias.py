"""Projection biases on the CUDA path ("第 9 章 多进程与张量并行", §3.2 切分:
a weight and its bias are cut along the output dimension; the bias of a
row-parallel output is added once, after the reduction), against the oracle:
decode and prefill layers with and without KV replication, both reduction
variants, the column- and row-parallel calls on their own, and sharded vs
unsharded on the GPU."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle as O  # noqa: E402
import synth  # noqa: E402
from megatron_tensor_layers_tp_gb300 import binding as B  # noqa: E402
from tests.parity_utils import (build_model, make_batch, oracle_batch, oracle_caches,  # noqa: E402
                                oracle_dims, oracle_layer, rel_err, to_f64)

LAYER_TOL = 2e-2
TOL = 2e-2


def _wl(mode, n_seqs, seq_len, ctx, hidden=512, n_heads=8, n_kv=2, head_dim=64, inter=1536):
    return synth.Workload(f"unit-bias-{mode}", hidden, n_heads, n_kv, head_dim, inter, 1001, 1,
                          (1,), mode, n_seqs, seq_len, ctx, False, seed=6, norm_weight_sigma=0.1,
                          bias=True, sigma_b=0.5)


def _layer(w, t, fused=True, pairs=0):
    model, _, _ = build_model(w, t, prefill_cta_pairs=pairs)
    batch, caches = make_batch(model, w)
    h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(h, w.seed, synth.tensor_id("hidden"), w.sigma_h)
    model.layer_forward(0, batch, h, fused=fused)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    return model, h


def _oracle(w):
    kc, vc = oracle_caches(w, 0, range(w.n_seqs))
    return O.layer_forward(synth.host_hidden(w), oracle_layer(w, 0), kc, vc, oracle_batch(w),
                           oracle_dims(w))


@pytest.mark.parametrize("t", [1, 2, 4, 8])
@pytest.mark.parametrize("n_kv", [8, 2])
@pytest.mark.parametrize("fused", [True, False])
def test_decode_layer_with_biases_matches_oracle(t, n_kv, fused):
    w = _wl("decode", n_seqs=5, seq_len=1, ctx=150, n_kv=n_kv)
    model, h = _layer(w, t, fused)
    ref = _oracle(w)
    assert rel_err(to_f64(h), ref) <= LAYER_TOL
    # the biases are large enough that dropping one would fail the check
    wb = _wl("decode", n_seqs=5, seq_len=1, ctx=150, n_kv=n_kv)
    W0 = oracle_layer(wb, 0)
    W0.bo = None
    kc, vc = oracle_caches(wb, 0, range(wb.n_seqs))
    nob = O.layer_forward(synth.host_hidden(wb), W0, kc, vc, oracle_batch(wb), oracle_dims(wb))
    assert rel_err(nob, ref) > 5 * LAYER_TOL
    model.close()


@pytest.mark.parametrize("t", [1, 4])
@pytest.mark.parametrize("pairs", [0, 1, 2])
def test_prefill_layer_with_biases_matches_oracle(t, pairs):
    # pairs: 0 chosen per GEMM (single CTAs at this size), 1 CTA pairs, 2 single CTAs
    w = _wl("prefill", n_seqs=3, seq_len=70, ctx=70)
    model, h = _layer(w, t, pairs=pairs)
    assert rel_err(to_f64(h), _oracle(w)) <= LAYER_TOL
    model.close()


def test_biased_sharded_equals_unsharded_on_gpu():
    w = _wl("decode", n_seqs=16, seq_len=1, ctx=300, hidden=1024, n_heads=16, n_kv=8,
            inter=2048)
    outs = {}
    for t in (1, 2, 4, 8):
        model, h = _layer(w, t)
        outs[t] = to_f64(h)
        model.close()
    for t in (2, 4, 8):
        assert rel_err(outs[t], outs[1]) <= 1e-2, t


@pytest.mark.parametrize("t", [2, 4])
@pytest.mark.parametrize("M,pairs", [(16, 0), (200, 0), (200, 1), (600, 1)])
def test_column_and_row_calls_carry_their_biases(t, M, pairs):
    w = _wl("decode", n_seqs=4, seq_len=1, ctx=8)
    model, _, _ = build_model(w, t, max_tokens=M, plain_column_shards=1, prefill_cta_pairs=pairs)
    W = oracle_layer(w, 0)
    dims = oracle_dims(w)
    p = O.plan(w.n_heads, w.n_kv_heads, w.intermediate, w.vocab, t)
    x = torch.empty((M, w.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(x, 8, synth.tensor_id("x", M), 1.0)
    xf = to_f64(x)
    y = model.column_linear(0, B.TP_QKV, x)
    for r, (sh, b) in enumerate(zip(O.shard_qkv(W, dims, p), O.shard_qkv_bias(W, dims, p))):
        assert rel_err(to_f64(y[r]), O.linear(xf, sh, b)) <= TOL, r
    y = model.column_linear(0, B.TP_GATE_UP, x)
    for r, (sh, b) in enumerate(zip(O.shard_gate_up(W, p), O.shard_gate_up_bias(W, p))):
        assert rel_err(to_f64(y[r]), O.linear(xf, sh, b)) <= TOL, r
    a = torch.empty((M, w.intermediate), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(a, 8, synth.tensor_id("x", M + 1), 1.0)
    res = torch.empty((M, w.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(res, 8, synth.tensor_id("x", M + 2), 1.0)
    ref = O.round_bf16(to_f64(res) + O.linear(to_f64(a), W.wd, W.bd))
    for fused in (True, False):
        out = model.row_linear_reduce(0, B.TP_DOWN, a, residual=res, fused=fused)
        assert rel_err(to_f64(out), ref) <= TOL, fused
    # bias added once: t-fold would miss by (t - 1) * bd
    bad = O.round_bf16(to_f64(res) + O.linear(to_f64(a), W.wd) + t * W.bd)
    assert rel_err(bad, ref) > 5 * TOL
    assert model.check_device() == 0
    model.close()
