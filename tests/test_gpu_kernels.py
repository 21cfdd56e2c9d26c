"""Kernel-level parity of the CUDA path against the oracle, through the C ABI.

Sizes span several tiles and ragged tails, both GEMM orientations (decode:
tokens <= 64 on the MMA N side; prefill: tokens on the M side), t = 1..8, and
padded vocabularies.  Lookup and logits placement are checked bit for bit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle as O  # noqa: E402
import synth  # noqa: E402
from megatron_tensor_layers_tp_gb300 import binding as B  # noqa: E402
from megatron_tensor_layers_tp_gb300.runtime import TPModel, make_config  # noqa: E402
from tests.parity_utils import device_layer, oracle_layer, rel_err, to_f64  # noqa: E402

TOL = 2e-2


def _wl(hidden=512, n_heads=8, n_kv=2, head_dim=64, inter=1536, vocab=1001, seed=3, norm_sigma=0.1):
    return synth.Workload("unit", hidden, n_heads, n_kv, head_dim, inter, vocab, 1, (1,), "decode",
                          4, 1, 8, True, seed=seed, norm_weight_sigma=norm_sigma)


def _model(w, t, head=True, prefill_cta_pairs=0):
    cfg = make_config(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab, 1, t,
                      max_positions=4096, plain_column_shards=1, prefill_cta_pairs=prefill_cta_pairs)
    layers = [device_layer(w, 0)]
    emb = lm = fn = None
    if head:
        emb = torch.empty((w.vocab, w.hidden), dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_(emb, w.seed, synth.tensor_id("embed"), 0.02)
        lm = torch.empty((w.vocab, w.hidden), dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_(lm, w.seed, synth.tensor_id("lm_head"), 0.02)
        fn = torch.ones(w.hidden, dtype=torch.bfloat16, device="cuda")
    m = TPModel(cfg, layers, emb, fn, lm, max_tokens=64)
    return m, emb, lm


def _x(M, K, seed=7, sigma=1.0):
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(x, seed, synth.tensor_id("x", M * 131 + K), sigma)
    return x


def test_device_generator_matches_host():
    t = torch.empty(100_003, dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(t, 5, 77, 0.02, start=12345)
    host = synth.normal_bf16_bits(5, 77, 100_003, 0.02, start=12345)
    assert np.array_equal(t.view(torch.int16).cpu().numpy().view(np.uint16), host)
    ids = torch.empty(5000, dtype=torch.int32, device="cuda")
    synth.fill_uniform_(ids, 5, 78, 1001)
    assert np.array_equal(ids.cpu().numpy(), synth.uniform_i32(5, 78, 5000, 1001))


@pytest.mark.parametrize("t", [1, 2, 4, 8])
def test_vocab_embedding_is_bit_exact(t):
    w = _wl()
    m, emb, _ = _model(w, t)
    ids_np = np.concatenate([synth.uniform_i32(1, 2, 300, w.vocab), [0, w.vocab - 1, 500, 999, 1000]])
    ids = torch.from_numpy(ids_np.astype(np.int32)).cuda()
    h = m.vocab_embed(ids)
    ref = emb[ids.long()]
    assert torch.equal(h.view(torch.int16), ref.view(torch.int16))
    # the oracle's masked lookup + rank-ordered sum gives the same bits
    E = to_f64(emb)
    p = O.plan(w.n_heads, w.n_kv_heads, w.intermediate, w.vocab, t)
    oref = O.sharded_embed(O.shard_vocab(E, p), ids_np, p)
    assert np.array_equal(to_f64(h), oref)
    assert m.check_device() == 0
    m.close()


def test_vocab_embedding_flags_out_of_range_ids():
    w = _wl()
    m, _, _ = _model(w, 2)
    ids = torch.tensor([3, w.vocab, 5, -1], dtype=torch.int32, device="cuda")
    h = m.vocab_embed(ids)
    assert m.check_device() == B.STATUS["TP_ERR_TOKEN_RANGE"]
    assert m.check_device() == 0          # cleared by the first read
    assert torch.count_nonzero(h[1].float()) == 0 and torch.count_nonzero(h[3].float()) == 0
    m.close()


@pytest.mark.parametrize("t", [1, 2, 4, 8])
@pytest.mark.parametrize("S", [1, 13, 64, 80])
def test_lm_head_placement_is_bit_exact(t, S):
    # W_lm[v] = c(v) e_0 with c(v) exactly representable; x = e_0  =>  logits[v] == c(v)
    w = _wl()
    V, H = w.vocab, w.hidden
    cv = ((np.arange(V) % 251) - 125) / 64.0
    lm = torch.zeros((V, H), dtype=torch.bfloat16, device="cuda")
    lm[:, 0] = torch.from_numpy(cv).to(torch.bfloat16).cuda()
    cfg = make_config(H, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, V, 1, t, max_positions=64)
    emb = torch.zeros((V, H), dtype=torch.bfloat16, device="cuda")
    m = TPModel(cfg, [device_layer(w, 0)], emb, torch.ones(H, dtype=torch.bfloat16, device="cuda"),
                lm, max_tokens=S)
    x = torch.zeros((S, H), dtype=torch.bfloat16, device="cuda")
    x[:, 0] = torch.arange(1, S + 1, dtype=torch.float32).cuda().to(torch.bfloat16) / 8
    logits = m.lm_head_gather(x)
    ref = (torch.arange(1, S + 1, dtype=torch.float64)[:, None] / 8) * torch.from_numpy(cv)[None, :]
    got = logits.double().cpu()
    assert torch.equal(got, ref.to(torch.bfloat16).double())
    m.close()


@pytest.mark.parametrize("t", [1, 2, 4])
def test_lm_head_matches_oracle(t):
    w = _wl()
    m, _, lm = _model(w, t)
    x = _x(37, w.hidden, seed=9)
    logits = m.lm_head_gather(x)
    p = O.plan(w.n_heads, w.n_kv_heads, w.intermediate, w.vocab, t)
    ref = O.sharded_lm_head(to_f64(x), O.shard_vocab(to_f64(lm), p), w.vocab)
    assert rel_err(to_f64(logits), ref) <= TOL
    m.close()


@pytest.mark.parametrize("head_dim,n_heads,n_kv", [(64, 8, 2), (128, 8, 4), (64, 8, 1)])
@pytest.mark.parametrize("t", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [1, 13, 64, 200])
def test_column_linear_matches_oracle_shards(head_dim, n_heads, n_kv, t, M):
    w = _wl(hidden=512, n_heads=n_heads, n_kv=n_kv, head_dim=head_dim, inter=1536 if t != 8 else 2048)
    if n_heads % t or (n_heads // t) * head_dim % 64:
        pytest.skip("shape outside the rule set")
    m, _, _ = _model(w, t, head=False)
    x = _x(M, w.hidden)
    W = oracle_layer(w, 0)
    dims = O.Dims(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab)
    p = O.plan(w.n_heads, w.n_kv_heads, w.intermediate, w.vocab, t)
    xf = to_f64(x)
    y = m.column_linear(0, B.TP_QKV, x)
    for r, sh in enumerate(O.shard_qkv(W, dims, p)):
        assert rel_err(to_f64(y[r]), O.linear(xf, sh)) <= TOL, ("qkv", r)
    y = m.column_linear(0, B.TP_GATE_UP, x)
    for r, sh in enumerate(O.shard_gate_up(W, p)):
        assert rel_err(to_f64(y[r]), O.linear(xf, sh)) <= TOL, ("gate_up", r)
    assert m.check_device() == 0
    m.close()


@pytest.mark.parametrize("t", [1, 2, 4, 8])
@pytest.mark.parametrize("M", [1, 16, 61, 64, 130, 300])
@pytest.mark.parametrize("fused", [True, False])
def test_row_linear_reduce_matches_oracle(t, M, fused):
    w = _wl(hidden=512, n_heads=8, n_kv=2, head_dim=64, inter=2048)
    m, _, _ = _model(w, t, head=False)
    W = oracle_layer(w, 0)
    for which, Wfull in ((B.TP_O, W.wo), (B.TP_DOWN, W.wd)):
        K = Wfull.shape[1]
        x = _x(M, K, seed=11)
        res = _x(M, w.hidden, seed=12)
        y = m.row_linear_reduce(0, which, x, residual=res, fused=fused)
        xf = to_f64(x)
        partials = [O.linear(xs, Ws) for xs, Ws in zip(O.shard_rows_by_input(xf, t),
                                                        O.shard_rows_by_input(Wfull, t))]
        ref = O.round_bf16(to_f64(res) + O.all_reduce_sum(partials))
        assert rel_err(to_f64(y), ref) <= TOL, (which, fused)
        if t > 1:
            # the debugging checklist: a single rank's partial is not the reduced result
            part0 = O.round_bf16(to_f64(res) + partials[0])
            assert rel_err(to_f64(y), part0) > 5 * TOL
        # without residual
        y2 = m.row_linear_reduce(0, which, x, residual=None, fused=fused)
        assert rel_err(to_f64(y2), O.round_bf16(O.all_reduce_sum(partials))) <= TOL
    assert m.check_device() == 0
    m.close()


def test_fused_and_unfused_reductions_agree_and_are_deterministic():
    w = _wl(hidden=1024, n_heads=8, n_kv=2, head_dim=128, inter=4096)
    m, _, _ = _model(w, 4, head=False)
    for M in (16, 256):
        x = _x(M, 4096, seed=21)
        a = m.row_linear_reduce(0, B.TP_DOWN, x, fused=True)
        b = m.row_linear_reduce(0, B.TP_DOWN, x, fused=True)
        c = m.row_linear_reduce(0, B.TP_DOWN, x, fused=False)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert rel_err(to_f64(a), to_f64(c)) <= 1e-2
    m.close()


@pytest.mark.parametrize("M", [1, 7, 64, 300])
def test_rmsnorm_matches_oracle(M):
    w = _wl(hidden=4096)
    m, _, _ = _model(_wl(), 1, head=False)
    x = _x(M, 512, seed=31, sigma=3.0)
    g = torch.empty(512, dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(g, 1, 99, 0.5)
    y = m.rmsnorm(x, g)
    ref = O.round_bf16(O.rmsnorm(to_f64(x), to_f64(g), 1e-5))
    assert rel_err(to_f64(y), ref) <= TOL
    m.close()


def test_zero_tokens_are_a_no_op():
    w = _wl()
    m, _, _ = _model(w, 2)
    ws, nws = m.ws_args
    assert B.tp_column_linear(m.handle, 0, B.TP_QKV, 0, 0, 0, 0, ws, nws, 0) == 0
    assert B.tp_vocab_embed(m.handle, 0, 0, 0, 0) == 0
    assert B.tp_column_linear(m.handle, 5, B.TP_QKV, 0, 4, 0, 0, ws, nws, 0) == B.STATUS["TP_ERR_ARG"]
    x = _x(16, w.hidden)
    y = torch.empty((2, 16, m.qkv_rows()), dtype=torch.bfloat16, device="cuda")
    assert B.tp_column_linear(m.handle, 0, B.TP_QKV, x.data_ptr(), 16, y.data_ptr(), 16 * m.qkv_rows(),
                              ws, 16, 0) == B.STATUS["TP_ERR_WORKSPACE"]
    m.close()


@pytest.mark.parametrize("M,inter,t", [(1024, 2432, 1), (2048, 2432, 1), (1100, 1536, 2)])
def test_prefill_orientation_schedules_match_oracle(M, inter, t):
    # M=1024, I=2432, t=1: 8 x 19 = 152 gate_up tiles = one whole data-parallel
    # wave on 152 SMs (empty stream-K part); M=2048: two waves; M=1100: a
    # ragged last token tile and a stream-K remainder
    w = _wl(hidden=512, n_heads=8, n_kv=2, head_dim=64, inter=inter)
    m, _, _ = _model(w, t, head=False)
    x = _x(M, w.hidden, seed=41)
    W = oracle_layer(w, 0)
    p = O.plan(w.n_heads, w.n_kv_heads, w.intermediate, w.vocab, t)
    xf = to_f64(x)
    y = m.column_linear(0, B.TP_GATE_UP, x)
    for r, sh in enumerate(O.shard_gate_up(W, p)):
        assert rel_err(to_f64(y[r]), O.linear(xf, sh)) <= TOL
    a = _x(M, inter, seed=42)
    res = _x(M, w.hidden, seed=43)
    out = m.row_linear_reduce(0, B.TP_DOWN, a, residual=res, fused=True)
    ref = O.round_bf16(to_f64(res) + O.linear(to_f64(a), W.wd))
    assert rel_err(to_f64(out), ref) <= TOL
    assert m.check_device() == 0
    m.close()


@pytest.mark.parametrize("t", [1, 2, 4])
@pytest.mark.parametrize("M", [65, 200, 300, 1100])
def test_cta_pair_gemms_match_oracle(t, M):
    # every GEMM above 64 tokens on CTA pairs (256-row tiles; M=65 and 200 a
    # single ragged pair tile whose odd CTA holds no or few tokens, 1100 five
    # tiles), each epilogue of the prefill orientation against the oracle,
    # and against the single-CTA kernel
    w = _wl(hidden=512, n_heads=8, n_kv=2, head_dim=64, inter=1536)
    mp, _, lm = _model(w, t, prefill_cta_pairs=1)
    ms, _, _ = _model(w, t, prefill_cta_pairs=2)
    W = oracle_layer(w, 0)
    dims = O.Dims(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab)
    p = O.plan(w.n_heads, w.n_kv_heads, w.intermediate, w.vocab, t)
    x = _x(M, w.hidden, seed=51)
    xf = to_f64(x)
    for which, shards in ((B.TP_QKV, O.shard_qkv(W, dims, p)), (B.TP_GATE_UP, O.shard_gate_up(W, p))):
        y = mp.column_linear(0, which, x)
        ys = ms.column_linear(0, which, x)
        for r, sh in enumerate(shards):
            ref = O.linear(xf, sh)
            assert rel_err(to_f64(y[r]), ref) <= TOL, (which, r)
            assert rel_err(to_f64(y[r]), to_f64(ys[r])) <= TOL, (which, r)
    for which, Wfull in ((B.TP_O, W.wo), (B.TP_DOWN, W.wd)):
        K = Wfull.shape[1]
        a = _x(M, K, seed=52)
        res = _x(M, w.hidden, seed=53)
        partials = [O.linear(xs, Ws) for xs, Ws in zip(O.shard_rows_by_input(to_f64(a), t),
                                                        O.shard_rows_by_input(Wfull, t))]
        ref = O.round_bf16(to_f64(res) + O.all_reduce_sum(partials))
        for fused in (True, False):
            y = mp.row_linear_reduce(0, which, a, residual=res, fused=fused)
            assert rel_err(to_f64(y), ref) <= TOL, (which, fused)
    logits = mp.lm_head_gather(x)
    ref = O.sharded_lm_head(xf, O.shard_vocab(to_f64(lm), p), w.vocab)
    assert rel_err(to_f64(logits), ref) <= TOL
    assert mp.check_device() == 0 and ms.check_device() == 0
    mp.close()
    ms.close()


def test_cta_pair_config_values():
    w = _wl()
    for mode in (0, 1, 2):
        m, _, _ = _model(w, 2, head=False, prefill_cta_pairs=mode)
        m.close()


@pytest.mark.parametrize("t", [1, 2, 8])
@pytest.mark.parametrize("M", [1, 16, 64])
@pytest.mark.parametrize("hidden,n_heads", [(4096, 32), (5120, 40)])
def test_decode_cluster_split_matches_oracle(t, M, hidden, n_heads):
    # hidden 4096: 32 row-parallel output tiles (clusters of 4) and 48 qkv
    # tiles; hidden 5120: 40 row-parallel tiles (clusters of 3) and 56 qkv
    # tiles (clusters of 2) -- above 16 tokens the decode schedule splits
    # them over clusters of CTAs whose K pieces are summed on chip; up to 16
    # tokens it runs stream-K over every SM
    w = _wl(hidden=hidden, n_heads=n_heads, n_kv=8, head_dim=128, inter=2048)
    m, _, _ = _model(w, t, head=False)
    W = oracle_layer(w, 0)
    x = _x(M, w.hidden, seed=51)
    dims = O.Dims(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab)
    p = O.plan(w.n_heads, w.n_kv_heads, w.intermediate, w.vocab, t)
    y = m.column_linear(0, B.TP_QKV, x)
    for r, sh in enumerate(O.shard_qkv(W, dims, p)):
        assert rel_err(to_f64(y[r]), O.linear(to_f64(x), sh)) <= TOL, r
    for which, Wfull in ((B.TP_O, W.wo), (B.TP_DOWN, W.wd)):
        a = _x(M, Wfull.shape[1], seed=52)
        res = _x(M, w.hidden, seed=53)
        out = m.row_linear_reduce(0, which, a, residual=res, fused=True)
        ref = O.round_bf16(to_f64(res) + O.linear(to_f64(a), Wfull))
        assert rel_err(to_f64(out), ref) <= TOL, which
        again = m.row_linear_reduce(0, which, a, residual=res, fused=True)
        assert torch.equal(out.view(torch.int16), again.view(torch.int16))
    assert m.check_device() == 0
    m.close()
