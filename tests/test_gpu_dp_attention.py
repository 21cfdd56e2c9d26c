"""DP attention on the CUDA path ("张量、流水线与数据并行", SGLang 的 DP
attention): the attention block tensor-parallel over attn_tp = t / attn_dp
ranks of each DP group, the MLP over all t ranks.  Checked against the
oracle's DP-attention layer and its unsharded layer, against plain tensor
parallelism at the same t on the GPU, and through the gather counters."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle as O  # noqa: E402
import synth  # noqa: E402
from tests.parity_utils import (build_model, make_batch, oracle_batch, oracle_caches,  # noqa: E402
                                oracle_dims, oracle_layer, rel_err, to_f64)

LAYER_TOL = 2e-2


def _wl(mode, n_seqs, seq_len, ctx, n_heads=8, n_kv=2, layers=1, embed=False, bias=False):
    return synth.Workload(f"unit-dpattn-{mode}", 512, n_heads, n_kv, 64, 1536, 1001, layers, (1,),
                          mode, n_seqs, seq_len, ctx, embed, seed=8, norm_weight_sigma=0.1,
                          bias=bias)


def _run(w, t, attn_dp, fused=True, pairs=0):
    model, _, _ = build_model(w, t, attn_dp=attn_dp, prefill_cta_pairs=pairs)
    batch, caches = make_batch(model, w)
    h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(h, w.seed, synth.tensor_id("hidden"), w.sigma_h)
    model.reset_stats()
    model.layer_forward(0, batch, h, fused=fused)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    return model, h, caches


@pytest.mark.parametrize("t,attn_dp", [(4, 2), (8, 2), (8, 4), (8, 8)])
@pytest.mark.parametrize("n_kv", [8, 2, 1])
@pytest.mark.parametrize("fused", [True, False])
def test_decode_layer_with_dp_attention_matches_oracle(t, attn_dp, n_kv, fused):
    w = _wl("decode", n_seqs=8, seq_len=1, ctx=150, n_kv=n_kv)
    model, h, (ks, vs) = _run(w, t, attn_dp, fused)
    st = model.stats()
    assert st.dp_gathers == 1
    assert st.dp_gather_recv_bytes_per_rank == (attn_dp - 1) * w.tokens * w.hidden * 2 // attn_dp
    dims = oracle_dims(w)
    kc, vc = oracle_caches(w, 0, range(w.n_seqs))
    ref = O.layer_forward(synth.host_hidden(w), oracle_layer(w, 0), kc, vc, oracle_batch(w), dims)
    assert rel_err(to_f64(h), ref) <= LAYER_TOL
    # the DP-attention restatement agrees with the plain layer
    pa = O.plan(w.n_heads, w.n_kv_heads, w.intermediate, w.vocab, O.attn_tp_size(t, attn_dp))
    kc2, vc2 = oracle_caches(w, 0, range(w.n_seqs))
    ref2 = O.dp_attention_layer_forward(synth.host_hidden(w), oracle_layer(w, 0),
                                        O.split_cache_copies(kc2, dims, pa),
                                        O.split_cache_copies(vc2, dims, pa), oracle_batch(w),
                                        dims, t, attn_dp)
    assert rel_err(to_f64(h), ref2) <= LAYER_TOL
    # the new token's K landed at position ctx - 1 in the attention ranks' caches
    c = model.cfg
    gk = to_f64(ks[0])
    for b in range(w.n_seqs):
        got = gk[:, b].reshape(c.kv_copies * c.kv_heads_per_rank, w.ctx, w.head_dim)
        assert rel_err(got[:, w.ctx - 1], kc[b][:, w.ctx - 1]) <= LAYER_TOL
    model.close()


@pytest.mark.parametrize("t,attn_dp", [(4, 2), (8, 4)])
@pytest.mark.parametrize("pairs", [0, 1])
def test_prefill_layer_with_dp_attention_matches_oracle(t, attn_dp, pairs):
    w = _wl("prefill", n_seqs=4, seq_len=70, ctx=70, bias=True)
    model, h, _ = _run(w, t, attn_dp, pairs=pairs)
    kc, vc = oracle_caches(w, 0, range(w.n_seqs))
    ref = O.layer_forward(synth.host_hidden(w), oracle_layer(w, 0), kc, vc, oracle_batch(w),
                          oracle_dims(w))
    assert rel_err(to_f64(h), ref) <= LAYER_TOL
    model.close()


def test_dp_attention_equals_plain_tp_on_gpu():
    w = _wl("decode", n_seqs=16, seq_len=1, ctx=300, n_heads=16, n_kv=2)
    outs = {}
    for attn_dp in (1, 2, 4, 8):
        model, h, _ = _run(w, 8, attn_dp)
        outs[attn_dp] = to_f64(h)
        model.close()
    for attn_dp in (2, 4, 8):
        assert rel_err(outs[attn_dp], outs[1]) <= 1e-2, attn_dp


def test_forward_with_dp_attention_counts_one_gather_per_layer():
    w = _wl("decode", n_seqs=6, seq_len=1, ctx=40, layers=2, embed=True)
    t, attn_dp = 4, 2
    model, _, _ = build_model(w, t, attn_dp=attn_dp)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    model.reset_stats()
    logits = model.forward(ids, batch)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    st = model.stats()
    assert st.dp_gathers == 2 and st.allreduces == 2 * 2 + 1 and st.allgathers == 1
    dims = oracle_dims(w)
    h = O.embed(synth.host_weight(w, "embed", 0, (w.vocab, w.hidden)), ids_np)
    ob = oracle_batch(w)
    for l in range(2):
        kc, vc = oracle_caches(w, l, range(w.n_seqs))
        h = O.layer_forward(h, oracle_layer(w, l), kc, vc, ob, dims)
    ref = O.lm_head(h[ob.sample_rows()], synth.host_weight(w, "final_norm", 0, (w.hidden,)),
                    synth.host_weight(w, "lm_head", 0, (w.vocab, w.hidden)), dims)
    assert rel_err(to_f64(logits), ref) <= 5e-2
    model.close()
