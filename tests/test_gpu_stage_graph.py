"""Pipeline-stage split ("张量、流水线与数据并行", 流水线并行: layers cut into
consecutive groups, the running hidden state handed from one stage to the
next) and CUDA-graph capture of a decode step (the fixed per-step cost that
CUDA graph addresses, "Tensor Parallelism 执行路径", 每 token 的通信量).

Both only re-package the same kernels, so they are checked bit for bit
against the eager tp_forward / tp_layer_forward, and also directly against
the oracle: the staged logits, the replayed forward's logits (twice, with
different token ids) and the replayed decode layer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle as O  # noqa: E402
import synth  # noqa: E402
from megatron_tensor_layers_tp_gb300 import binding as B  # noqa: E402
from tests.parity_utils import (build_model, make_batch, oracle_batch, oracle_caches,  # noqa: E402
                                oracle_dims, oracle_forward, oracle_layer, rel_err, to_f64)

LOGIT_TOL = 5e-2
LAYER_TOL = 2e-2


def _wl(n_seqs=6, ctx=40, layers=4, hidden=256, n_heads=4, n_kv=2, head_dim=64, inter=768,
        vocab=1001):
    return synth.Workload("unit-stages", hidden, n_heads, n_kv, head_dim, inter, vocab, layers,
                          (1,), "decode", n_seqs, 1, ctx, True, seed=9, norm_weight_sigma=0.1)


def _bits(x):
    return x.view(torch.int16)


def _eager(model, w, batch, ids):
    h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    logits = model.forward(ids, batch, h=h)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    return h, logits


@pytest.mark.parametrize("t", [2, 4])
@pytest.mark.parametrize("cuts", [(2,), (1, 2, 3)])
def test_stage_split_equals_forward(t, cuts):
    w = _wl()
    model, _, _ = build_model(w, t)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    h_ref, logits_ref = _eager(model, w, batch, ids)

    bounds = [0, *cuts, w.n_layers]
    bufs = [torch.full((w.tokens, w.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
            for _ in range(len(bounds) - 1)]
    logits = torch.empty_like(logits_ref)
    model.reset_stats()
    for s in range(len(bounds) - 1):
        first, last = bounds[s], bounds[s + 1]
        if s > 0:
            model.stage_send(bufs[s - 1], bufs[s])
        model.stage_forward(first, last - first, batch, bufs[s],
                            ids=ids if s == 0 else None,
                            logits=logits if s == len(bounds) - 2 else None)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    assert torch.equal(_bits(bufs[-1]), _bits(h_ref))
    assert torch.equal(_bits(logits), _bits(logits_ref))
    st = model.stats()
    n_bound = len(bounds) - 2
    assert st.stage_sends == n_bound
    assert st.stage_send_bytes == n_bound * w.tokens * w.hidden * 2
    # the layers' own reductions are unchanged by the split: 2 per layer + embedding
    assert st.allreduces == 2 * w.n_layers + 1
    assert st.allgathers == 1
    model.close()


def test_staged_logits_match_oracle():
    w = _wl(layers=2)
    t = 2
    model, _, _ = build_model(w, t)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    a = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    logits = torch.empty((w.n_seqs, w.vocab), dtype=torch.bfloat16, device="cuda")
    model.stage_forward(0, 1, batch, a, ids=ids)
    model.stage_send(a, b)
    model.stage_forward(1, 1, batch, b, logits=logits)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    ref = oracle_forward(w, ids_np)
    assert rel_err(to_f64(logits), ref) <= LOGIT_TOL
    model.close()


def test_stage_arguments_rejected():
    w = _wl(layers=2)
    model, _, _ = build_model(w, 2)
    batch, _ = make_batch(model, w)
    ids = torch.from_numpy(synth.token_ids(w)).cuda()
    h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    logits = torch.empty((w.n_seqs, w.vocab), dtype=torch.bfloat16, device="cuda")
    cb = batch.to_c()
    ws, nws = model.ws_args
    s = torch.cuda.current_stream().cuda_stream
    H = model.handle
    # embedding only on a stage that starts at layer 0; logits only on the last
    assert B.tp_stage_forward(H, 1, 1, ids.data_ptr(), cb, h.data_ptr(), 0, w.vocab, 1, ws, nws,
                              s) == B.STATUS["TP_ERR_ARG"]
    assert B.tp_stage_forward(H, 0, 1, 0, cb, h.data_ptr(), logits.data_ptr(), w.vocab, 1, ws,
                              nws, s) == B.STATUS["TP_ERR_ARG"]
    assert B.tp_stage_forward(H, 1, 2, 0, cb, h.data_ptr(), 0, w.vocab, 1, ws, nws,
                              s) == B.STATUS["TP_ERR_ARG"]
    # overlapping hand-off buffers
    assert B.tp_stage_send(H, h.data_ptr(), h[1:].data_ptr(), w.tokens, s) == B.STATUS["TP_ERR_ARG"]
    assert B.tp_stage_send(H, h.data_ptr(), 0, w.tokens, s) == B.STATUS["TP_ERR_ARG"]
    model.close()


@pytest.mark.parametrize("t", [1, 2])
def test_graph_forward_replays_eager(t):
    w = _wl(layers=2)
    model, _, _ = build_model(w, t)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    h_ref, logits_ref = _eager(model, w, batch, ids)
    stream = torch.cuda.Stream()
    h = torch.empty_like(h_ref)
    logits = torch.empty_like(logits_ref)
    graph = model.capture_forward(ids, batch, h, logits, stream)
    model.reset_stats()
    graph.launch(stream)
    stream.synchronize()
    assert model.check_device() == 0
    assert torch.equal(_bits(logits), _bits(logits_ref))
    assert torch.equal(_bits(h), _bits(h_ref))
    # and the replay against the oracle itself
    assert rel_err(to_f64(logits), oracle_forward(w, ids_np)) <= LOGIT_TOL
    st = model.stats()
    assert st.allreduces == 2 * w.n_layers + 1 and st.allgathers == 1
    assert st.kernel_launches > 0
    # new token ids in the same buffer: the replay reads them
    ids2_np = (ids_np * 7 + 3) % w.vocab
    ids.copy_(torch.from_numpy(ids2_np))
    graph.launch(stream)
    stream.synchronize()
    _, logits_ref2 = _eager(model, w, batch, ids)
    assert torch.equal(_bits(logits), _bits(logits_ref2))
    assert not torch.equal(_bits(logits_ref2), _bits(logits_ref))
    assert rel_err(to_f64(logits), oracle_forward(w, ids2_np)) <= LOGIT_TOL
    graph.close()
    model.close()


@pytest.mark.parametrize("pairs", [1, 2])
def test_graph_prefill_forward_replays_eager(pairs):
    # a prefill forward (2 x 40 tokens, above the decode orientation) captured
    # with its GEMMs on CTA pairs (cluster launches, pairs = 1) or single CTAs
    w = synth.Workload("unit-stages-prefill", 256, 4, 2, 64, 768, 1001, 2, (1,), "prefill", 2,
                       40, 40, True, seed=9, norm_weight_sigma=0.1)
    model, _, _ = build_model(w, 2, prefill_cta_pairs=pairs)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    h_ref, logits_ref = _eager(model, w, batch, ids)
    stream = torch.cuda.Stream()
    h = torch.empty_like(h_ref)
    logits = torch.empty_like(logits_ref)
    graph = model.capture_forward(ids, batch, h, logits, stream)
    graph.launch(stream)
    stream.synchronize()
    assert model.check_device() == 0
    assert torch.equal(_bits(logits), _bits(logits_ref))
    assert torch.equal(_bits(h), _bits(h_ref))
    assert rel_err(to_f64(logits), oracle_forward(w, ids_np)) <= LOGIT_TOL
    graph.close()
    model.close()


def test_graph_layer_replays_eager_at_decode_shape():
    # one Llama-3.1-8B-shaped layer at t = 8, 16 sequences, 256-token context
    w = synth.Workload("unit-graph-layer", 4096, 32, 8, 128, 14336, 1000, 1, (8,), "decode", 16,
                       1, 256, False, seed=3)
    model, _, _ = build_model(w, 8)
    batch, _ = make_batch(model, w)
    h0 = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(h0, w.seed, synth.tensor_id("hidden"), w.sigma_h)
    ref = h0.clone()
    model.layer_forward(0, batch, ref)
    stream = torch.cuda.Stream()
    h = h0.clone()
    torch.cuda.synchronize()
    graph = model.capture_layer(0, batch, h, stream)
    graph.launch(stream)
    stream.synchronize()
    assert model.check_device() == 0
    assert torch.equal(_bits(h), _bits(ref))
    # the replayed layer against the oracle
    kc, vc = oracle_caches(w, 0, range(w.n_seqs))
    want = O.layer_forward(synth.host_hidden(w), oracle_layer(w, 0), kc, vc, oracle_batch(w),
                           oracle_dims(w))
    assert rel_err(to_f64(h), want) <= LAYER_TOL
    # replay twice more from the same input: identical
    for _ in range(2):
        with torch.cuda.stream(stream):
            h.copy_(h0)  # ordered before the replay on the same stream
        graph.launch(stream)
    stream.synchronize()
    assert torch.equal(_bits(h), _bits(ref))
    graph.close()
    model.close()


def test_graph_capture_rejects_default_stream_and_profiling():
    w = _wl(layers=1)
    model, _, _ = build_model(w, 2)
    batch, _ = make_batch(model, w)
    h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    cb = batch.to_c()
    ws, nws = model.ws_args
    st, g = B.tp_graph_capture_layer(model.handle, 0, cb, h.data_ptr(), 1, ws, nws, 0)
    assert st == B.STATUS["TP_ERR_ARG"] and not g
    stream = torch.cuda.Stream()
    B.tp_profile(model.handle, True)
    st, g = B.tp_graph_capture_layer(model.handle, 0, cb, h.data_ptr(), 1, ws, nws,
                                     stream.cuda_stream)
    assert st == B.STATUS["TP_ERR_ARG"] and not g
    B.tp_profile(model.handle, False)
    model.close()
