"""Parity at the full workload sizes, in the launch configuration the
benchmark times (decode batches use the swapped orientation, the 2048-token
prefill the normal one).

- tiny (H256, t=2): embed + 1 layer + LM head, full check.
- Llama-3.1-8B-shaped decode layer, B=16, ctx 1024, t = 1, 2, 4, 8: full check.
- Qwen2.5-32B-shaped decode layer, B=64, ctx 2048, t=8, with 8 and with 4 KV
  heads (each KV head replicated on 2 ranks): full check.
- Llama-3.1-8B-shaped prefill, 8 x 256 tokens, t=4, embedding + 1 layer + LM
  head on the last position of each sequence: full check.
- 32-layer Llama-3.1-8B-shaped decode forward, B=64, ctx 4096, t=8: decode
  sequences are independent, so the oracle computes sampled sequences one by
  one through all 32 layers (weights regenerated per layer).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle as O  # noqa: E402
import synth  # noqa: E402
from tests.parity_utils import (build_model, make_batch, oracle_batch, oracle_caches,  # noqa: E402
                                oracle_dims, oracle_forward, oracle_layer, rel_err,
                                run_tiny_forward_check, to_f64)

LAYER_TOL = 2e-2
LOGIT_TOL = 5e-2


def test_config_tiny_forward():
    assert run_tiny_forward_check(2) <= LOGIT_TOL


def _layer_parity(w, t):
    model, _, _ = build_model(w, t)
    batch, (ks, vs) = make_batch(model, w)
    h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(h, w.seed, synth.tensor_id("hidden"), w.sigma_h)
    model.layer_forward(0, batch, h)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    dims = oracle_dims(w)
    kc, vc = oracle_caches(w, 0, range(w.n_seqs))
    ref = O.layer_forward(synth.host_hidden(w), oracle_layer(w, 0), kc, vc, oracle_batch(w), dims)
    err = rel_err(to_f64(h), ref)
    out = to_f64(h)
    model.close()
    del ks, vs
    torch.cuda.empty_cache()
    return err, out


def test_config_llama8b_decode_layer_all_t():
    w = synth.WORKLOADS["llama8b_decode"]
    outs = {}
    for t in (1, 2, 4, 8):
        err, outs[t] = _layer_parity(w, t)
        assert err <= LAYER_TOL, (t, err)
    for t in (2, 4, 8):  # sharded vs unsharded on the GPU
        assert rel_err(outs[t], outs[1]) <= 1e-2, t


@pytest.mark.parametrize("name", ["qwen32b_decode", "qwen32b_decode_kv4"])
def test_config_qwen32b_decode_layer(name):
    w = synth.WORKLOADS[name]
    err, _ = _layer_parity(w, 8)
    assert err <= LAYER_TOL, err


def test_config_llama8b_prefill_with_embed_and_head():
    w = synth.WORKLOADS["llama8b_prefill"]
    t = 4
    model, _, _ = build_model(w, t)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    logits = model.forward(ids, batch)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    gpu = to_f64(logits)
    model.close()
    torch.cuda.empty_cache()
    ref = oracle_forward(w, ids_np)
    assert gpu.shape == (8, w.vocab)
    assert rel_err(gpu, ref) <= LOGIT_TOL


def test_config_llama8b_full_32_layers_sampled_sequences():
    w = synth.WORKLOADS["llama8b_full"]
    t = 8
    model, _, _ = build_model(w, t)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    model.reset_stats()
    logits = model.forward(ids, batch)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    st = model.stats()
    assert st.allreduces == 65 and st.allgathers == 1       # 2 x 32 + 1, plus the logits gather
    assert st.allreduce_payload_bytes == 65 * 8192 * w.tokens
    gpu = to_f64(logits)
    model.close()
    del batch
    torch.cuda.empty_cache()
    # decode sequences are independent: the oracle takes 8 of the 64, spread
    # over the batch (first and last included), through all 32 layers
    sample = [0, 9, 18, 27, 37, 46, 55, 63]
    ref = oracle_forward(w, ids_np, seqs=sample)
    for i, b in enumerate(sample):
        assert rel_err(gpu[b], ref[i]) <= LOGIT_TOL, b
