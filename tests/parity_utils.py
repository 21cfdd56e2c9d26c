"""Helpers shared by the parity tests, the smoke check and the benchmark's CPU
baseline: build the same seeded inputs for the CUDA path (device fills) and
for the oracle (host fills), and compare outputs."""
from __future__ import annotations

import os
import sys
from typing import Dict, List, Sequence

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from synth import Workload  # noqa: E402

LAYER_KINDS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(gpu - ref)) / (np.max(np.abs(ref)) + 1e-6))


# ---------------------------------------------------------------------------
# host side (oracle inputs)
# ---------------------------------------------------------------------------
def oracle_dims(w: Workload):
    import oracle as O
    return O.Dims(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab,
                  w.rms_eps, w.rope_theta)


def oracle_layer(w: Workload, layer: int):
    import oracle as O
    shapes = synth.weight_shapes(w, layer)
    shapes.update(synth.bias_shapes(w))
    return O.LayerWeights(**{k: synth.host_weight(w, k, layer, shapes[k])
                             for k in (*LAYER_KINDS, *synth.bias_shapes(w))})


def oracle_caches(w: Workload, layer: int, seqs: Sequence[int]):
    k = {i: synth.host_kv(w, "k_cache", layer, b) for i, b in enumerate(seqs)}
    v = {i: synth.host_kv(w, "v_cache", layer, b) for i, b in enumerate(seqs)}
    return k, v


# ---------------------------------------------------------------------------
# device side (CUDA path inputs)
# ---------------------------------------------------------------------------
def device_weight(w: Workload, kind: str, layer: int, shape):
    import torch
    t = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    if kind in ("attn_norm", "mlp_norm", "final_norm") and w.norm_weight_sigma == 0.0:
        t.fill_(1.0)
    elif kind in ("attn_norm", "mlp_norm", "final_norm"):
        h = synth.host_weight(w, kind, layer, shape)
        t.copy_(torch.from_numpy(h.astype(np.float32)).to(torch.bfloat16))
    else:
        synth.fill_normal_(t, w.seed, synth.tensor_id(kind, layer), synth.sigma_for(w, kind))
    return t


def device_layer(w: Workload, layer: int) -> Dict[str, "torch.Tensor"]:
    shapes = synth.weight_shapes(w, layer)
    shapes.update(synth.bias_shapes(w))
    return {k: device_weight(w, k, layer, shapes[k]) for k in (*LAYER_KINDS, *synth.bias_shapes(w))}


def fill_device_kv(model, w: Workload, cache, kind: str, layer: int) -> None:
    """Fill the library-layout cache [copies, n_seqs, kv_r, l_max, d] with the
    logical synthetic cache [n_seqs, n_kv, l_max, d]."""
    c = model.cfg
    for cp in range(c.kv_copies):
        for b in range(w.n_seqs):
            synth.fill_normal_(cache[cp, b], w.seed, synth.tensor_id(kind, layer), w.sigma_kv,
                               start=synth.kv_logical_start(w, b, cp * c.kv_heads_per_rank))


def to_f64(t) -> np.ndarray:
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def build_model(w: Workload, t: int, layers: int = None, with_head: bool = None, max_tokens=None,
                attn_dp: int = 1, host_io: int = 0, plain_column_shards: int = 0,
                prefill_bn: int = 0, prefill_cta_pairs: int = 0):
    """Device weights + TPModel for workload w at t ranks (attention over
    t / attn_dp ranks per DP group); host_io, plain_column_shards,
    prefill_bn and prefill_cta_pairs as in tp_config_t."""
    import torch
    from megatron_tensor_layers_tp_gb300.runtime import TPModel, make_config
    n_layers = w.n_layers if layers is None else layers
    head = w.with_embed if with_head is None else with_head
    cfg = make_config(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab,
                      n_layers, t, w.rms_eps, w.rope_theta, max_positions=max(w.l_max, 16),
                      attn_dp=attn_dp, host_io=host_io, plain_column_shards=plain_column_shards,
                      prefill_bn=prefill_bn, prefill_cta_pairs=prefill_cta_pairs)
    dev_layers = []
    for l in range(n_layers):
        dev_layers.append(device_layer(w, l))
    embed = final_norm = lm = None
    if head:
        embed = device_weight(w, "embed", 0, (w.vocab, w.hidden))
        lm = device_weight(w, "lm_head", 0, (w.vocab, w.hidden))
        final_norm = device_weight(w, "final_norm", 0, (w.hidden,))
    model = TPModel(cfg, dev_layers, embed, final_norm, lm,
                    max_tokens=max_tokens or max(w.tokens, 1))
    torch.cuda.synchronize()
    return model, dev_layers, (embed, final_norm, lm)


def make_batch(model, w: Workload, caches=None):
    from megatron_tensor_layers_tp_gb300.runtime import decode_batch, prefill_batch
    n_layers = model.cfg.n_layers
    if caches is None:
        ks, vs = [], []
        for l in range(n_layers):
            k = model.alloc_kv(w.n_seqs, w.l_max)
            v = model.alloc_kv(w.n_seqs, w.l_max)
            fill_device_kv(model, w, k, "k_cache", l)
            fill_device_kv(model, w, v, "v_cache", l)
            ks.append(k)
            vs.append(v)
        caches = (ks, vs)
    ks, vs = caches
    if w.mode == "decode":
        return decode_batch(w.n_seqs, w.ctx, ks, vs, w.l_max), caches
    return prefill_batch(w.n_seqs, w.seq_len, ks, vs, w.l_max), caches


def oracle_forward(w: Workload, ids_np, seqs: Sequence[int] = None):
    """The oracle's logits for workload w (embedding, every layer, final norm,
    LM head at each sequence's last token); ``seqs`` restricts a decode
    workload to those sequences (independent of the others), weights and
    caches regenerated layer by layer."""
    import oracle as O
    dims = oracle_dims(w)
    if seqs is None:
        seqs = list(range(w.n_seqs))
        ob = oracle_batch(w)
        ids_sel = ids_np
    else:
        assert w.mode == "decode"
        ob = O.Batch.decode(len(seqs), w.ctx)
        ids_sel = np.asarray(ids_np)[list(seqs)]

    def layers():
        for l in range(w.n_layers):
            kc, vc = oracle_caches(w, l, seqs)
            yield oracle_layer(w, l), kc, vc
    return O.forward(ids_sel, synth.host_weight(w, "embed", 0, (w.vocab, w.hidden)), layers(),
                     synth.host_weight(w, "final_norm", 0, (w.hidden,)),
                     synth.host_weight(w, "lm_head", 0, (w.vocab, w.hidden)), ob, dims)


def oracle_batch(w: Workload):
    import oracle as O
    if w.mode == "decode":
        return O.Batch.decode(w.n_seqs, w.ctx)
    return O.Batch.prefill(w.n_seqs, w.seq_len)


# ---------------------------------------------------------------------------
# the smoke check: config-1 forward at t = 2
# ---------------------------------------------------------------------------
def run_tiny_forward_check(t: int = 2, tol: float = 5e-2) -> float:
    import torch
    import oracle as O
    w = synth.WORKLOADS["tiny"]
    model, _, _ = build_model(w, t)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    logits = model.forward(ids, batch, fused=True)
    torch.cuda.synchronize()
    st = model.check_device()
    assert st == 0, f"device status {st}"
    gpu = to_f64(logits)
    ref = oracle_forward(w, ids_np)
    err = rel_err(gpu, ref)
    model.close()
    if not err <= tol:
        raise AssertionError(f"tiny forward parity failed: rel err {err:.3e} > {tol}")
    return err
