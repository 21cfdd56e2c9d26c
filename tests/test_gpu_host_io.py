"""The host-buffer entry point tp_layer_forward_host: pinned host rows in,
the layer on the device, host rows out.  Its result must equal
tp_layer_forward's bit for bit (same kernels), also when one pinned buffer is
both input and output over consecutive calls (each call's transfers wait for
the previous call), and pageable host memory is refused.  Both transfer
paths are run: kernels over the coherent host link (GB300) and the copy
engine (forced with host_io = 1)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402
from megatron_tensor_layers_tp_gb300 import binding as B  # noqa: E402
from tests.parity_utils import build_model, make_batch  # noqa: E402


def _wl(mode, n_seqs, seq_len, ctx, layers=1):
    return synth.Workload(f"unit-hostio-{mode}", 512, 8, 2, 64, 1536, 1001, layers, (1,), mode,
                          n_seqs, seq_len, ctx, False, seed=9, norm_weight_sigma=0.1)


def _hidden(w):
    h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(h, w.seed, synth.tensor_id("hidden"), w.sigma_h)
    return h


@pytest.mark.parametrize("mode,n_seqs,seq_len,ctx", [("decode", 16, 1, 300), ("decode", 48, 1, 90),
                                                     ("prefill", 4, 30, 30)])
@pytest.mark.parametrize("fused,attn_dp", [(True, 1), (False, 1), (True, 2)])
@pytest.mark.parametrize("host_io", [0, 1])
def test_host_entry_point_equals_device_layer(mode, n_seqs, seq_len, ctx, fused, attn_dp, host_io):
    # host_io 0: on GB300 the transfers are two kernels over NVLink-C2C;
    # host_io 1: cudaMemcpyAsync on the stream (the path of other GPUs)
    w = _wl(mode, n_seqs, seq_len, ctx)
    model, _, _ = build_model(w, 4, attn_dp=attn_dp, host_io=host_io)
    batch, _ = make_batch(model, w)
    h0 = _hidden(w)
    ref = h0.clone()
    model.reset_stats()
    model.layer_forward(0, batch, ref, fused=fused)
    layer_launches = model.stats().kernel_launches
    hin = h0.cpu().pin_memory()
    hout = torch.zeros_like(hin).pin_memory()
    hdev = torch.empty_like(h0)
    model.reset_stats()
    model.layer_forward_host(0, batch, hin, hout, hdev, fused=fused)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    assert model.stats().kernel_launches == layer_launches + (2 if host_io == 0 else 0)
    assert torch.equal(hout.view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(hdev.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(hin.view(torch.int16), h0.cpu().view(torch.int16))  # input untouched
    model.close()


@pytest.mark.parametrize("host_io", [0, 1])
def test_one_pinned_buffer_through_consecutive_layers(host_io):
    w = _wl("decode", 16, 1, 120, layers=3)
    model, _, _ = build_model(w, 2, host_io=host_io)
    batch, _ = make_batch(model, w)
    h0 = _hidden(w)
    ref = h0.clone()
    for l in range(3):
        model.layer_forward(l, batch, ref)
    hbuf = h0.cpu().pin_memory()
    hdev = torch.empty_like(h0)
    for l in range(3):
        model.layer_forward_host(l, batch, hbuf, hbuf, hdev)  # no synchronisation in between
    torch.cuda.synchronize()
    assert model.check_device() == 0
    assert torch.equal(hbuf.view(torch.int16), ref.cpu().view(torch.int16))
    model.close()


def test_pageable_host_memory_is_refused():
    w = _wl("decode", 4, 1, 20)
    model, _, _ = build_model(w, 2)
    batch, _ = make_batch(model, w)
    hin = _hidden(w).cpu()  # pageable
    hout = torch.empty_like(hin).pin_memory()
    hdev = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.TPError) as ei:
        model.layer_forward_host(0, batch, hin, hout, hdev)
    assert ei.value.status == B.STATUS["TP_ERR_ARG"]
    model.close()
