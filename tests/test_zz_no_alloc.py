"""The no-allocation variant of the fused row-parallel reduction.

Callers that cannot allocate device memory (a plug-in handed only its input
and output tensors by a host framework, or a loop that cannot afford the
implicit synchronisation of cudaMalloc) call tp_row_linear_reduce_noalloc,
whose scratch is a fixed array inside the library.  It runs the same kernel
with the same schedule as the workspace entry point, so its result must equal
that entry point's bit for bit, call after call (every call reuses the same
array), and must match the oracle's rank-ordered all-reduce.  Both GEMM
schedules are covered: stream-K with partials in the array (hidden 1024) and
cluster split-K (hidden 4096, 32 output tiles).  This file is collected last
on purpose.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle as O  # noqa: E402
import synth  # noqa: E402
from megatron_tensor_layers_tp_gb300 import binding as B  # noqa: E402
from megatron_tensor_layers_tp_gb300.runtime import TPModel, make_config  # noqa: E402
from tests.parity_utils import device_layer, rel_err, to_f64  # noqa: E402

TOL = 2e-2


def _setup(t=4, M=16, hidden=1024):
    if hidden == 1024:
        w = synth.Workload("noalloc", 1024, 16, 4, 64, 2048, 1000, 1, (t,), "decode", M, 1, 8, False,
                           seed=6)
    else:
        w = synth.Workload("noalloc4096", 4096, 32, 8, 128, 2048, 1000, 1, (t,), "decode", M, 1, 8,
                           False, seed=6)
    cfg = make_config(w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.vocab, 1, t,
                      max_positions=64)
    model = TPModel(cfg, [device_layer(w, 0)], max_tokens=M)
    return w, model


def _inputs(M, K, H):
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(x, 6, 4242 + K, 1.0)
    res = torch.empty((M, H), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(res, 6, 4343 + K, 1.0)
    return x, res


def _oracle(w, which, x, res, t):
    """residual + the rank-ordered sum of the t partials, rounded once."""
    shapes = synth.weight_shapes(w, 0)
    kind = "wo" if which == B.TP_O else "wd"
    W = synth.host_weight(w, kind, 0, shapes[kind])
    xs = to_f64(x)
    parts = [O.linear(xr, Wr) for xr, Wr in zip(O.shard_rows_by_input(xs, t),
                                                 O.shard_rows_by_input(W, t))]
    return O.round_bf16(to_f64(res) + O.all_reduce_sum(parts))


@pytest.mark.parametrize("hidden,M", [(1024, 1), (1024, 16), (1024, 64), (4096, 1), (4096, 16),
                                      (4096, 64)])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(hidden, M):
    t = 4 if hidden == 1024 else 8
    w, model = _setup(t=t, M=M, hidden=hidden)
    s = torch.cuda.current_stream().cuda_stream
    for which, K in ((B.TP_O, w.n_heads * w.head_dim), (B.TP_DOWN, w.intermediate)):
        x, res = _inputs(M, K, w.hidden)
        ref = model.row_linear_reduce(0, which, x, residual=res, fused=True)
        torch.cuda.synchronize()
        want = _oracle(w, which, x, res, t)
        assert rel_err(to_f64(ref), want) <= TOL
        for _ in range(2):  # the shared array keeps the previous call's contents
            y = torch.empty((M, w.hidden), dtype=torch.bfloat16, device="cuda")
            st = B.tp_row_linear_reduce_noalloc(model.handle, 0, which, x.data_ptr(), K // t,
                                                x.stride(0), M, res.data_ptr(), y.data_ptr(), s)
            assert st == B.TP_OK, B.strerror(st)
            torch.cuda.synchronize()
            assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
            assert rel_err(to_f64(y), want) <= TOL
    assert model.check_device() == 0
    model.close()


def test_noalloc_rejects_requests_beyond_its_fixed_scratch():
    w, model = _setup(M=80)
    K = w.n_heads * w.head_dim
    x, res = _inputs(80, K, w.hidden)
    y = torch.empty((80, w.hidden), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = B.tp_row_linear_reduce_noalloc(model.handle, 0, B.TP_O, x.data_ptr(), K // model.cfg.t,
                                        x.stride(0), 80, res.data_ptr(), y.data_ptr(), s)
    assert st == B.STATUS["TP_ERR_WORKSPACE"]
    model.close()
