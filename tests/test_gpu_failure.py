"""Failure detection on the GPU without a fault: every wait in the library's
kernels is bounded; a wait that runs out records TP_ERR_DEVICE_TIMEOUT in the
model's status word and the kernel returns.  The self-test makes one wait run
out (an mbarrier phase nothing completes), the host reads the status, and the
context keeps working."""
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import synth  # noqa: E402
from megatron_tensor_layers_tp_gb300 import binding as B  # noqa: E402
from tests.parity_utils import build_model, run_tiny_forward_check  # noqa: E402


def test_bounded_wait_runs_out_reports_and_leaves_the_context_usable():
    w = synth.WORKLOADS["tiny"]
    model, _, _ = build_model(w, 2)
    s = torch.cuda.current_stream().cuda_stream
    assert model.check_device() == B.TP_OK
    assert B.lib().tp_selftest_wait_timeout(model.handle, 100, s) == B.TP_OK
    assert model.check_device() == B.STATUS["TP_ERR_DEVICE_TIMEOUT"]
    assert model.check_device() == B.TP_OK          # read once, then cleared
    assert B.lib().tp_selftest_wait_timeout(model.handle, 0, s) == B.STATUS["TP_ERR_ARG"]
    model.close()
    # kernels still run and agree with the oracle afterwards
    assert run_tiny_forward_check(2) <= 5e-2
