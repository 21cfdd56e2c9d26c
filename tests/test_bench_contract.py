"""The benchmark's contract on the CPU: the algorithmic bytes behind the HBM
roofline, and the JSON line of the reference arm (the oracle timed on the
host cores)."""
import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_algorithmic_bytes_of_the_llama8b_decode_layer():
    """Bytes one decode step of a Llama-3.1-8B layer must move, written out
    from the shape (hidden 4096, 32 query / 8 KV heads of 128, intermediate
    14336; 16 tokens, 1024-token context, bf16): each weight matrix once, the
    activations in and out, the residual read and written by the row-parallel
    steps, and the K and V cache read once by attention."""
    w = synth.WORKLOADS["llama8b_decode"]
    assert (w.hidden, w.n_heads, w.n_kv_heads, w.head_dim, w.intermediate, w.tokens, w.ctx) == \
        (4096, 32, 8, 128, 14336, 16, 1024)
    want = {
        # W_qkv [(32 + 2*8) * 128, 4096]; x in [16, 4096]; q, k, v out [16, 6144]
        "gemm_qkv": 6144 * 4096 * 2 + 16 * 4096 * 2 + 16 * 6144 * 2,
        # W_o [4096, 4096]; attention out in; residual in, h out
        "gemm_o": 4096 * 4096 * 2 + 16 * 4096 * 2 + 2 * 16 * 4096 * 2,
        # W_gate, W_up [14336, 4096] each; x in; SiLU(gate) * up out [16, 14336]
        "gemm_gate_up": 2 * 14336 * 4096 * 2 + 16 * 4096 * 2 + 16 * 14336 * 2,
        # W_down [4096, 14336]; activations in; residual in, h out
        "gemm_down": 4096 * 14336 * 2 + 16 * 14336 * 2 + 2 * 16 * 4096 * 2,
        # K and V of 16 sequences x 8 heads x 1024 positions x 128; q in, o out
        "attn_decode": 2 * 16 * 8 * 1024 * 128 * 2 + 2 * 16 * 4096 * 2,
    }
    assert want["gemm_gate_up"] == 235_470_848
    for t in (1, 2, 4, 8):
        kb, total = bench.layer_bytes(w, t)
        for k, v in want.items():
            assert kb[k] == v, (t, k)
        assert total == sum(want.values()) == 505_610_240


def test_reference_arm_prints_the_contract_line():
    saved = sys.argv
    sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                "--reference-budget-s", "1"]
    try:
        args = bench.parse()
    finally:
        sys.argv = saved
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, rank=0, world=1)
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"].startswith("Llama-3.1-8B")
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    # value = tokens of the steps run / their wall time
    w = synth.WORKLOADS["llama8b_decode"]
    assert d["value"] == pytest.approx(d["steps_run"] * w.tokens / (d["ms_per_step"] * d["steps_run"] / 1e3),
                                       rel=1e-2)
