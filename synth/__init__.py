"""Seeded synthetic inputs: shapes of the Llama/Qwen-style workloads and the
counter-based generator that fills them (definition in ``synth_def.h``).

This module holds no arithmetic of the tensor-parallel method.  It serves both
sides of every parity check: the oracle reads host fills, the CUDA path is fed
device fills of the same (seed, tensor id, flat index) values.

The KV cache content is defined on a *logical* layout ``[B, n_kv, L_max, d]``
per (layer, K|V); a consumer with another physical layout maps its blocks onto
logical flat-index ranges (``kv_logical_start``).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_HOST_SO = os.path.join(_BUILD, "libsynth_host.so")
_CUDA_SO = os.path.join(_BUILD, "libsynth_cuda.so")

SQRT3 = math.sqrt(3.0)


# ---------------------------------------------------------------------------
# build
# ---------------------------------------------------------------------------
def build_commands(cuda: bool = True):
    os.makedirs(_BUILD, exist_ok=True)
    cmds = [["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC",
             "-o", _HOST_SO, os.path.join(_HERE, "synth_host.c"), "-lm"]]
    if cuda:
        cmds.append(["nvcc", "-O2", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                     "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "shared",
                     "-o", _CUDA_SO, os.path.join(_HERE, "synth_cuda.cu")])
    return cmds


def build(cuda: bool = True) -> None:
    procs = [subprocess.Popen(c) for c in build_commands(cuda)]
    for p, c in zip(procs, build_commands(cuda)):
        if p.wait() != 0:
            raise RuntimeError("synth build failed: " + " ".join(c))


_host_lib = None
_cuda_lib = None


def _host():
    global _host_lib
    if _host_lib is None:
        if not os.path.exists(_HOST_SO):
            build(cuda=False)
        lib = ctypes.CDLL(_HOST_SO)
        lib.synth_fill_normal_bf16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                               ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double]
        lib.synth_fill_normal_bf16.restype = None
        lib.synth_fill_uniform_i32.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                               ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32]
        lib.synth_fill_uniform_i32.restype = None
        _host_lib = lib
    return _host_lib


def _cuda():
    global _cuda_lib
    if _cuda_lib is None:
        if not os.path.exists(_CUDA_SO):
            raise RuntimeError("synth CUDA library not built; run synth.build()")
        lib = ctypes.CDLL(_CUDA_SO)
        for name, last in (("synth_fill_normal_bf16_dev", ctypes.c_double),
                           ("synth_fill_uniform_i32_dev", ctypes.c_uint32)):
            fn = getattr(lib, name)
            fn.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                           ctypes.c_uint64, last, ctypes.c_void_p]
            fn.restype = ctypes.c_int
        _cuda_lib = lib
    return _cuda_lib


# ---------------------------------------------------------------------------
# tensor identities
# ---------------------------------------------------------------------------
_KINDS = {
    "embed": 1, "lm_head": 2, "final_norm": 3, "attn_norm": 4, "mlp_norm": 5,
    "wq": 6, "wk": 7, "wv": 8, "wo": 9, "wg": 10, "wu": 11, "wd": 12,
    "k_cache": 13, "v_cache": 14, "hidden": 15, "ids": 16, "x": 17,
    "bq": 18, "bk": 19, "bv": 20, "bo": 21, "bg": 22, "bu": 23, "bd": 24,
}
BIAS_KINDS = ("bq", "bk", "bv", "bo", "bg", "bu", "bd")


def tensor_id(kind: str, layer: int = 0) -> int:
    return (_KINDS[kind] << 32) | (layer & 0xFFFFFFFF)


# ---------------------------------------------------------------------------
# host fills (numpy)
# ---------------------------------------------------------------------------
def normal_bf16_bits(seed: int, tid: int, count: int, sigma: float, start: int = 0) -> np.ndarray:
    """uint16 bf16 bit patterns of flat indices [start, start+count)."""
    out = np.empty(count, dtype=np.uint16)
    if count:
        _host().synth_fill_normal_bf16(out.ctypes.data, seed, tid, start, count, sigma * SQRT3)
    return out


def uniform_i32(seed: int, tid: int, count: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(count, dtype=np.int32)
    if count:
        _host().synth_fill_uniform_i32(out.ctypes.data, seed, tid, start, count, n)
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def normal_f64(seed: int, tid: int, shape: Sequence[int], sigma: float, start: int = 0) -> np.ndarray:
    n = int(np.prod(shape)) if len(shape) else 1
    return bf16_bits_to_f64(normal_bf16_bits(seed, tid, n, sigma, start)).reshape(shape)


# ---------------------------------------------------------------------------
# device fills (torch tensors, CUDA)
# ---------------------------------------------------------------------------
def fill_normal_(tensor, seed: int, tid: int, sigma: float, start: int = 0, stream=None) -> None:
    """Fill a contiguous bf16 CUDA tensor with flat indices [start, start+numel)."""
    import torch
    assert tensor.dtype == torch.bfloat16 and tensor.is_cuda and tensor.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _cuda().synth_fill_normal_bf16_dev(tensor.data_ptr(), seed, tid, start, tensor.numel(),
                                            sigma * SQRT3, s)
    if rc != 0:
        raise RuntimeError(f"synth device fill failed: cuda error {rc}")


def fill_uniform_(tensor, seed: int, tid: int, n: int, start: int = 0, stream=None) -> None:
    import torch
    assert tensor.dtype == torch.int32 and tensor.is_cuda and tensor.is_contiguous()
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    rc = _cuda().synth_fill_uniform_i32_dev(tensor.data_ptr(), seed, tid, start, tensor.numel(), n, s)
    if rc != 0:
        raise RuntimeError(f"synth device fill failed: cuda error {rc}")


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    """Shapes and value recipe of one synthetic workload.

    mode "decode": n_seqs tokens, one per sequence, each at position ctx-1 and
    attending to ctx cached positions (ctx-1 random entries plus its own).
    mode "prefill": n_seqs sequences of seq_len tokens each, positions 0..,
    causal attention within a sequence, logits at each sequence's last token.
    """
    name: str
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    n_layers: int
    t_values: tuple
    mode: str
    n_seqs: int
    seq_len: int          # prefill tokens per sequence (1 in decode)
    ctx: int              # decode: attended context incl. the new token; prefill: seq_len
    with_embed: bool      # token ids -> embedding -> layers -> final norm -> LM head
    seed: int = 0
    sigma_w: float = 0.02
    sigma_kv: float = 1.0
    sigma_h: float = 1.0
    norm_weight_sigma: float = 0.0   # 0: norm weights are exactly 1
    bias: bool = False               # projections carry biases (BIAS_KINDS)
    sigma_b: float = 0.5
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0

    @property
    def tokens(self) -> int:
        return self.n_seqs * self.seq_len

    @property
    def l_max(self) -> int:
        return self.ctx


WORKLOADS = {
    "tiny": Workload("tiny", 256, 4, 2, 64, 1024, 1000, 1, (2,), "prefill", 1, 16, 16, True),
    "llama8b_decode": Workload("llama8b_decode", 4096, 32, 8, 128, 14336, 128256, 1, (1, 2, 4, 8),
                               "decode", 16, 1, 1024, False),
    "qwen32b_decode": Workload("qwen32b_decode", 5120, 40, 8, 128, 27648, 152064, 1, (8,),
                               "decode", 64, 1, 2048, False),
    "qwen32b_decode_kv4": Workload("qwen32b_decode_kv4", 5120, 40, 4, 128, 27648, 152064, 1, (8,),
                                   "decode", 64, 1, 2048, False),
    "llama8b_prefill": Workload("llama8b_prefill", 4096, 32, 8, 128, 14336, 128256, 1, (4,),
                                "prefill", 8, 256, 256, True),
    "llama8b_full": Workload("llama8b_full", 4096, 32, 8, 128, 14336, 128256, 32, (8,),
                             "decode", 64, 1, 4096, True),
}


def scaled(w: Workload, **kw) -> Workload:
    return replace(w, **kw)


def weight_shapes(w: Workload, layer: int) -> dict:
    H, d = w.hidden, w.head_dim
    return {
        "attn_norm": (H,), "mlp_norm": (H,),
        "wq": (w.n_heads * d, H), "wk": (w.n_kv_heads * d, H), "wv": (w.n_kv_heads * d, H),
        "wo": (H, w.n_heads * d),
        "wg": (w.intermediate, H), "wu": (w.intermediate, H), "wd": (H, w.intermediate),
    }


def bias_shapes(w: Workload) -> dict:
    """Shapes of the projection biases (empty when the workload has none)."""
    if not w.bias:
        return {}
    H, d = w.hidden, w.head_dim
    return {"bq": (w.n_heads * d,), "bk": (w.n_kv_heads * d,), "bv": (w.n_kv_heads * d,),
            "bo": (H,), "bg": (w.intermediate,), "bu": (w.intermediate,), "bd": (H,)}


def sigma_for(w: Workload, kind: str) -> float:
    if kind in ("attn_norm", "mlp_norm", "final_norm"):
        return w.norm_weight_sigma
    if kind in ("k_cache", "v_cache"):
        return w.sigma_kv
    if kind in ("hidden", "x"):
        return w.sigma_h
    if kind in BIAS_KINDS:
        return w.sigma_b
    return w.sigma_w


def host_weight(w: Workload, kind: str, layer: int, shape) -> np.ndarray:
    """float64 array holding the bf16 values of one unsharded weight."""
    if kind in ("attn_norm", "mlp_norm", "final_norm"):
        if w.norm_weight_sigma == 0.0:
            return np.ones(shape, dtype=np.float64)
        return 1.0 + normal_f64(w.seed, tensor_id(kind, layer), shape, w.norm_weight_sigma)
    return normal_f64(w.seed, tensor_id(kind, layer), shape, sigma_for(w, kind))


def token_ids(w: Workload) -> np.ndarray:
    return uniform_i32(w.seed, tensor_id("ids"), w.tokens, w.vocab)


def kv_logical_start(w: Workload, b: int, g: int) -> int:
    """Flat index of logical cache element [b, g, 0, 0] in [B, n_kv, L_max, d]."""
    return ((b * w.n_kv_heads + g) * w.l_max) * w.head_dim


def host_kv(w: Workload, kind: str, layer: int, b: int) -> np.ndarray:
    """Logical cache block [n_kv, L_max, d] of sequence b (float64 of bf16)."""
    n = w.n_kv_heads * w.l_max * w.head_dim
    vals = normal_f64(w.seed, tensor_id(kind, layer), (n,), w.sigma_kv, kv_logical_start(w, b, 0))
    return vals.reshape(w.n_kv_heads, w.l_max, w.head_dim)


def host_hidden(w: Workload) -> np.ndarray:
    return normal_f64(w.seed, tensor_id("hidden"), (w.tokens, w.hidden), w.sigma_h)
