"""Thin ctypes binding of the C ABI in ``include/tp.h``: same names, argument
marshalling only.  Every step of the forward path runs in the library's CUDA
kernels; there is no Python or CPU fallback.  Loading fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, Structure, c_char_p, c_float, c_int32, c_int64, c_size_t, c_void_p

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libtp_gb300.so")

TP_OK = 0
TP_QKV, TP_GATE_UP, TP_O, TP_DOWN = 0, 1, 2, 3
TP_DECODE, TP_PREFILL = 0, 1

STATUS_NAMES = {
    0: "TP_OK", 1: "TP_ERR_ARG", 2: "TP_ERR_DIVISIBILITY", 3: "TP_ERR_KV_REPLICA",
    4: "TP_ERR_TOKEN_RANGE", 5: "TP_ERR_OOM", 6: "TP_ERR_CUDA", 7: "TP_ERR_DEVICE_TIMEOUT",
    8: "TP_ERR_UNSUPPORTED", 9: "TP_ERR_WORKSPACE",
}
STATUS = {v: k for k, v in STATUS_NAMES.items()}


class tp_config_t(Structure):
    _fields_ = [(n, c_int32) for n in ("hidden", "n_heads", "n_kv_heads", "head_dim", "intermediate",
                                       "vocab", "n_layers", "t")] + \
               [("rms_eps", c_float), ("rope_theta", c_float), ("max_positions", c_int32),
                ("attn_dp", c_int32), ("host_io", c_int32), ("plain_column_shards", c_int32),
                ("prefill_bn", c_int32), ("prefill_cta_pairs", c_int32)] + \
               [(n, c_int32) for n in ("vocab_padded", "vocab_per_rank", "q_heads_per_rank",
                                       "kv_heads_per_rank", "kv_replicas", "kv_copies",
                                       "inter_per_rank", "attn_tp")]


class tp_layer_weights_t(Structure):
    _fields_ = [(n, c_void_p) for n in ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu",
                                        "wd", "bq", "bk", "bv", "bo", "bg", "bu", "bd")]


class tp_weights_t(Structure):
    _fields_ = [("embed", c_void_p), ("final_norm", c_void_p), ("lm_head", c_void_p),
                ("layers", POINTER(tp_layer_weights_t))]


class tp_batch_t(Structure):
    _fields_ = [("mode", c_int32), ("n_seqs", c_int32), ("n_tokens", c_int32),
                ("max_q_per_seq", c_int32), ("max_ctx", c_int32), ("l_max", c_int32),
                ("seq_start", c_void_p), ("positions", c_void_p), ("token_seq", c_void_p),
                ("k_cache", POINTER(c_void_p)), ("v_cache", POINTER(c_void_p)),
                ("sample_rows", c_void_p), ("n_samples", c_int32)]


class tp_stats_t(Structure):
    _fields_ = [(n, c_int64) for n in ("allreduces", "allreduce_payload_bytes", "allgathers",
                                       "allgather_recv_bytes_per_rank", "kernel_launches",
                                       "stage_sends", "stage_send_bytes", "dp_gathers",
                                       "dp_gather_recv_bytes_per_rank")]


class tp_kernel_time_t(Structure):
    _fields_ = [("name", ctypes.c_char * 24), ("launches", c_int64), ("total_ms", ctypes.c_double)]


class TPError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({strerror(status)})")


_lib = None

# name -> (restype, argtypes)
_SIGS = {
    "tp_config": (c_int32, [POINTER(tp_config_t)]),
    "tp_load_shards": (c_int32, [POINTER(tp_config_t), POINTER(tp_weights_t), c_void_p,
                                 POINTER(c_void_p)]),
    "tp_free": (None, [c_void_p]),
    "tp_get_config": (c_int32, [c_void_p, POINTER(tp_config_t)]),
    "tp_model_bytes": (c_int32, [c_void_p, POINTER(c_int64)]),
    "tp_workspace_bytes": (c_size_t, [c_void_p, c_int32]),
    "tp_workspace_init": (c_int32, [c_void_p, c_size_t, c_void_p]),
    "tp_column_linear": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_int32, c_void_p, c_int64,
                                   c_void_p, c_size_t, c_void_p]),
    "tp_row_linear_reduce": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_int64, c_int64,
                                       c_int32, c_void_p, c_void_p, c_int32, c_void_p, c_size_t,
                                       c_void_p]),
    "tp_vocab_embed": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_void_p]),
    "tp_lm_head_gather": (c_int32, [c_void_p, c_void_p, c_int32, c_void_p, c_int64, c_void_p,
                                    c_size_t, c_void_p]),
    "tp_layer_forward": (c_int32, [c_void_p, c_int32, POINTER(tp_batch_t), c_void_p, c_int32,
                                   c_void_p, c_size_t, c_void_p]),
    "tp_layer_forward_host": (c_int32, [c_void_p, c_int32, POINTER(tp_batch_t), c_void_p, c_void_p,
                                        c_void_p, c_int32, c_void_p, c_size_t, c_void_p]),
    "tp_forward": (c_int32, [c_void_p, c_void_p, POINTER(tp_batch_t), c_void_p, c_void_p, c_int64,
                             c_int32, c_void_p, c_size_t, c_void_p]),
    "tp_stage_forward": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, POINTER(tp_batch_t),
                                   c_void_p, c_void_p, c_int64, c_int32, c_void_p, c_size_t,
                                   c_void_p]),
    "tp_stage_send": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_void_p]),
    "tp_graph_capture_forward": (c_int32, [c_void_p, c_void_p, POINTER(tp_batch_t), c_void_p,
                                           c_void_p, c_int64, c_int32, c_void_p, c_size_t,
                                           c_void_p, POINTER(c_void_p)]),
    "tp_graph_capture_layer": (c_int32, [c_void_p, c_int32, POINTER(tp_batch_t), c_void_p, c_int32,
                                         c_void_p, c_size_t, c_void_p, POINTER(c_void_p)]),
    "tp_graph_launch": (c_int32, [c_void_p, c_void_p]),
    "tp_graph_free": (None, [c_void_p]),
    "tp_row_linear_reduce_noalloc": (c_int32, [c_void_p, c_int32, c_int32, c_void_p, c_int64,
                                               c_int64, c_int32, c_void_p, c_void_p, c_void_p]),
    "tp_row_linear_reduce_noalloc_fits": (c_int32, [c_int32, c_int32, c_int32]),
    "tp_rmsnorm": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p]),
    "tp_get_stats": (c_int32, [c_void_p, POINTER(tp_stats_t)]),
    "tp_reset_stats": (None, [c_void_p]),
    "tp_check_device": (c_int32, [c_void_p, c_void_p]),
    "tp_selftest_wait_timeout": (c_int32, [c_void_p, c_int32, c_void_p]),
    "tp_strerror": (c_char_p, [c_int32]),
    "tp_profile": (c_int32, [c_void_p, c_int32]),
    "tp_profile_read": (c_int32, [c_void_p, c_void_p, POINTER(tp_kernel_time_t), c_int32,
                                  POINTER(c_int32)]),
}


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded C library.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"CUDA library missing: {_LIB_PATH} (run __graft_entry__.build())")
        L = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def exported_symbols():
    return list(_SIGS)


def strerror(status: int) -> str:
    return lib().tp_strerror(status).decode()


def check(status: int, where: str) -> None:
    if status != TP_OK:
        raise TPError(status, where)


# ---------------------------------------------------------------------------
# Same-named wrappers.  Pointers are ints (device addresses); `stream` is a
# cudaStream_t as int (0 = legacy default stream).
# ---------------------------------------------------------------------------
def tp_config(cfg: tp_config_t) -> int:
    return lib().tp_config(ctypes.byref(cfg))


def tp_load_shards(cfg: tp_config_t, weights: tp_weights_t, stream: int) -> int:
    out = c_void_p()
    check(lib().tp_load_shards(ctypes.byref(cfg), ctypes.byref(weights), stream, ctypes.byref(out)),
          "tp_load_shards")
    return out.value


def tp_free(model: int) -> None:
    lib().tp_free(model)


def tp_get_config(model: int) -> tp_config_t:
    c = tp_config_t()
    check(lib().tp_get_config(model, ctypes.byref(c)), "tp_get_config")
    return c


def tp_model_bytes(model: int) -> int:
    v = c_int64(0)
    check(lib().tp_model_bytes(model, ctypes.byref(v)), "tp_model_bytes")
    return v.value


def tp_workspace_bytes(model: int, max_tokens: int) -> int:
    return lib().tp_workspace_bytes(model, max_tokens)


def tp_workspace_init(ws: int, nbytes: int, stream: int) -> None:
    check(lib().tp_workspace_init(ws, nbytes, stream), "tp_workspace_init")


def tp_column_linear(model, layer, which, x, M, y, y_rank_stride, ws, ws_bytes, stream) -> int:
    return lib().tp_column_linear(model, layer, which, x, M, y, y_rank_stride, ws, ws_bytes, stream)


def tp_row_linear_reduce(model, layer, which, x, x_rank_stride, ldx, M, residual, y, fused, ws,
                         ws_bytes, stream) -> int:
    return lib().tp_row_linear_reduce(model, layer, which, x, x_rank_stride, ldx, M, residual, y,
                                      fused, ws, ws_bytes, stream)


def tp_row_linear_reduce_noalloc(model, layer, which, x, x_rank_stride, ldx, M, residual, y,
                                 stream) -> int:
    return lib().tp_row_linear_reduce_noalloc(model, layer, which, x, x_rank_stride, ldx, M,
                                              residual, y, stream)


def tp_row_linear_reduce_noalloc_fits(M, hidden, num_sms) -> int:
    return lib().tp_row_linear_reduce_noalloc_fits(M, hidden, num_sms)


def tp_vocab_embed(model, ids, M, h, stream) -> int:
    return lib().tp_vocab_embed(model, ids, M, h, stream)


def tp_lm_head_gather(model, x, S, logits, ld_logits, ws, ws_bytes, stream) -> int:
    return lib().tp_lm_head_gather(model, x, S, logits, ld_logits, ws, ws_bytes, stream)


def tp_layer_forward(model, layer, batch: tp_batch_t, h, fused, ws, ws_bytes, stream) -> int:
    return lib().tp_layer_forward(model, layer, ctypes.byref(batch), h, fused, ws, ws_bytes, stream)


def tp_layer_forward_host(model, layer, batch: tp_batch_t, h_in_host, h_out_host, h_dev, fused, ws,
                          ws_bytes, stream) -> int:
    return lib().tp_layer_forward_host(model, layer, ctypes.byref(batch), h_in_host, h_out_host,
                                       h_dev, fused, ws, ws_bytes, stream)


def tp_forward(model, ids, batch: tp_batch_t, h, logits, ld_logits, fused, ws, ws_bytes,
               stream) -> int:
    return lib().tp_forward(model, ids, ctypes.byref(batch), h, logits, ld_logits, fused, ws,
                            ws_bytes, stream)


def tp_stage_forward(model, first_layer, n_layers, ids, batch: tp_batch_t, h, logits, ld_logits,
                     fused, ws, ws_bytes, stream) -> int:
    return lib().tp_stage_forward(model, first_layer, n_layers, ids, ctypes.byref(batch), h, logits,
                                  ld_logits, fused, ws, ws_bytes, stream)


def tp_stage_send(model, src, dst, M, stream) -> int:
    return lib().tp_stage_send(model, src, dst, M, stream)


def tp_graph_capture_forward(model, ids, batch: tp_batch_t, h, logits, ld_logits, fused, ws,
                             ws_bytes, stream):
    """Returns (status, graph handle)."""
    g = c_void_p()
    st = lib().tp_graph_capture_forward(model, ids, ctypes.byref(batch), h, logits, ld_logits,
                                        fused, ws, ws_bytes, stream, ctypes.byref(g))
    return st, g.value


def tp_graph_capture_layer(model, layer, batch: tp_batch_t, h, fused, ws, ws_bytes, stream):
    """Returns (status, graph handle)."""
    g = c_void_p()
    st = lib().tp_graph_capture_layer(model, layer, ctypes.byref(batch), h, fused, ws, ws_bytes,
                                      stream, ctypes.byref(g))
    return st, g.value


def tp_graph_launch(graph, stream) -> int:
    return lib().tp_graph_launch(graph, stream)


def tp_graph_free(graph) -> None:
    lib().tp_graph_free(graph)


def tp_rmsnorm(model, x, w, M, y, stream) -> int:
    return lib().tp_rmsnorm(model, x, w, M, y, stream)


def tp_get_stats(model) -> tp_stats_t:
    s = tp_stats_t()
    check(lib().tp_get_stats(model, ctypes.byref(s)), "tp_get_stats")
    return s


def tp_reset_stats(model) -> None:
    lib().tp_reset_stats(model)


def tp_check_device(model, stream) -> int:
    return lib().tp_check_device(model, stream)


def tp_profile(model, enable: bool) -> int:
    return lib().tp_profile(model, int(enable))


def tp_profile_read(model, stream) -> dict:
    """{kernel name: (launches, total_ms)} since the last read."""
    arr = (tp_kernel_time_t * 64)()
    n = c_int32()
    check(lib().tp_profile_read(model, stream, arr, 64, ctypes.byref(n)), "tp_profile_read")
    return {arr[i].name.decode(): (arr[i].launches, arr[i].total_ms) for i in range(n.value)}
