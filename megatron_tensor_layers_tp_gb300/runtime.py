"""PyTorch-facing wrapper over the C ABI.

PyTorch provides device memory and streams only: every tensor here is a buffer
whose address is handed to the library, and every computation is one of the
library's kernels.  Nothing falls back to PyTorch or the CPU.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import torch

from . import binding as B


def _ptr(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_config(hidden, n_heads, n_kv_heads, head_dim, intermediate, vocab, n_layers, t,
                rms_eps=1e-5, rope_theta=10000.0, max_positions=8192,
                attn_dp=1, host_io=0, plain_column_shards=0, prefill_bn=0,
                prefill_cta_pairs=0) -> B.tp_config_t:
    c = B.tp_config_t()
    c.hidden, c.n_heads, c.n_kv_heads, c.head_dim = hidden, n_heads, n_kv_heads, head_dim
    c.intermediate, c.vocab, c.n_layers, c.t = intermediate, vocab, n_layers, t
    c.rms_eps, c.rope_theta, c.max_positions = rms_eps, rope_theta, max_positions
    c.attn_dp = attn_dp
    c.host_io = host_io
    c.plain_column_shards = plain_column_shards
    c.prefill_bn = prefill_bn
    c.prefill_cta_pairs = prefill_cta_pairs
    return c


@dataclass
class Batch:
    """Device-side description of one forward step (see tp_batch_t)."""
    mode: int
    n_seqs: int
    n_tokens: int
    max_q_per_seq: int
    max_ctx: int
    l_max: int
    positions: torch.Tensor
    token_seq: torch.Tensor
    seq_start: Optional[torch.Tensor]
    k_cache: List[torch.Tensor]
    v_cache: List[torch.Tensor]
    sample_rows: Optional[torch.Tensor] = None

    def to_c(self) -> B.tp_batch_t:
        b = B.tp_batch_t()
        b.mode, b.n_seqs, b.n_tokens = self.mode, self.n_seqs, self.n_tokens
        b.max_q_per_seq, b.max_ctx, b.l_max = self.max_q_per_seq, self.max_ctx, self.l_max
        b.seq_start = _ptr(self.seq_start)
        b.positions, b.token_seq = _ptr(self.positions), _ptr(self.token_seq)
        self._k = (ctypes.c_void_p * len(self.k_cache))(*[t.data_ptr() for t in self.k_cache])
        self._v = (ctypes.c_void_p * len(self.v_cache))(*[t.data_ptr() for t in self.v_cache])
        b.k_cache = ctypes.cast(self._k, ctypes.POINTER(ctypes.c_void_p))
        b.v_cache = ctypes.cast(self._v, ctypes.POINTER(ctypes.c_void_p))
        b.sample_rows = _ptr(self.sample_rows)
        b.n_samples = 0 if self.sample_rows is None else int(self.sample_rows.numel())
        return b


class TPModel:
    """Owns one tp_model (the t ranks' shards) plus a workspace."""

    LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wg", "wu", "wd")
    BIAS_KEYS = ("bq", "bk", "bv", "bo", "bg", "bu", "bd")

    def __init__(self, cfg: B.tp_config_t, layers: Sequence[Dict[str, torch.Tensor]],
                 embed: Optional[torch.Tensor] = None, final_norm: Optional[torch.Tensor] = None,
                 lm_head: Optional[torch.Tensor] = None, max_tokens: int = 64, stream=None):
        B.check(B.tp_config(cfg), "tp_config")
        self.cfg = cfg
        arr = (B.tp_layer_weights_t * max(len(layers), 1))()
        for i, L in enumerate(layers):
            for k in self.LAYER_KEYS:
                t = L[k]
                assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous(), k
                setattr(arr[i], k, t.data_ptr())
            for k in self.BIAS_KEYS:  # optional
                t = L.get(k)
                if t is not None:
                    assert t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous(), k
                    setattr(arr[i], k, t.data_ptr())
        w = B.tp_weights_t()
        w.embed, w.final_norm, w.lm_head = _ptr(embed), _ptr(final_norm), _ptr(lm_head)
        w.layers = ctypes.cast(arr, ctypes.POINTER(B.tp_layer_weights_t))
        self.handle = B.tp_load_shards(cfg, w, _stream(stream))
        self.max_tokens = 0
        self.ws = None
        self.ensure_workspace(max_tokens, stream)

    # ------------------------------------------------------------------ utils
    def close(self):
        if getattr(self, "handle", None):
            B.tp_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def ensure_workspace(self, max_tokens: int, stream=None):
        if max_tokens <= self.max_tokens and self.ws is not None:
            return
        n = B.tp_workspace_bytes(self.handle, max_tokens)
        self.ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        B.tp_workspace_init(self.ws.data_ptr(), n, _stream(stream))
        self.max_tokens = max_tokens

    @property
    def ws_args(self):
        return self.ws.data_ptr(), self.ws.numel()

    def alloc_kv(self, n_seqs: int, l_max: int) -> torch.Tensor:
        c = self.cfg
        return torch.empty((c.kv_copies, n_seqs, c.kv_heads_per_rank, l_max, c.head_dim),
                           dtype=torch.bfloat16, device="cuda")

    def model_bytes(self) -> int:
        return B.tp_model_bytes(self.handle)

    def check_device(self, stream=None) -> int:
        return B.tp_check_device(self.handle, _stream(stream))

    def stats(self) -> B.tp_stats_t:
        return B.tp_get_stats(self.handle)

    def reset_stats(self):
        B.tp_reset_stats(self.handle)

    def qkv_rows(self) -> int:
        c = self.cfg
        return (c.q_heads_per_rank + 2 * c.kv_heads_per_rank) * c.head_dim

    # ------------------------------------------------------------------ ops
    def column_linear(self, layer: int, which: int, x: torch.Tensor, stream=None) -> torch.Tensor:
        M = x.shape[0]
        n = self.qkv_rows() if which == B.TP_QKV else 2 * self.cfg.inter_per_rank
        ranks = self.cfg.attn_tp if which == B.TP_QKV else self.cfg.t
        y = torch.empty((ranks, M, n), dtype=torch.bfloat16, device="cuda")
        self.ensure_workspace(M, stream)
        B.check(B.tp_column_linear(self.handle, layer, which, x.data_ptr(), M, y.data_ptr(), M * n,
                                   *self.ws_args, _stream(stream)), "tp_column_linear")
        return y

    def row_linear_reduce(self, layer: int, which: int, x: torch.Tensor, residual=None,
                          fused: bool = True, out: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
        """x: [M, t*K_r] (rank r's shard in columns [r K_r, (r+1) K_r))."""
        M = x.shape[0]
        t = self.cfg.attn_tp if which == B.TP_O else self.cfg.t
        kr = x.shape[1] // t
        y = out if out is not None else torch.empty((M, self.cfg.hidden), dtype=torch.bfloat16,
                                                    device="cuda")
        self.ensure_workspace(M, stream)
        B.check(B.tp_row_linear_reduce(self.handle, layer, which, x.data_ptr(), kr, x.stride(0), M,
                                       _ptr(residual), y.data_ptr(), int(fused), *self.ws_args,
                                       _stream(stream)), "tp_row_linear_reduce")
        return y

    def vocab_embed(self, ids: torch.Tensor, stream=None) -> torch.Tensor:
        h = torch.empty((ids.numel(), self.cfg.hidden), dtype=torch.bfloat16, device="cuda")
        B.check(B.tp_vocab_embed(self.handle, ids.data_ptr(), ids.numel(), h.data_ptr(),
                                 _stream(stream)), "tp_vocab_embed")
        return h

    def lm_head_gather(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        S = x.shape[0]
        logits = torch.empty((S, self.cfg.vocab), dtype=torch.bfloat16, device="cuda")
        self.ensure_workspace(S, stream)
        B.check(B.tp_lm_head_gather(self.handle, x.data_ptr(), S, logits.data_ptr(), self.cfg.vocab,
                                    *self.ws_args, _stream(stream)), "tp_lm_head_gather")
        return logits

    def rmsnorm(self, x: torch.Tensor, w: torch.Tensor, stream=None) -> torch.Tensor:
        y = torch.empty_like(x)
        B.check(B.tp_rmsnorm(self.handle, x.data_ptr(), w.data_ptr(), x.shape[0], y.data_ptr(),
                             _stream(stream)), "tp_rmsnorm")
        return y

    def layer_forward(self, layer: int, batch: Batch, h: torch.Tensor, fused: bool = True,
                      stream=None, cbatch: Optional[B.tp_batch_t] = None) -> torch.Tensor:
        self.ensure_workspace(batch.n_tokens, stream)
        cb = cbatch if cbatch is not None else batch.to_c()
        B.check(B.tp_layer_forward(self.handle, layer, cb, h.data_ptr(), int(fused), *self.ws_args,
                                   _stream(stream)), "tp_layer_forward")
        return h

    def layer_forward_host(self, layer: int, batch: Batch, h_in_host: torch.Tensor,
                           h_out_host: torch.Tensor, h_dev: torch.Tensor, fused: bool = True,
                           stream=None, cbatch: Optional[B.tp_batch_t] = None) -> torch.Tensor:
        """tp_layer_forward_host: pinned host rows in, the layer on h_dev, host rows out."""
        self.ensure_workspace(batch.n_tokens, stream)
        cb = cbatch if cbatch is not None else batch.to_c()
        B.check(B.tp_layer_forward_host(self.handle, layer, cb, h_in_host.data_ptr(),
                                        h_out_host.data_ptr(), h_dev.data_ptr(), int(fused),
                                        *self.ws_args, _stream(stream)), "tp_layer_forward_host")
        return h_out_host

    def forward(self, ids: torch.Tensor, batch: Batch, fused: bool = True, stream=None,
                h: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                cbatch: Optional[B.tp_batch_t] = None):
        M = batch.n_tokens
        S = int(batch.sample_rows.numel())
        self.ensure_workspace(max(M, S), stream)
        if h is None:
            h = torch.empty((M, self.cfg.hidden), dtype=torch.bfloat16, device="cuda")
        if logits is None:
            logits = torch.empty((S, self.cfg.vocab), dtype=torch.bfloat16, device="cuda")
        cb = cbatch if cbatch is not None else batch.to_c()
        B.check(B.tp_forward(self.handle, ids.data_ptr(), cb, h.data_ptr(), logits.data_ptr(),
                             self.cfg.vocab, int(fused), *self.ws_args, _stream(stream)),
                "tp_forward")
        return logits


    def stage_forward(self, first_layer: int, n_layers: int, batch: Batch, h: torch.Tensor,
                      ids: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
                      fused: bool = True, stream=None,
                      cbatch: Optional[B.tp_batch_t] = None) -> torch.Tensor:
        M = batch.n_tokens
        S = int(batch.sample_rows.numel()) if batch.sample_rows is not None else 0
        self.ensure_workspace(max(M, S), stream)
        cb = cbatch if cbatch is not None else batch.to_c()
        B.check(B.tp_stage_forward(self.handle, first_layer, n_layers, _ptr(ids), cb, h.data_ptr(),
                                   _ptr(logits), self.cfg.vocab, int(fused), *self.ws_args,
                                   _stream(stream)), "tp_stage_forward")
        return h

    def stage_send(self, src: torch.Tensor, dst: torch.Tensor, stream=None) -> torch.Tensor:
        B.check(B.tp_stage_send(self.handle, src.data_ptr(), dst.data_ptr(), src.shape[0],
                                _stream(stream)), "tp_stage_send")
        return dst

    def capture_forward(self, ids: torch.Tensor, batch: Batch, h: torch.Tensor,
                        logits: torch.Tensor, stream, fused: bool = True,
                        cbatch: Optional[B.tp_batch_t] = None) -> "Graph":
        """CUDA graph of tp_forward with these buffers (see tp_graph_capture_forward)."""
        M = batch.n_tokens
        S = int(batch.sample_rows.numel())
        self.ensure_workspace(max(M, S), stream)
        cb = cbatch if cbatch is not None else batch.to_c()
        st, g = B.tp_graph_capture_forward(self.handle, ids.data_ptr(), cb, h.data_ptr(),
                                           logits.data_ptr(), self.cfg.vocab, int(fused),
                                           *self.ws_args, _stream(stream))
        B.check(st, "tp_graph_capture_forward")
        return Graph(g, keep=(ids, batch, cb, h, logits, self.ws))

    def capture_layer(self, layer: int, batch: Batch, h: torch.Tensor, stream, fused: bool = True,
                      cbatch: Optional[B.tp_batch_t] = None) -> "Graph":
        """CUDA graph of tp_layer_forward with these buffers."""
        self.ensure_workspace(batch.n_tokens, stream)
        cb = cbatch if cbatch is not None else batch.to_c()
        st, g = B.tp_graph_capture_layer(self.handle, layer, cb, h.data_ptr(), int(fused),
                                         *self.ws_args, _stream(stream))
        B.check(st, "tp_graph_capture_layer")
        return Graph(g, keep=(batch, cb, h, self.ws))


class Graph:
    """An executable graph of one captured call; keeps the captured buffers alive."""

    def __init__(self, handle, keep):
        self.handle = handle
        self._keep = keep

    def launch(self, stream=None) -> None:
        B.check(B.tp_graph_launch(self.handle, _stream(stream)), "tp_graph_launch")

    def close(self) -> None:
        if self.handle:
            B.tp_graph_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def decode_batch(n_seqs: int, ctx: int, k_cache, v_cache, l_max: Optional[int] = None,
                 with_samples: bool = True) -> Batch:
    dev = "cuda"
    pos = torch.full((n_seqs,), ctx - 1, dtype=torch.int32, device=dev)
    seq = torch.arange(n_seqs, dtype=torch.int32, device=dev)
    return Batch(B.TP_DECODE, n_seqs, n_seqs, 1, ctx, l_max or ctx, pos, seq, None,
                 list(k_cache), list(v_cache), seq.clone() if with_samples else None)


def prefill_batch(n_seqs: int, seq_len: int, k_cache, v_cache, l_max: Optional[int] = None) -> Batch:
    dev = "cuda"
    M = n_seqs * seq_len
    pos = torch.arange(seq_len, dtype=torch.int32, device=dev).repeat(n_seqs)
    seq = torch.arange(n_seqs, dtype=torch.int32, device=dev).repeat_interleave(seq_len)
    start = torch.arange(0, M + 1, seq_len, dtype=torch.int32, device=dev)
    samples = torch.arange(seq_len - 1, M, seq_len, dtype=torch.int32, device=dev)
    return Batch(B.TP_PREFILL, n_seqs, M, seq_len, seq_len, l_max or seq_len, pos, seq, start,
                 list(k_cache), list(v_cache), samples)
