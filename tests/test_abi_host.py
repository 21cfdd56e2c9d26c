"""The C ABI on the host (no GPU needed): the library loads, exports every
symbol that include/tp.h declares, and applies the sharding rules of the pages
through tp_config with the documented status codes."""
import json
import os
import re

import pytest

import megatron_tensor_layers_tp_gb300.binding as B
from megatron_tensor_layers_tp_gb300.runtime import make_config

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "tp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tp_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = B.lib()
    declared = _declared_symbols()
    assert "tp_layer_forward" in declared and len(declared) >= 15
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(B.exported_symbols()) == declared


def _cfg(n_heads, n_kv, inter, vocab, t, hidden=None, head_dim=128):
    hidden = hidden or n_heads * head_dim
    return make_config(hidden, n_heads, n_kv, head_dim, inter, vocab, 1, t)


def test_config_rules_match_the_golden_cases():
    g = json.load(open(os.path.join(GOLDEN, "sharding_rules.json")))
    for c in g["cases"]:
        if c["t"] > 8:
            continue  # outside the kernels' envelope; the rule itself is pinned in the oracle
        inter = c["intermediate"]
        cfg = _cfg(c["n_heads"], c["n_kv_heads"], inter, c["vocab"], c["t"],
                   head_dim=64 if c["n_heads"] * 64 % 64 == 0 else 128)
        st = B.tp_config(cfg)
        if st == B.STATUS["TP_ERR_UNSUPPORTED"]:
            # the rule fields are filled before the envelope check
            pass
        else:
            assert st == B.TP_OK, (c, st)
        assert (cfg.q_heads_per_rank, cfg.kv_heads_per_rank, cfg.kv_replicas, cfg.vocab_padded) == \
            (c["q_per_rank"], c["kv_per_rank"], c["replicas"], c["vocab_padded"]), c
        assert cfg.vocab_per_rank * c["t"] == cfg.vocab_padded
        assert cfg.kv_copies == min(c["t"], c["n_kv_heads"])


def test_config_rejections_have_the_named_status():
    ST = B.STATUS
    assert B.tp_config(_cfg(40, 8, 27648, 152064, 3)) == ST["TP_ERR_DIVISIBILITY"]     # n_h % t
    assert B.tp_config(_cfg(32, 8, 14337, 128256, 2)) == ST["TP_ERR_DIVISIBILITY"]     # I % t
    assert B.tp_config(_cfg(48, 12, 1536, 1000, 8)) == ST["TP_ERR_KV_REPLICA"]         # n_kv % t
    assert B.tp_config(_cfg(8, 3, 1536, 1000, 2)) == ST["TP_ERR_DIVISIBILITY"]         # GQA groups
    assert B.tp_config(_cfg(20, 4, 1280, 1000, 10)) == ST["TP_ERR_KV_REPLICA"]         # t % n_kv
    assert B.tp_config(_cfg(32, 8, 14336, 128256, 16)) == ST["TP_ERR_UNSUPPORTED"]     # t > 8
    assert B.tp_config(_cfg(32, 8, 14336, 128256, 0)) == ST["TP_ERR_ARG"]
    bad = _cfg(32, 8, 14336, 128256, 2, head_dim=96)
    assert B.tp_config(bad) == ST["TP_ERR_UNSUPPORTED"]
    ok = _cfg(32, 8, 14336, 128256, 8)
    assert B.tp_config(ok) == B.TP_OK
    assert (ok.q_heads_per_rank, ok.kv_heads_per_rank, ok.inter_per_rank, ok.vocab_per_rank) == \
        (4, 1, 1792, 16032)
    for bn, want in ((0, B.TP_OK), (224, B.TP_OK), (128, B.TP_OK), (100, ST["TP_ERR_ARG"]),
                     (240, ST["TP_ERR_ARG"]), (-256, ST["TP_ERR_ARG"])):
        c = _cfg(32, 8, 14336, 128256, 8)
        c.prefill_bn = bn
        assert B.tp_config(c) == want, bn
    for mode, want in ((0, B.TP_OK), (1, B.TP_OK), (2, B.TP_OK), (3, ST["TP_ERR_ARG"]),
                       (-1, ST["TP_ERR_ARG"])):
        c = _cfg(32, 8, 14336, 128256, 8)
        c.prefill_cta_pairs = mode
        assert B.tp_config(c) == want, mode


def test_calls_without_a_model_are_rejected_on_the_host():
    ST = B.STATUS
    assert B.tp_workspace_bytes(None, 16) == 0
    assert B.tp_column_linear(None, 0, 0, 0, 16, 0, 0, 0, 0, 0) == ST["TP_ERR_ARG"]
    assert B.tp_row_linear_reduce(None, 0, 2, 0, 0, 0, 16, 0, 0, 1, 0, 0, 0) == ST["TP_ERR_ARG"]
    assert B.tp_vocab_embed(None, 0, 4, 0, 0) == ST["TP_ERR_ARG"]
    assert B.tp_lm_head_gather(None, 0, 1, 0, 0, 0, 0, 0) == ST["TP_ERR_ARG"]
    assert B.tp_rmsnorm(None, 0, 0, 1, 0, 0) == ST["TP_ERR_ARG"]
    assert B.lib().tp_layer_forward_host(None, 0, None, None, None, None, 1, None, 0, None) == \
        ST["TP_ERR_ARG"]
    assert B.lib().tp_get_stats(None, None) == ST["TP_ERR_ARG"]
    for code, name in B.STATUS_NAMES.items():
        assert B.strerror(code) and B.strerror(code) != "unknown status", name


def test_dp_attention_config_rules():
    # attention ranks per group = t / attn_dp; head and KV rules against them
    c = make_config(4096, 32, 8, 128, 14336, 1000, 1, 8, attn_dp=2)
    assert B.tp_config(c) == B.TP_OK
    assert (c.attn_tp, c.q_heads_per_rank, c.kv_heads_per_rank, c.kv_replicas, c.kv_copies,
            c.inter_per_rank) == (4, 8, 2, 1, 4, 1792)
    c = make_config(2048, 16, 1, 128, 14336, 1000, 1, 8, attn_dp=8)
    assert B.tp_config(c) == B.TP_OK
    assert (c.attn_tp, c.q_heads_per_rank, c.kv_heads_per_rank, c.kv_replicas, c.kv_copies) == \
        (1, 16, 1, 1, 1)
    c = make_config(4096, 32, 2, 128, 14336, 1000, 1, 8, attn_dp=2)
    assert B.tp_config(c) == B.TP_OK
    assert (c.attn_tp, c.kv_heads_per_rank, c.kv_replicas, c.kv_copies) == (4, 1, 2, 2)
    c = make_config(4096, 32, 8, 128, 14336, 1000, 1, 8, attn_dp=3)
    assert B.tp_config(c) == B.STATUS["TP_ERR_DIVISIBILITY"]
    c = make_config(4096, 32, 8, 128, 14336, 1000, 1, 8, attn_dp=0)
    assert B.tp_config(c) == B.TP_OK and c.attn_dp == 1 and c.attn_tp == 8
    # the same shapes from the oracle's plan
    import oracle as O
    p = O.plan(32, 8, 14336, 1000, O.attn_tp_size(8, 2))
    assert (p.q_heads_per_rank, p.kv_heads_per_rank, p.kv_replicas, p.kv_copies) == (8, 2, 1, 4)


def test_noalloc_scratch_limits():
    # the fixed scratch holds one ticket per 128-row output tile and two fp32
    # [BN][128] partial tiles per SM: up to 64 tokens, and at 64 tokens
    # (BN = 64) up to 160 SMs; fewer tokens leave room for more SMs
    fits = B.tp_row_linear_reduce_noalloc_fits
    assert fits(1, 4096, 152) == 1 and fits(64, 4096, 152) == 1 and fits(64, 5120, 160) == 1
    assert fits(65, 4096, 152) == 0            # beyond the decode orientation
    assert fits(64, 4096, 161) == 0            # 161 x 2 x 64 x 128 x 4 B > 10 MiB
    assert fits(16, 4096, 161) == 1            # BN = 16: a quarter of the partial bytes
    assert fits(16, 4096 * 1024 + 128, 152) == 0   # more than 4096 output tiles of tickets
    assert fits(-1, 4096, 152) == 0 and fits(16, 0, 152) == 0 and fits(16, 4096, 0) == 0
