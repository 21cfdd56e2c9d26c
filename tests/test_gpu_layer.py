"""Decoder-layer and full-forward parity of the CUDA path against the oracle at
sizes the oracle finishes in seconds (several tiles, ragged tails, KV
replication), plus GPU-side invariants: sharded vs unsharded (t vs t=1),
decode step vs prefill row, determinism and the collective counters."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle as O  # noqa: E402
import synth  # noqa: E402
from megatron_tensor_layers_tp_gb300 import binding as B  # noqa: E402
from megatron_tensor_layers_tp_gb300.runtime import Batch  # noqa: E402
from tests.parity_utils import (build_model, make_batch, oracle_batch, oracle_caches,  # noqa: E402
                                oracle_dims, oracle_forward, oracle_layer, rel_err, to_f64)

LAYER_TOL = 2e-2
LOGIT_TOL = 5e-2


def _wl(mode, n_seqs, seq_len, ctx, hidden=512, n_heads=8, n_kv=2, head_dim=64, inter=1536,
        vocab=1001, layers=1, embed=False, norm_sigma=0.1):
    return synth.Workload(f"unit-{mode}", hidden, n_heads, n_kv, head_dim, inter, vocab, layers, (1,),
                          mode, n_seqs, seq_len, ctx, embed, seed=4, norm_weight_sigma=norm_sigma)


def _run_layer(w, t, fused=True):
    model, _, _ = build_model(w, t)
    batch, caches = make_batch(model, w)
    h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(h, w.seed, synth.tensor_id("hidden"), w.sigma_h)
    model.layer_forward(0, batch, h, fused=fused)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    return model, h, caches


def _oracle_layer(w):
    dims = oracle_dims(w)
    h = synth.host_hidden(w)
    kc, vc = oracle_caches(w, 0, range(w.n_seqs))
    out = O.layer_forward(h, oracle_layer(w, 0), kc, vc, oracle_batch(w), dims)
    return out, kc, vc


def _cache_logical(model, cache, w):
    """library layout [copies, seqs, kv_r, L, d] -> logical {b: [n_kv, L, d]}"""
    c = model.cfg
    arr = to_f64(cache)
    return {b: arr[:, b].reshape(c.kv_copies * c.kv_heads_per_rank, w.l_max, w.head_dim)
            for b in range(w.n_seqs)}


@pytest.mark.parametrize("t", [1, 2, 4, 8])
@pytest.mark.parametrize("n_kv", [8, 2, 1])
@pytest.mark.parametrize("fused", [True, False])
def test_decode_layer_matches_oracle(t, n_kv, fused):
    w = _wl("decode", n_seqs=5, seq_len=1, ctx=150, n_kv=n_kv)
    model, h, (ks, vs) = _run_layer(w, t, fused)
    ref, kc, vc = _oracle_layer(w)
    assert rel_err(to_f64(h), ref) <= LAYER_TOL
    # the new token's K/V landed in the rank caches at position ctx-1
    gk = _cache_logical(model, ks[0], w)
    for b in range(w.n_seqs):
        assert rel_err(gk[b][:, w.ctx - 1], kc[b][:, w.ctx - 1]) <= LAYER_TOL
        assert np.array_equal(gk[b][:, : w.ctx - 1], kc[b][:, : w.ctx - 1])
    model.close()


@pytest.mark.parametrize("t", [1, 2, 4])
@pytest.mark.parametrize("n_heads,n_kv", [(8, 1), (12, 1), (16, 1), (16, 2)])
def test_decode_layer_query_groups_match_oracle(t, n_heads, n_kv):
    # query rows per KV head: 8 (the largest taken on the MMA N side), 12 and
    # 16 (16-row query tiles), 8 with two KV heads
    w = _wl("decode", n_seqs=5, seq_len=1, ctx=150, n_heads=n_heads, n_kv=n_kv)
    model, h, _ = _run_layer(w, t)
    ref, _, _ = _oracle_layer(w)
    assert rel_err(to_f64(h), ref) <= LAYER_TOL
    model.close()


@pytest.mark.parametrize("t", [1, 2, 4])
@pytest.mark.parametrize("head_dim,n_heads,n_kv", [(64, 8, 2), (128, 4, 4)])
def test_prefill_layer_matches_oracle(t, head_dim, n_heads, n_kv):
    w = _wl("prefill", n_seqs=3, seq_len=70, ctx=70, head_dim=head_dim, n_heads=n_heads, n_kv=n_kv)
    model, h, (ks, vs) = _run_layer(w, t)
    ref, kc, vc = _oracle_layer(w)
    assert rel_err(to_f64(h), ref) <= LAYER_TOL
    gv = _cache_logical(model, vs[0], w)
    for b in range(w.n_seqs):
        assert rel_err(gv[b], vc[b]) <= LAYER_TOL
    model.close()


def test_ragged_prefill_matches_oracle():
    w = _wl("prefill", n_seqs=3, seq_len=70, ctx=70)
    lens = [5, 70, 33]
    model, _, _ = build_model(w, 2, max_tokens=sum(lens))
    ks = [model.alloc_kv(3, 70)]
    vs = [model.alloc_kv(3, 70)]
    from tests.parity_utils import fill_device_kv
    fill_device_kv(model, w, ks[0], "k_cache", 0)
    fill_device_kv(model, w, vs[0], "v_cache", 0)
    pos = np.concatenate([np.arange(n) for n in lens]).astype(np.int32)
    seq = np.concatenate([np.full(n, b) for b, n in enumerate(lens)]).astype(np.int32)
    start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    M = sum(lens)
    batch = Batch(B.TP_PREFILL, 3, M, max(lens), max(lens), 70, torch.from_numpy(pos).cuda(),
                  torch.from_numpy(seq).cuda(), torch.from_numpy(start).cuda(), ks, vs, None)
    hx = synth.normal_f64(4, 555, (M, w.hidden), 1.0)
    h = torch.from_numpy(hx.astype(np.float32)).to(torch.bfloat16).cuda()
    model.layer_forward(0, batch, h)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    kc, vc = oracle_caches(w, 0, range(3))
    ref = O.layer_forward(hx, oracle_layer(w, 0), kc, vc, O.Batch(seq, pos), oracle_dims(w))
    assert rel_err(to_f64(h), ref) <= LAYER_TOL
    model.close()


def _ragged_prefill(w, t, lens, seed, fused=True, prefill_bn=0, prefill_cta_pairs=0):
    model, _, _ = build_model(w, t, max_tokens=sum(lens), prefill_bn=prefill_bn,
                              prefill_cta_pairs=prefill_cta_pairs)
    n = len(lens)
    ks = [model.alloc_kv(n, w.ctx)]
    vs = [model.alloc_kv(n, w.ctx)]
    from tests.parity_utils import fill_device_kv
    fill_device_kv(model, w, ks[0], "k_cache", 0)
    fill_device_kv(model, w, vs[0], "v_cache", 0)
    pos = np.concatenate([np.arange(k) for k in lens]).astype(np.int32)
    seq = np.concatenate([np.full(k, b) for b, k in enumerate(lens)]).astype(np.int32)
    start = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    M = sum(lens)
    batch = Batch(B.TP_PREFILL, n, M, max(lens), max(lens), w.ctx, torch.from_numpy(pos).cuda(),
                  torch.from_numpy(seq).cuda(), torch.from_numpy(start).cuda(), ks, vs, None)
    hx = synth.normal_f64(seed, 555, (M, w.hidden), 1.0)
    h = torch.from_numpy(hx.astype(np.float32)).to(torch.bfloat16).cuda()
    model.reset_stats()
    model.layer_forward(0, batch, h, fused=fused)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    launches = model.stats().kernel_launches
    kc, vc = oracle_caches(w, 0, range(n))
    ref = O.layer_forward(hx, oracle_layer(w, 0), kc, vc, O.Batch(seq, pos), oracle_dims(w))
    err = rel_err(to_f64(h), ref)
    model.close()
    return err, launches


@pytest.mark.parametrize("t", [1, 4])
def test_short_prefill_with_norm_inside_the_gemms_matches_oracle(t):
    # 27 tokens: the decode orientation, RMSNorm folded into qkv / gate_up,
    # causal prefill attention over ragged sequences
    w = _wl("prefill", n_seqs=3, seq_len=16, ctx=16)
    err, launches = _ragged_prefill(w, t, [3, 16, 8], 6)
    assert err <= LAYER_TOL
    assert launches == 5  # qkv, attention, o_proj, gate_up, down_proj: no norm kernel


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("lens,pairs", [([16, 16, 16], 0), ([30, 50, 60], 1), ([30, 50, 60], 2)])
def test_norm_paths_above_32_tokens(fused, lens, pairs):
    # 48 tokens (decode orientation) or 140 (prefill orientation, CTA pairs or
    # single CTAs): the first RMSNorm runs as a kernel (unit weight: its
    # weight is folded into qkv); with the fused reduction o_proj leaves the
    # sums of squares of h and gate_up applies the second norm itself, with
    # the unfused one (per-rank partials + reduction kernel) it is a kernel too
    w = _wl("prefill", n_seqs=3, seq_len=max(lens), ctx=max(lens))
    err, launches = _ragged_prefill(w, 2, lens, 7, fused=fused, prefill_cta_pairs=pairs)
    assert err <= LAYER_TOL
    assert launches == (6 if fused else 9)


@pytest.mark.parametrize("bn", [256, 224, 192, 160, 128])
@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("pairs", [2, 1])
def test_prefill_tile_widths_match_oracle(bn, fused, pairs):
    # 2100 tokens (17 row tiles of 128, 9 of 256, the last ragged) at every
    # output-feature tile width, on single CTAs (pairs=2: at t=2 gate_up has
    # 2 x 17 x ceil(1536/bn) >= 152 tiles, whole-tile waves plus a last partial
    # wave; qkv and o_proj fewer than 152, stream-K) and on CTA pairs
    # (pairs=1); widths that do not divide 384 (qkv rows per rank), 1536 or
    # 512 leave a last tile of each rank partly outside the weight
    w = _wl("prefill", n_seqs=3, seq_len=1000, ctx=1000)
    err, _ = _ragged_prefill(w, 2, [700, 1000, 400], 8, fused=fused, prefill_bn=bn,
                             prefill_cta_pairs=pairs)
    assert err <= LAYER_TOL


@pytest.mark.parametrize("t", [1, 4])
@pytest.mark.parametrize("fused", [True, False])
def test_prefill_layer_on_cta_pairs_matches_oracle(t, fused):
    # short ragged sequences (one pair tile whose odd CTA is idle) and longer
    w = _wl("prefill", n_seqs=3, seq_len=300, ctx=300)
    for lens in ([3, 70, 8], [300, 17, 260]):
        err, _ = _ragged_prefill(w, t, lens, 9, fused=fused, prefill_cta_pairs=1)
        assert err <= LAYER_TOL, lens


def test_sharded_equals_unsharded_on_gpu():
    w = _wl("decode", n_seqs=16, seq_len=1, ctx=300, hidden=1024, n_heads=16, n_kv=8, head_dim=64,
            inter=2048)
    outs = {}
    for t in (1, 2, 4, 8):
        model, h, _ = _run_layer(w, t)
        outs[t] = to_f64(h)
        model.close()
    for t in (2, 4, 8):
        assert rel_err(outs[t], outs[1]) <= 1e-2, t


def test_decode_step_equals_last_prefill_row_on_gpu():
    L = 90
    wp = _wl("prefill", n_seqs=2, seq_len=L, ctx=L)
    model, _, _ = build_model(wp, 2, max_tokens=2 * L)
    batch, (ks, vs) = make_batch(model, wp)
    h = torch.empty((2 * L, wp.hidden), dtype=torch.bfloat16, device="cuda")
    synth.fill_normal_(h, 8, 8, 1.0)
    h_in = h.clone()
    model.layer_forward(0, batch, h)
    # decode the last token of each sequence against the cache the prefill wrote
    kd, vd = ks[0].clone(), vs[0].clone()
    kd[:, :, :, L - 1] = 0
    vd[:, :, :, L - 1] = 0
    from megatron_tensor_layers_tp_gb300.runtime import decode_batch
    db = decode_batch(2, L, [kd], [vd], L)
    hd = h_in[[L - 1, 2 * L - 1]].contiguous()
    model.layer_forward(0, db, hd)
    torch.cuda.synchronize()
    assert rel_err(to_f64(hd), to_f64(h[[L - 1, 2 * L - 1]])) <= 1e-2
    model.close()


def test_layer_is_deterministic():
    w = _wl("decode", n_seqs=16, seq_len=1, ctx=500)
    a_model, a, _ = _run_layer(w, 4)
    b_model, b, _ = _run_layer(w, 4)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    a_model.close(); b_model.close()


@pytest.mark.parametrize("t", [1, 2])
def test_tiny_forward_matches_oracle(t):
    from tests.parity_utils import run_tiny_forward_check
    assert run_tiny_forward_check(t) <= LOGIT_TOL


def test_two_layer_forward_with_padded_vocab_and_counters():
    w = _wl("decode", n_seqs=6, seq_len=1, ctx=40, vocab=1001, layers=2, embed=True)
    t = 4
    model, _, _ = build_model(w, t)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    model.reset_stats()
    logits = model.forward(ids, batch)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    st = model.stats()
    assert st.allreduces == 2 * 2 + 1
    assert st.allreduce_payload_bytes == (2 * 2 + 1) * w.tokens * w.hidden * 2
    assert st.allgathers == 1
    assert st.allgather_recv_bytes_per_rank == w.n_seqs * ((t - 1) * w.vocab * 2 // t)
    ref = oracle_forward(w, ids_np)
    assert logits.shape == (w.n_seqs, w.vocab)
    assert rel_err(to_f64(logits), ref) <= LOGIT_TOL
    model.close()


@pytest.mark.parametrize("n_seqs,fused", [(6, True), (48, True), (48, False)])
def test_three_layer_forward_norm_paths_match_oracle(n_seqs, fused):
    # 6 tokens: every RMSNorm inside qkv / gate_up, from h's rows.  48
    # tokens, fused: every norm inside the GEMMs, from the sums of squares the
    # embedding (layer 0's first norm) and the fused row-parallel GEMMs leave.
    # 48 unfused: every norm a kernel but layer 0's first.
    w = _wl("decode", n_seqs=n_seqs, seq_len=1, ctx=40, vocab=1001, layers=3, embed=True)
    t = 4
    model, _, _ = build_model(w, t)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    model.reset_stats()
    logits = model.forward(ids, batch, fused=fused)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    per_layer = 5 if fused else 7  # qkv, attention, o_proj, gate_up, down (+2 reductions)
    norms = 0 if n_seqs <= 32 or fused else 5
    assert model.stats().kernel_launches == 1 + 3 * per_layer + norms + 2  # embed ... head
    ref = oracle_forward(w, ids_np)
    assert rel_err(to_f64(logits), ref) <= LOGIT_TOL
    model.close()


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("pairs", [1, 2])
def test_three_layer_prefill_forward_norm_paths_match_oracle(fused, pairs):
    # 2 x 80 tokens (the prefill orientation), on CTA pairs or single CTAs.
    # Fused: every RMSNorm inside qkv / gate_up, scaled by the 1/rms from the
    # sums of squares the embedding and the fused row-parallel GEMMs leave
    # (per output tile of the prefill orientation); unfused: every norm but
    # layer 0's first a kernel.
    w = _wl("prefill", n_seqs=2, seq_len=80, ctx=80, vocab=1001, layers=3, embed=True)
    t = 2
    model, _, _ = build_model(w, t, prefill_cta_pairs=pairs)
    batch, _ = make_batch(model, w)
    ids_np = synth.token_ids(w)
    ids = torch.from_numpy(ids_np).cuda()
    model.reset_stats()
    logits = model.forward(ids, batch, fused=fused)
    torch.cuda.synchronize()
    assert model.check_device() == 0
    per_layer = 5 if fused else 7
    norms = 0 if fused else 5
    assert model.stats().kernel_launches == 1 + 3 * per_layer + norms + 2
    ref = oracle_forward(w, ids_np)
    assert rel_err(to_f64(logits), ref) <= LOGIT_TOL
    model.close()


@pytest.mark.parametrize("n_seqs", [1, 7, 16, 40])
def test_decode_layer_4096_wide_ragged_tokens_matches_oracle(n_seqs):
    # hidden 4096: o_proj and down_proj run as 32 clusters of 4 CTAs, qkv and
    # gate_up as stream-K, at 1, 7 and 16 tokens (ragged 8-column units; the
    # RMSNorms applied inside qkv / gate_up) and 40 (RMSNorm kernels first)
    w = _wl("decode", n_seqs=n_seqs, seq_len=1, ctx=64, hidden=4096, n_heads=32, n_kv=8,
            head_dim=128, inter=2048)
    model, h, _ = _run_layer(w, 8, fused=True)
    ref, _, _ = _oracle_layer(w)
    assert rel_err(to_f64(h), ref) <= LAYER_TOL
    # the unfused reduction (per-rank partials, then the ordered sum): same result
    model2, h2, _ = _run_layer(w, 8, fused=False)
    assert rel_err(to_f64(h2), to_f64(h)) <= 1e-2
    model.close(); model2.close()


@pytest.mark.parametrize("t", [1, 8])
@pytest.mark.parametrize("ctx", [1, 2, 65, 129])
def test_decode_context_edges_match_oracle(t, ctx):
    # ctx 1: the new token is the whole context (its attention output is its
    # own v); ctx 2: one cached key; ctx 65 / 129: the last 64-key tile holds
    # a single key
    w = _wl("decode", n_seqs=5, seq_len=1, ctx=ctx, n_kv=8)
    model, h, (ks, vs) = _run_layer(w, t)
    ref, kc, vc = _oracle_layer(w)
    assert rel_err(to_f64(h), ref) <= LAYER_TOL
    gv = _cache_logical(model, vs[0], w)
    for b in range(w.n_seqs):
        assert rel_err(gv[b][:, ctx - 1], vc[b][:, ctx - 1]) <= LAYER_TOL
    model.close()


def _set_cache_rows(model, cache, rows):
    """Writes logical cache rows {(b, g, p): values [d]} into the library
    layout [copies, seqs, kv_r, L, d]: KV head g sits in copy g // kv_r at
    local index g % kv_r (replica ranks share that copy)."""
    c = model.cfg
    for (b, g, p), v in rows.items():
        cache[g // c.kv_heads_per_rank, b, g % c.kv_heads_per_rank, p] = \
            torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("n_seqs", [6, 64])
def test_attention_with_one_dominant_key_matches_oracle(n_seqs):
    # In every (sequence, KV head) one cached key points along the group's
    # queries with a large norm, so its score exceeds every other by more
    # than 15: the softmax is one-hot to fp32 precision and the attention
    # output is that position's v.  A slip in the running maximum or in the
    # rescaling of the online softmax (or of the combine across CTAs) breaks
    # this at once, while the result stays insensitive to the last-bit
    # rounding differences of q.  6 sequences: each pair's key tiles are
    # split over several CTAs and combined; 64: whole pairs per CTA.
    w = _wl("decode", n_seqs=n_seqs, seq_len=1, ctx=300, n_kv=2)
    dims = oracle_dims(w)
    W = oracle_layer(w, 0)
    h = synth.host_hidden(w)
    ob = oracle_batch(w)
    nh, nkv, d = w.n_heads, w.n_kv_heads, w.head_dim
    group = nh // nkv
    u = O.round_bf16(O.rmsnorm(h, W.attn_norm, dims.rms_eps))
    q = O.round_bf16(O.rope(O.linear(u, W.wq).reshape(w.tokens, nh, d), ob.pos, dims.rope_theta))
    kc, vc = oracle_caches(w, 0, range(n_seqs))
    rows = {}
    for b in range(n_seqs):
        p = (37 * b + 11) % (w.ctx - 1)
        for g in range(nkv):
            qg = q[b, g * group:(g + 1) * group]
            dirn = qg.sum(axis=0)
            k = O.round_bf16(600.0 * dirn / np.linalg.norm(dirn))
            kc[b][g, p] = k
            rows[(b, g, p)] = k
            s = qg @ kc[b][g, : w.ctx - 1].T / np.sqrt(d)       # the cached keys' scores
            top = np.sort(s, axis=1)
            assert np.all(top[:, -1] - top[:, -2] > 15.0)        # one-hot softmax
            assert np.all(np.argmax(s, axis=1) == p)
    ref = O.layer_forward(h, W, kc, vc, ob, dims)
    for t in (1, 4):
        model, _, _ = build_model(w, t)
        batch, (ks, vs) = make_batch(model, w)
        _set_cache_rows(model, ks[0], rows)
        hd = torch.from_numpy(h.astype(np.float32)).to(torch.bfloat16).cuda()
        model.layer_forward(0, batch, hd)
        torch.cuda.synchronize()
        assert model.check_device() == 0
        assert rel_err(to_f64(hd), ref) <= LAYER_TOL, t
        model.close()


def test_unfolded_shards_kept_only_on_request():
    # non-unit norm weights: the decoder layer reads the norm-folded qkv and
    # gate_up shards; the unfolded copies tp_column_linear needs are kept only
    # with plain_column_shards = 1, and cost exactly their weight bytes
    w = _wl("decode", n_seqs=4, seq_len=1, ctx=40)
    outs, sizes = {}, {}
    for keep in (0, 1):
        model, _, _ = build_model(w, 2, plain_column_shards=keep)
        batch, _ = make_batch(model, w)
        h = torch.empty((w.tokens, w.hidden), dtype=torch.bfloat16, device="cuda")
        synth.fill_normal_(h, w.seed, synth.tensor_id("hidden"), w.sigma_h)
        model.layer_forward(0, batch, h)
        torch.cuda.synchronize()
        outs[keep], sizes[keep] = h.clone(), model.model_bytes()
        x = torch.zeros((3, w.hidden), dtype=torch.bfloat16, device="cuda")
        if keep:
            model.column_linear(0, B.TP_QKV, x)
        else:
            with pytest.raises(B.TPError) as ei:
                model.column_linear(0, B.TP_QKV, x)
            assert ei.value.status == B.STATUS["TP_ERR_UNSUPPORTED"]
        model.close()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    d = w.head_dim
    plain = ((w.n_heads + 2 * w.n_kv_heads) * d + 2 * w.intermediate) * w.hidden * 2
    assert sizes[1] - sizes[0] == plain
    # unit norm weights: folded and unfolded shards are the same buffer
    wu = replace(w, norm_weight_sigma=0.0)
    m0, _, _ = build_model(wu, 2, plain_column_shards=0)
    m1, _, _ = build_model(wu, 2, plain_column_shards=1)
    assert m0.model_bytes() == m1.model_bytes()
    m0.column_linear(0, B.TP_GATE_UP, torch.zeros((3, w.hidden), dtype=torch.bfloat16, device="cuda"))
    m0.close(); m1.close()
