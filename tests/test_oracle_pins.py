"""Pins of the fp64 oracle against closed forms, invariants and library routines.

Each test targets one step of the forward so that a plausible slip (a dropped
term, a wrong sign or index, a transposed operand, eps outside the square root,
the wrong RoPE pairing, gate/up swapped, a modulo GQA mapping, a stale cache
row) fails at least one of them. None of these checks calls the CUDA library.
"""
import math
import os

import numpy as np
import pytest
import torch

from oracle import Oracle, OracleCache, attend_one, rms_norm, rope_neox, silu, softmax
from kv_cached_qwen3_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.txt")


def golden():
    out = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, _, vals = [p.strip() for p in line.split("|")]
            out[name] = np.array([float(v) for v in vals.split()])
    return out


G = golden()


# ----------------------------------------------------------------------------- RMSNorm

def test_rms_norm_closed_form():
    np.testing.assert_allclose(rms_norm([3.0, 4.0], [1.0, 1.0], 0.0), G["rms_norm_34"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(rms_norm([3.0, 4.0], [2.0, 2.0], 0.0), G["rms_norm_gain2"], rtol=0, atol=1e-15)


def test_rms_norm_eps_inside_sqrt():
    out = rms_norm(np.full(8, 1e-3), np.ones(8), 1e-6)
    np.testing.assert_allclose(out, np.full(8, G["rms_norm_eps"][0]), rtol=1e-15)


def test_rms_norm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((7, 128))
    y = rms_norm(x, np.ones(128), 1e-6)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, -1)), 1.0, atol=1e-5)
    np.testing.assert_allclose(rms_norm(37.0 * x, np.ones(128), 1e-6), y, rtol=1e-6)
    w = rng.standard_normal(128)
    np.testing.assert_allclose(rms_norm(x, w, 1e-6), y * w, rtol=1e-14)


# ----------------------------------------------------------------------------- RoPE

@pytest.mark.parametrize("name,x,p", [
    ("rope_e0_p1", [1, 0, 0, 0], 1), ("rope_e1_p1", [0, 1, 0, 0], 1), ("rope_e2_p1", [0, 0, 1, 0], 1),
    ("rope_e0_p2", [1, 0, 0, 0], 2), ("rope_e3_p2", [0, 0, 0, 1], 2)])
def test_rope_closed_form_hd4(name, x, p):
    out = rope_neox(np.array(x, float)[None, None, :], np.array([p]), 1e6)[0, 0]
    np.testing.assert_allclose(out, G[name], rtol=0, atol=1e-15)


def test_rope_identity_at_zero_and_norm_preserving():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, 128))
    np.testing.assert_array_equal(rope_neox(x, np.zeros(5), 1e6), x)
    pos = np.array([1, 7, 100, 4095, 32767])
    y = rope_neox(x, pos, 1e6)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_relative_position():
    """<R_p q, R_p' k> depends only on p - p'."""
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 1, 64))
    k = rng.standard_normal((1, 1, 64))
    for p, pp, d in [(5, 2, 11), (100, 0, 3000), (17, 17, 999)]:
        a = np.sum(rope_neox(q, np.array([p]), 1e6) * rope_neox(k, np.array([pp]), 1e6))
        b = np.sum(rope_neox(q, np.array([p + d]), 1e6) * rope_neox(k, np.array([pp + d]), 1e6))
        assert abs(a - b) < 1e-10


# ----------------------------------------------------------------------------- SwiGLU

def test_silu_closed_form():
    assert silu(1.0) * 2.0 == pytest.approx(G["swiglu_g1_u2"][0], abs=1e-15)
    assert silu(0.5) / 0.5 == pytest.approx(G["silu_half_over_half"][0], abs=1e-15)
    assert abs(silu(-40.0)) < 1e-15 and silu(40.0) == pytest.approx(40.0, rel=1e-15)


def _mlp_probe_oracle(c):
    """One layer of width 4 whose MLP computes x[1] += silu(2c) * 2 for x = [2, 0, 0, 0]."""
    g = inputs.Geometry(n_layers=1, hidden=4, n_q_heads=1, n_kv_heads=1, head_dim=4, intermediate=1,
                        vocab=4, rms_eps=0.0, weight_dtype="f32", kv_dtype="f32")
    lw = {"input_norm": np.ones(4), "q_proj": np.eye(4), "k_proj": np.eye(4), "v_proj": np.eye(4),
          "q_norm": np.ones(4), "k_norm": np.ones(4), "o_proj": np.zeros((4, 4)), "post_norm": np.ones(4),
          "gate_proj": np.array([[c, 0, 0, 0]], float), "up_proj": np.array([[1.0, 0, 0, 0]]),
          "down_proj": np.array([[0.0], [1.0], [0.0], [0.0]])}
    return Oracle(g, {"layers": [lw], "final_norm": np.ones(4), "codec_head": np.eye(4)})


def test_swiglu_gate_and_up_not_swapped():
    x = np.array([[2.0, 0, 0, 0]])
    attn = np.zeros((1, 4))
    # gate = 2c, up = 2: silu(gate) * up.
    out = _mlp_probe_oracle(0.5).post_attention(0, x, attn)
    np.testing.assert_allclose(out[0], [2.0, G["swiglu_g1_u2"][0], 0, 0], atol=1e-15)
    # A strongly negative gate closes the MLP even though up is large (gate * silu(up) would not).
    out = _mlp_probe_oracle(-20.0).post_attention(0, x, attn)
    assert abs(out[0, 1]) < 1e-12
    out = _mlp_probe_oracle(20.0).post_attention(0, x, attn)
    assert out[0, 1] == pytest.approx(80.0, rel=1e-12)


# ----------------------------------------------------------------------------- attention

def test_attention_single_key_returns_v():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((4, 32))
    K = rng.standard_normal((2, 5, 32))
    V = rng.standard_normal((2, 5, 32))
    out = attend_one(q, K, V, 1)
    np.testing.assert_array_equal(out, V[[0, 0, 1, 1], 0])


def test_attention_zero_query_gives_mean_of_window():
    rng = np.random.default_rng(4)
    K = rng.standard_normal((2, 9, 32))
    V = rng.standard_normal((2, 9, 32))
    out = attend_one(np.zeros((4, 32)), K, V, 6)
    np.testing.assert_allclose(out, V[[0, 0, 1, 1], :6].mean(axis=1), rtol=1e-14)


def test_attention_scale_two_keys_closed_form():
    """Two keys with scores a/sqrt(hd) and 0: weight of key 0 = 1 / (1 + exp(-a / sqrt(hd)))."""
    hd, a = 16, 3.0
    q = np.zeros((1, hd))
    q[0, 0] = a
    K = np.zeros((1, 2, hd))
    K[0, 0, 0] = 1.0
    V = np.zeros((1, 2, hd))
    V[0, 0, 0], V[0, 1, 1] = 1.0, 1.0
    out = attend_one(q, K, V, 2)
    w0 = 1.0 / (1.0 + math.exp(-a / math.sqrt(hd)))
    np.testing.assert_allclose(out[0, :2], [w0, 1 - w0], rtol=1e-14)


def _bruteforce_attention(q, K, V, n_visible, group):
    """Pure-Python loops: scores, max, exp, normalise, weighted sum (tiny shapes only)."""
    n_q, hd = len(q), len(q[0])
    out = []
    for h in range(n_q):
        g = h // group
        sc = []
        for j in range(n_visible):
            sc.append(sum(q[h][d] * K[g][j][d] for d in range(hd)) / math.sqrt(hd))
        m = max(sc)
        e = [math.exp(s - m) for s in sc]
        z = sum(e)
        out.append([sum(e[j] / z * V[g][j][d] for j in range(n_visible)) for d in range(hd)])
    return np.array(out)


def test_attention_matches_bruteforce_loops():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((4, 8))
    K = rng.standard_normal((2, 7, 8))
    V = rng.standard_normal((2, 7, 8))
    for n in (1, 3, 7):
        np.testing.assert_allclose(attend_one(q, K, V, n),
                                   _bruteforce_attention(q.tolist(), K.tolist(), V.tolist(), n, 2), rtol=1e-12)


def test_attention_matches_torch_sdpa_causal_gqa():
    """Mode-A attention on one layer against torch SDPA (fp64, explicit repeat_interleave)."""
    rng = np.random.default_rng(7)
    T, nq, nkv, hd = 11, 4, 2, 32
    q = rng.standard_normal((T, nq, hd))
    k = rng.standard_normal((T, nkv, hd))
    v = rng.standard_normal((T, nkv, hd))
    # Oracle: per-row cached attention over [0, t].
    Kc, Vc = k.transpose(1, 0, 2), v.transpose(1, 0, 2)
    ours = np.stack([attend_one(q[t], Kc, Vc, t + 1) for t in range(T)])
    tq = torch.from_numpy(q).permute(1, 0, 2)[None]
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(nq // nkv, dim=0)[None]
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(nq // nkv, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)[0].permute(1, 0, 2)
    np.testing.assert_allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_softmax_masked_entries_are_zero():
    p = softmax(np.array([[1.0, 2.0, -np.inf, -np.inf]]))
    assert p[0, 2] == 0.0 and p[0, 3] == 0.0
    np.testing.assert_allclose(p[0, :2], [1 / (1 + math.e), math.e / (1 + math.e)], rtol=1e-15)


# ----------------------------------------------------------------------------- model-level invariants

TINY = inputs.TINY


@pytest.fixture(scope="module")
def tiny():
    w = inputs.make_weights(TINY, 0)
    return w, Oracle(TINY, w)


def test_gqa_equals_repeated_heads(tiny):
    """n_kv = n_q with K/V weights repeated head by head (repeat_interleave) gives the GQA output."""
    w, o = tiny
    g = TINY
    grp = g.n_q_heads // g.n_kv_heads
    w2 = {"layers": [], "final_norm": w["final_norm"], "codec_head": w["codec_head"]}
    for lw in w["layers"]:
        lw2 = dict(lw)
        for name in ("k_proj", "v_proj"):
            heads = lw[name].reshape(g.n_kv_heads, g.head_dim, g.hidden)
            lw2[name] = np.repeat(heads, grp, axis=0).reshape(g.n_q_heads * g.head_dim, g.hidden)
        w2["layers"].append(lw2)
    g2 = inputs.Geometry(**{**g.__dict__, "n_kv_heads": g.n_q_heads})
    emb = inputs.make_embeddings(g, 0, 0, 9)
    _, la = o.forward_full(emb)
    _, lb = Oracle(g2, w2).forward_full(emb)
    np.testing.assert_allclose(la, lb, rtol=1e-11, atol=1e-12)


def test_zero_o_and_down_make_layers_identity(tiny):
    w, _ = tiny
    w0 = {"layers": [], "final_norm": w["final_norm"], "codec_head": w["codec_head"]}
    for lw in w["layers"]:
        lw0 = dict(lw)
        lw0["o_proj"] = np.zeros_like(lw["o_proj"])
        lw0["down_proj"] = np.zeros_like(lw["down_proj"])
        w0["layers"].append(lw0)
    o0 = Oracle(TINY, w0)
    emb = inputs.make_embeddings(TINY, 0, 0, 5)
    hid, logits = o0.forward_full(emb)
    x = np.asarray(emb, np.float64)
    y = x / np.sqrt(np.mean(x * x, -1, keepdims=True) + TINY.rms_eps) * w["final_norm"]
    np.testing.assert_allclose(hid, y, rtol=1e-13)
    np.testing.assert_allclose(logits, y @ np.asarray(w["codec_head"], np.float64).T, rtol=1e-12, atol=1e-13)


def test_qk_norm_is_per_head(tiny):
    """Scaling one q head's projection rows (or all of k_proj) leaves the output unchanged (eps = 0)."""
    w, _ = tiny
    g = inputs.Geometry(**{**TINY.__dict__, "rms_eps": 0.0})
    o = Oracle(g, w)
    w2 = {"layers": [], "final_norm": w["final_norm"], "codec_head": w["codec_head"]}
    for lw in w["layers"]:
        lw2 = dict(lw)
        qp = lw["q_proj"].astype(np.float64).copy()
        qp[: g.head_dim] *= 13.0
        lw2["q_proj"] = qp
        lw2["k_proj"] = lw["k_proj"].astype(np.float64) * 0.25
        w2["layers"].append(lw2)
    emb = inputs.make_embeddings(g, 0, 0, 6)
    _, la = o.forward_full(emb)
    _, lb = Oracle(g, w2).forward_full(emb)
    np.testing.assert_allclose(la, lb, rtol=1e-11, atol=1e-12)
    # The same scaling without a per-head norm would change the output: check the probe bites.
    w3 = {"layers": [dict(lw, q_norm=lw["q_norm"] * 2.0) for lw in w["layers"]],
          "final_norm": w["final_norm"], "codec_head": w["codec_head"]}
    _, lc = Oracle(g, w3).forward_full(emb)
    assert np.max(np.abs(lc - la)) > 1e-3


def test_causality(tiny):
    _, o = tiny
    emb = inputs.make_embeddings(TINY, 0, 0, 8)
    _, la = o.forward_full(emb)
    emb2 = emb.copy()
    emb2[5] += 3.0
    _, lb = o.forward_full(emb2)
    np.testing.assert_array_equal(la[:5], lb[:5])
    assert np.max(np.abs(la[5:] - lb[5:])) > 1e-3


def test_cached_equals_uncached(tiny):
    """Mode B (prefill T then sequential decodes) equals mode A (full recompute) row by row."""
    _, o = tiny
    T0, n_dec = 16, 16
    emb = inputs.make_embeddings(TINY, 0, 0, T0 + n_dec)
    hid_a, log_a = o.forward_full(emb)
    c = OracleCache(o, 1, 64)
    h, lg = c.prefill(0, emb[:T0])
    np.testing.assert_allclose(lg, log_a[T0 - 1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h, hid_a[T0 - 1], rtol=1e-12, atol=1e-13)
    for t in range(n_dec):
        h, lg = c.decode(emb[T0 + t:T0 + t + 1])
        np.testing.assert_allclose(lg[0], log_a[T0 + t], rtol=1e-12, atol=1e-13)
    assert c.cur_len[0] == T0 + n_dec


def test_chunked_append_equals_prefill(tiny):
    _, o = tiny
    emb = inputs.make_embeddings(TINY, 0, 0, 20)
    c = OracleCache(o, 1, 32)
    c.prefill(0, emb[:7])
    _, lg = c.append_rows(0, emb[7:20])
    _, la = o.forward_full(emb)
    np.testing.assert_allclose(lg, la[7:20], rtol=1e-12, atol=1e-13)


def test_batched_streams_are_independent(tiny):
    _, o = tiny
    e0 = inputs.make_embeddings(TINY, 0, 0, 12, stream=0)
    e1 = inputs.make_embeddings(TINY, 0, 0, 12, stream=1)
    c = OracleCache(o, 2, 32)
    c.prefill(0, e0[:5])
    c.prefill(1, e1[:9])
    _, lg = c.decode(np.stack([e0[5], e1[9]]))
    _, la0 = o.forward_full(e0[:6])
    _, la1 = o.forward_full(e1[:10])
    np.testing.assert_allclose(lg[0], la0[-1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lg[1], la1[-1], rtol=1e-12, atol=1e-13)
    assert c.cur_len == [6, 10]


def test_rewind_then_decode(tiny):
    _, o = tiny
    emb = inputs.make_embeddings(TINY, 0, 0, 12)
    other = inputs.make_embeddings(TINY, 0, 0, 3, stream=5)
    c = OracleCache(o, 1, 32)
    c.prefill(0, emb[:8])
    for r in other:                     # three rows that the rewind discards
        c.decode(r[None])
    c.rewind(0, 8)
    _, lg = c.decode(emb[8:9])
    _, la = o.forward_full(emb[:9])
    np.testing.assert_allclose(lg[0], la[-1], rtol=1e-12, atol=1e-13)
    with pytest.raises(ValueError):
        c.rewind(0, 10)


def test_overflow_leaves_state_unchanged(tiny):
    _, o = tiny
    c = OracleCache(o, 1, 4)
    emb = inputs.make_embeddings(TINY, 0, 0, 5)
    with pytest.raises(ValueError):
        c.prefill(0, emb)
    c.prefill(0, emb[:4])
    with pytest.raises(ValueError):
        c.decode(emb[4:5])
    assert c.cur_len == [4]


def test_export_import_roundtrip(tiny):
    _, o = tiny
    emb = inputs.make_embeddings(TINY, 0, 0, 10)
    c = OracleCache(o, 1, 32)
    c.prefill(0, emb[:9])
    k, v = c.kv_export(0, 9)
    c2 = OracleCache(o, 1, 32)
    c2.kv_import(0, k, v, 9)
    _, l1 = c.decode(emb[9:10])
    _, l2 = c2.decode(emb[9:10])
    np.testing.assert_array_equal(l1, l2)


def test_padded_cache_tail_is_ignored(tiny):
    """NaN in cache rows past cur_len changes nothing (the padded tail contributes nothing)."""
    _, o = tiny
    emb = inputs.make_embeddings(TINY, 0, 0, 9)
    c = OracleCache(o, 1, 32)
    c.prefill(0, emb[:8])
    c.K[0][:, :, 8:] = np.nan
    c.V[0][:, :, 8:] = np.nan
    _, lg = c.decode(emb[8:9])
    _, la = o.forward_full(emb)
    np.testing.assert_allclose(lg[0], la[-1], rtol=1e-12, atol=1e-13)


def test_generator_is_deterministic_and_chunk_independent():
    a = inputs.make_embeddings(TINY, 3, 10, 80)
    b = inputs.make_embeddings(TINY, 3, 0, 100)
    np.testing.assert_array_equal(a, b[10:80])
    w1 = inputs.make_weights(TINY, 0)
    w2 = inputs.make_weights(TINY, 0)
    np.testing.assert_array_equal(w1["layers"][1]["up_proj"], w2["layers"][1]["up_proj"])
    assert abs(np.std(w1["layers"][0]["gate_proj"]) - 0.02) < 0.001
    assert abs(np.mean(w1["layers"][0]["input_norm"]) - 1.0) < 0.02


def test_bf16_weights_are_representable():
    g = inputs.Geometry(n_layers=1, hidden=64, n_q_heads=2, n_kv_heads=1, head_dim=32, intermediate=96,
                        vocab=32)
    w = inputs.make_weights(g, 9)
    a = w["layers"][0]["q_proj"]
    assert np.all((a.view(np.uint32) & 0xFFFF) == 0)


def test_lazy_cache_decode_equals_cached_decode(tiny):
    """decode_row_lazy_cache against OracleCache.decode on an imported cache."""
    from oracle import decode_row_lazy_cache
    _, o = tiny
    g = TINY
    L = 37
    layers = [inputs.make_kv_layer(g, 5, l, L) for l in range(g.n_layers)]
    c = OracleCache(o, 1, 64)
    c.kv_import(0, np.stack([k for k, _ in layers]), np.stack([v for _, v in layers]), L)
    x = inputs.make_embeddings(g, 5, 0, 1)
    h1, l1 = c.decode(x)
    h2, l2 = decode_row_lazy_cache(o, x[0], L, lambda l: layers[l])
    np.testing.assert_allclose(l2, l1[0], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(h2, h1[0], rtol=1e-13, atol=1e-14)


def test_embed_codes_hand_example():
    """Group-major ids: slot n sums row ids[g, n] of every table, plus its overlay row."""
    from oracle import embed_codes
    t0 = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0]])   # codec table, V=3, H=2
    t1 = np.array([[0.5, -0.5], [3.0, 4.0]])                    # acoustic table 1, V=2
    t2 = np.array([[7.0, 0.0], [0.0, 7.0], [1.0, 1.0], [2.0, 2.0]])
    ids = np.array([[2, 0], [1, 0], [3, 1]])                    # [G=3, N=2]
    ov = np.array([[0.25, 0.25], [-1.0, 1.0]])
    x = embed_codes([t0, t1, t2], ids, ov)
    np.testing.assert_array_equal(x, [[100 + 3 + 2 + 0.25, 200 + 4 + 2 + 0.25],
                                      [1 + 0.5 + 0 - 1.0, 2 - 0.5 + 7 + 1.0]])
    np.testing.assert_array_equal(embed_codes([t0], np.array([[1, 1]])), [[10, 20], [10, 20]])


def test_suppress_logits_tail_keeps_eos():
    from oracle import suppress_logits, argmax_low
    V = 3072
    lg = np.zeros(V)
    lg[V - 1] = 9.0        # in the suppressed tail, not EOS -> -inf
    lg[V - 1024] = 8.0     # first suppressed index
    lg[V - 1025] = 1.0     # last kept index below the tail
    eos = V - 500
    lg[eos] = 5.0
    out = suppress_logits(lg, 1024, eos)
    assert out[V - 1] == -np.inf and out[V - 1024] == -np.inf
    assert out[eos] == 5.0 and out[V - 1025] == 1.0
    assert np.isinf(out[V - 1024:]).sum() == 1023
    assert argmax_low(out) == eos
    # EOS below the tail: the whole tail goes
    out2 = suppress_logits(lg, 1024, 7)
    assert np.isinf(out2[V - 1024:]).all() and argmax_low(out2) == V - 1025
    # vocab smaller than the tail: everything but EOS
    small = suppress_logits(np.arange(10.0), 1024, 3)
    assert argmax_low(small) == 3 and np.isinf(small).sum() == 9


def test_argmax_low_breaks_ties_by_lowest_index():
    """The greedy token of a row with equal maxima is the lowest of their indices (the
    reading taken where the pages leave ties open), including an all-equal row and rows of
    -inf where suppression removed every other candidate."""
    from oracle import argmax_low
    assert argmax_low([1.0, 3.0, 3.0, 2.0]) == 1
    assert argmax_low([0.0, 0.0, 0.0]) == 0
    assert argmax_low([-np.inf, 2.5, -np.inf, 2.5]) == 1
    assert argmax_low([-np.inf, -np.inf]) == 0
    assert argmax_low([-1.0, -3.0, -1.0]) == 0
    v = np.full(3072, -0.5)
    v[[17, 900, 3071]] = 4.0
    assert argmax_low(v) == 17


def test_code_predictor_frame_heads_per_generation_step(tiny):
    """The frame projects its prefill with heads[0] and step i with heads[i + 1] (generation
    step i + 1 on the rightkit-qts page). Head g is zero except rows 7g (+1) and 7g + 1 (-1), so
    its greedy code is 7g or 7g + 1 whatever the hidden state: code j // 7 must equal j."""
    from oracle import OracleCache, code_predictor_frame
    w, o = tiny
    g = TINY
    n = 15
    rng = np.random.Generator(np.random.PCG64(5))
    tables = [rng.standard_normal((g.vocab, g.hidden)) for _ in range(n)]
    heads = []
    for j in range(n + 1):
        h = np.zeros((g.vocab, g.hidden))
        h[7 * j] = 1.0
        h[7 * j + 1] = -1.0
        heads.append(h)
    emb = rng.standard_normal((2, g.hidden))
    lg, codes = code_predictor_frame(OracleCache(o, 1, 20), emb, tables, list(range(n)), heads)
    assert list(codes // 7) == list(range(n + 1))
    assert lg.shape == (n + 1, g.vocab)


def test_code_predictor_frame_matches_plain_steps(tiny):
    """With every head = codec_head, the frame equals a prefill followed by decode steps whose
    input is the table row of the previous greedy code; another head equals an oracle built
    with that head as codec_head."""
    from oracle import Oracle, OracleCache, code_predictor_frame, argmax_low
    w, o = tiny
    g = TINY
    n = 4
    rng = np.random.Generator(np.random.PCG64(6))
    tables = [rng.standard_normal((g.vocab, g.hidden)) for _ in range(n)]
    emb = rng.standard_normal((3, g.hidden))
    lg, codes = code_predictor_frame(OracleCache(o, 1, 10), emb, tables, [2, 0, 3, 1], [o.codec_head] * (n + 1))
    oc = OracleCache(o, 1, 10)
    _, r = oc.prefill(0, emb)
    ref, c = [r], [argmax_low(r)]
    for i, tab in enumerate([2, 0, 3, 1]):
        _, r = oc.decode(tables[tab][c[i]][None])
        ref.append(r[0])
        c.append(argmax_low(r[0]))
    np.testing.assert_array_equal(lg, np.stack(ref))
    assert list(codes) == c
    W2 = rng.standard_normal((g.vocab, g.hidden))
    o2 = Oracle(g, {**w, "codec_head": W2})
    _, a = OracleCache(o, 1, 10).prefill(0, emb, W2)
    _, b = OracleCache(o2, 1, 10).prefill(0, emb)
    np.testing.assert_array_equal(a, b)


def test_q8_0_hand_block():
    """Block 0..31: d = 31/127 -> fp16 0.244140625; codes round(x * 127/31) half away from zero."""
    from oracle import q8_0_quantize, q8_0_dequantize
    x = np.arange(32, dtype=np.float32)
    q, d = q8_0_quantize(x)
    assert d.dtype == np.float16 and float(d[0]) == 0.244140625
    assert q[31] == 127 and q[1] == 4 and q[15] == 61 and q[16] == 66 and q[0] == 0
    deq = q8_0_dequantize(q, d)
    assert deq[31] == 127 * 0.244140625


def test_q8_0_rounds_half_away_from_zero_and_zero_block():
    from oracle import q8_0_quantize
    x = np.zeros(64, np.float32)
    x[0] = 127.0            # d = 1 exactly, so x * (1/d) = x
    x[1], x[2], x[3], x[4] = 2.5, -2.5, 0.5, -0.5
    q, d = q8_0_quantize(x)
    assert float(d[0]) == 1.0 and list(q[1:5]) == [3, -3, 1, -1]
    assert float(d[1]) == 0.0 and not q[32:].any()      # all-zero block


def test_q8_0_error_bound_random():
    """|x - dequant| <= d16 / 2 + 127 |d - d16| (rounding of the code, rounding of the scale)."""
    from oracle import q8_0_quantize, q8_0_dequantize
    rng = np.random.Generator(np.random.PCG64(7))
    x = (rng.standard_normal((50, 128)) * np.exp(rng.uniform(-4, 4, (50, 1)))).astype(np.float32)
    q, d = q8_0_quantize(x)
    err = np.abs(q8_0_dequantize(q, d) - x.astype(np.float64)).reshape(50, 4, 32)
    xb = x.reshape(50, 4, 32).astype(np.float64)
    d32 = np.max(np.abs(xb), axis=-1) / 127.0
    d16 = d.astype(np.float64)
    bound = d16 / 2 + 127 * np.abs(d32 - d16) + 1e-6 * d16
    assert np.all(err <= bound[..., None])


def test_q8_cache_attends_own_row_exactly(tiny):
    """Q8_0 storage: earlier rows dequantized, the step's own row exact, the stored row quantized."""
    from oracle import q8_0_roundtrip
    _, o = tiny
    g = TINY
    L = 20
    layers = [inputs.make_kv_layer(g, 8, l, L) for l in range(g.n_layers)]
    K = np.stack([k for k, _ in layers])
    V = np.stack([v for _, v in layers])
    x = inputs.make_embeddings(g, 8, 0, 1)
    cq = OracleCache(o, 1, 64, kv_q8=True)
    cq.kv_import(0, K, V, L)
    cp = OracleCache(o, 1, 64)
    cp.kv_import(0, q8_0_roundtrip(K), q8_0_roundtrip(V), L)
    hq, lq = cq.decode(x)
    hp, lp = cp.decode(x)
    np.testing.assert_array_equal(lq, lp)
    np.testing.assert_array_equal(hq, hp)
    kq, _ = cq.kv_export(0, L + 1)
    kp, _ = cp.kv_export(0, L + 1)
    np.testing.assert_array_equal(kq[:, :, L], q8_0_roundtrip(kp[:, :, L]))
    assert not np.array_equal(kp[:, :, L], kq[:, :, L])   # the plain cache keeps it exact


def test_q8_cache_chunk_attends_own_rows_exactly(tiny):
    """Q8_0 storage, an appended chunk of several rows: the earlier rows enter dequantized, the
    chunk's own rows (each other's keys included) exactly, and they are stored quantized. Same
    outputs as a plain cache whose earlier rows hold the Q8_0 round trip."""
    from oracle import q8_0_roundtrip
    _, o = tiny
    g = TINY
    L, T = 20, 9
    layers = [inputs.make_kv_layer(g, 9, l, L) for l in range(g.n_layers)]
    K = np.stack([k for k, _ in layers])
    V = np.stack([v for _, v in layers])
    x = inputs.make_embeddings(g, 9, 0, T)
    cq = OracleCache(o, 1, 64, kv_q8=True)
    cq.kv_import(0, K, V, L)
    cp = OracleCache(o, 1, 64)
    cp.kv_import(0, q8_0_roundtrip(K), q8_0_roundtrip(V), L)
    hq, lq = cq.append_rows(0, x)
    hp, lp = cp.append_rows(0, x)
    np.testing.assert_array_equal(lq, lp)
    np.testing.assert_array_equal(hq, hp)
    kq, vq = cq.kv_export(0, L + T)
    kp, vp = cp.kv_export(0, L + T)
    np.testing.assert_array_equal(kq[:, :, L:], q8_0_roundtrip(kp[:, :, L:]))
    np.testing.assert_array_equal(vq[:, :, L:], q8_0_roundtrip(vp[:, :, L:]))


def test_q8_0_rounding_just_below_half():
    """x * (1/d) = 0.5 - 2^-25 must round to 0 (adding 0.5 in f32 would give 1.0)."""
    from oracle import q8_0_quantize
    x = np.zeros(32, np.float32)
    x[0] = 127.0
    x[1] = np.float32(0.5) - np.float32(2.0 ** -25)
    q, d = q8_0_quantize(x)
    assert float(d[0]) == 1.0 and q[1] == 0
