"""GPU parity of the Q8_0 KV storage ("qwen3-tts" talker, TurboQuantQ8_0).

Oracle: OracleCache(kv_q8=True): a call attends the rows cached by earlier calls
dequantized (ggml Q8_0 blocks of 32, fp16 scale) and its own rows exactly.
"""
import numpy as np
import pytest

from kv_cached_qwen3_gb300 import inputs
from oracle import Oracle, OracleCache, decode_row_lazy_cache, q8_0_roundtrip
from parity_util import check_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cached_qwen3_gb300 import talker
    talker.load_library()
    return torch.device("cuda", 0)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def host(t):
    return t.detach().float().cpu().numpy()


def q8_geom(n_layers):
    return inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": n_layers, "kv_dtype": "q8_0"})


@pytest.mark.parametrize("mode", [pytest.param(2, id="graph"), pytest.param(3, id="tensor-core-graph")])
def test_q8_prefill_then_decode(cuda, mode):
    from kv_cached_qwen3_gb300.talker import Talker
    g = q8_geom(4)
    w = inputs.make_weights(g, 71)
    T0, n = 100, 4
    emb = inputs.make_embeddings(g, 71, 0, T0 + n)
    tk = Talker(g, w)
    tk.set_decode_mode(mode)
    tk.kv_init_batched(1, T0 + n + 1)
    oc = OracleCache(Oracle(g, w), 1, T0 + n + 1, kv_q8=True)
    hd, lg, am = tk.prefill(0, dev(emb[:T0]))
    rh, rl = oc.prefill(0, emb[:T0])
    check_rows(host(hd), rh[None], bf16=True, what="q8 prefill hidden")
    check_rows(host(lg), rl[None], bf16=True, what="q8 prefill logits")
    lgo, hdo = torch.empty(1, g.vocab, device="cuda"), torch.empty(1, g.hidden, device="cuda")
    for t in range(n):
        e = emb[T0 + t:T0 + t + 1]
        tk.decode(dev(e), lgo, hdo)
        rh, rl = oc.decode(e)
        check_rows(host(hdo), rh, bf16=True, what="q8 decode %d hidden" % t)
        check_rows(host(lgo), rl, bf16=True, what="q8 decode %d logits" % t)
    # the stored rows are the dequantized codes of the rows
    k = torch.empty(g.n_layers, g.n_kv_heads, T0 + n, g.head_dim, device="cuda")
    v = torch.empty_like(k)
    tk.kv_export(0, k, v, T0 + n)
    rk, rv = oc.kv_export(0, T0 + n)
    check_rows(host(k).reshape(-1, g.head_dim), rk.reshape(-1, g.head_dim), bf16=True, what="q8 exported K")
    check_rows(host(v).reshape(-1, g.head_dim), rv.reshape(-1, g.head_dim), bf16=True, what="q8 exported V")
    assert tk.sync_status() == 0
    tk.close()


def test_q8_import_codes_exact(cuda):
    """Import quantizes on the device with the oracle's Q8_0 definition: the exported values equal the
    oracle's round trip (same f32 inputs, so the codes and scales agree exactly)."""
    from kv_cached_qwen3_gb300.talker import Talker
    g = q8_geom(2)
    w = inputs.make_weights(g, 72)
    L = 150
    K = np.stack([inputs.make_kv_layer(g, 72, l, L)[0] for l in range(g.n_layers)])
    V = np.stack([inputs.make_kv_layer(g, 72, l, L)[1] for l in range(g.n_layers)])
    K[0, 0, 5] = 0.0                       # an all-zero row: scale 0, codes 0
    tk = Talker(g, w)
    tk.kv_init_batched(1, L + 1)
    tk.kv_import(0, dev(K), dev(V), L)
    k = torch.empty(g.n_layers, g.n_kv_heads, L, g.head_dim, device="cuda")
    v = torch.empty_like(k)
    tk.kv_export(0, k, v, L)
    np.testing.assert_array_equal(host(k), q8_0_roundtrip(K).astype(np.float32))
    np.testing.assert_array_equal(host(v), q8_0_roundtrip(V).astype(np.float32))
    tk.close()


@pytest.mark.parametrize("L", [8192])
def test_q8_long_context_decode(cuda, L):
    from kv_cached_qwen3_gb300.talker import Talker
    g = q8_geom(28)
    w = inputs.make_weights(g, 4)
    o = Oracle(g, w)
    nl = g.n_layers
    K = torch.empty(nl, g.n_kv_heads, L, g.head_dim, device="cuda")
    V = torch.empty_like(K)
    stored = []
    for l in range(nl):
        k, v = inputs.make_kv_layer(g, 4, l, L)
        K[l].copy_(torch.from_numpy(k))
        V[l].copy_(torch.from_numpy(v))
        stored.append((q8_0_roundtrip(k), q8_0_roundtrip(v)))
    emb = inputs.make_embeddings(g, 4, L, L + 1)
    rh, rl = decode_row_lazy_cache(o, emb[0], L, lambda l: stored[l])
    tk = Talker(g, w)
    tk.kv_init_batched(1, L + 1)
    tk.kv_import(0, K, V, L)
    del K, V
    lg, hd = torch.empty(1, g.vocab, device="cuda"), torch.empty(1, g.hidden, device="cuda")
    for mode in (2, 3):
        tk.set_decode_mode(mode)
        tk.rewind(0, L)
        tk.decode(dev(emb), lg, hd)
        check_rows(host(hd), rh[None], bf16=True, what="q8 L=%d mode %d hidden" % (L, mode))
        check_rows(host(lg), rl[None], bf16=True, what="q8 L=%d mode %d logits" % (L, mode))
    assert tk.sync_status() == 0
    tk.close()


def test_q8_refusals(cuda):
    from kv_cached_qwen3_gb300.talker import Talker, TalkerError
    g = q8_geom(1)
    for bad in ({"weight_dtype": "f32"}, {"head_dim": 32, "intermediate": 384}):
        gb = inputs.Geometry(**{**g.__dict__, **bad})
        with pytest.raises(TalkerError):
            Talker(gb, inputs.make_weights(gb, 73))
