"""GPU edge cases of the cache bookkeeping: overflow, rewind, stale rows, empty caches, call order.

Error codes come back through the C-ABI status; after every refused call the stream's
length is unchanged and the device status word stays clear.
"""
import numpy as np
import pytest

from kv_cached_qwen3_gb300 import inputs
from oracle import Oracle, OracleCache
from parity_util import check_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EINVAL, EOVERFLOW, ESTATE = 1, 2, 5


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


def status_of(fn, *args):
    from kv_cached_qwen3_gb300.talker import TalkerError
    try:
        fn(*args)
    except TalkerError as e:
        return e.status
    return 0


@pytest.fixture(scope="module")
def tiny():
    g = inputs.TINY
    w = inputs.make_weights(g, 41)
    return g, w, Oracle(g, w)


def test_call_order_and_overflow(cuda, tiny):
    from kv_cached_qwen3_gb300.talker import Talker
    g, w, o = tiny
    tk = Talker(g, w)
    e1 = dev(inputs.make_embeddings(g, 41, 0, 1))
    # nothing works before the cache exists
    assert status_of(tk.decode, e1) == ESTATE
    assert status_of(tk.prefill, 0, e1) == ESTATE
    tk.kv_init_batched(2, 20)
    emb = inputs.make_embeddings(g, 41, 0, 21)
    assert status_of(tk.prefill, 0, dev(emb)) == EOVERFLOW          # T > max_seq_len
    assert status_of(tk.prefill, 2, e1) == EINVAL                   # no such stream
    assert status_of(tk.decode, dev(emb[:3])) == EINVAL             # B > n_streams
    tk.prefill(0, dev(emb[:20]))
    assert tk.cur_len(0) == 20
    assert status_of(tk.decode, e1) == EOVERFLOW                    # stream 0 is full
    assert tk.cur_len(0) == 20 and tk.cur_len(1) == 0
    assert status_of(tk.rewind, 0, 21) == EINVAL                    # rewind only shortens
    assert status_of(tk.rewind, 0, -1) == EINVAL
    kt = torch.zeros(g.n_layers, g.n_kv_heads, 21, g.head_dim, device="cuda")
    assert status_of(tk.kv_import, 1, kt, kt, 21) == EOVERFLOW
    tk.rewind(0, 19)
    lg, _, _ = tk.decode(e1)                                        # now it fits again
    assert tk.cur_len(0) == 20
    assert np.all(np.isfinite(host(lg)))
    assert tk.sync_status() == 0
    tk.close()


def poisoned_cache(g, seed, L, extra, n_layers):
    """Cache rows [0, L) seeded, rows [L, L + extra) NaN."""
    ks, vs = [], []
    for l in range(n_layers):
        k, v = inputs.make_kv_layer(g, seed, l, L + extra)
        k[:, L:] = np.nan
        v[:, L:] = np.nan
        ks.append(k)
        vs.append(v)
    return np.stack(ks), np.stack(vs)


@pytest.mark.parametrize("L", [0, 1, 63, 64, 65, 128, 150])
@pytest.mark.parametrize("mode", [pytest.param(0, id="auto"), pytest.param(2, id="graph")])
def test_stale_rows_past_length_never_read_fp32(cuda, tiny, L, mode):
    """NaN rows beyond the rewound length (same page and next pages) leave decode unchanged."""
    from kv_cached_qwen3_gb300.talker import Talker
    g, w, o = tiny
    extra = 70
    K, V = poisoned_cache(g, 42, L, extra, g.n_layers)
    tk = Talker(g, w)
    tk.set_decode_mode(mode)
    tk.kv_init_batched(1, L + extra)
    tk.kv_import(0, dev(K), dev(V), L + extra)
    tk.rewind(0, L)
    oc = OracleCache(o, 1, L + extra)
    oc.kv_import(0, K[:, :, :L], V[:, :, :L], L)
    for t in range(3):
        emb = inputs.make_embeddings(g, 43, t, t + 1)
        lg = torch.empty(1, g.vocab, device="cuda")
        hd = torch.empty(1, g.hidden, device="cuda")
        tk.decode(dev(emb), lg, hd)
        rh, rl = oc.decode(emb)
        check_rows(host(hd), rh, bf16=False, what="L=%d step %d hidden" % (L, t))
        check_rows(host(lg), rl, bf16=False, what="L=%d step %d logits" % (L, t))
    assert tk.cur_len(0) == L + 3
    assert tk.sync_status() == 0
    tk.close()


@pytest.mark.parametrize("mode", [pytest.param(2, id="graph"), pytest.param(3, id="tensor-core-graph")])
def test_stale_rows_past_length_never_read_bf16(cuda, mode):
    """The same on a 2-layer bf16 Talker geometry, with a rewound length inside a page."""
    from kv_cached_qwen3_gb300.talker import Talker
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 2})
    w = inputs.make_weights(g, 44)
    L, extra = 100, 90
    K, V = poisoned_cache(g, 44, L, extra, g.n_layers)
    tk = Talker(g, w)
    tk.set_decode_mode(mode)
    tk.kv_init_batched(1, L + extra)
    tk.kv_import(0, torch.from_numpy(K).to(torch.bfloat16).cuda(), torch.from_numpy(V).to(torch.bfloat16).cuda(),
                 L + extra)
    tk.rewind(0, L)
    oc = OracleCache(Oracle(g, w), 1, L + extra)
    oc.kv_import(0, K[:, :, :L], V[:, :, :L], L)
    for t in range(2):
        emb = inputs.make_embeddings(g, 45, t, t + 1)
        lg, hd = torch.empty(1, g.vocab, device="cuda"), torch.empty(1, g.hidden, device="cuda")
        tk.decode(dev(emb), lg, hd)
        rh, rl = oc.decode(emb)
        check_rows(host(hd), rh, bf16=True, what="bf16 step %d hidden" % t)
        check_rows(host(lg), rl, bf16=True, what="bf16 step %d logits" % t)
    assert tk.sync_status() == 0
    tk.close()


def test_export_round_trip_and_prefill_rewinds(cuda, tiny):
    """Export returns what prefill wrote; a second prefill starts again from position 0."""
    from kv_cached_qwen3_gb300.talker import Talker
    g, w, o = tiny
    tk = Talker(g, w)
    tk.kv_init_batched(1, 100)
    emb = inputs.make_embeddings(g, 46, 0, 40)
    tk.prefill(0, dev(emb))
    k = torch.empty(g.n_layers, g.n_kv_heads, 40, g.head_dim, device="cuda")
    v = torch.empty_like(k)
    tk.kv_export(0, k, v, 40)
    oc = OracleCache(o, 1, 100)
    oc.prefill(0, emb)
    rk, rv = oc.kv_export(0, 40)
    check_rows(host(k).reshape(-1, g.head_dim), rk.reshape(-1, g.head_dim), bf16=False, what="exported K")
    check_rows(host(v).reshape(-1, g.head_dim), rv.reshape(-1, g.head_dim), bf16=False, what="exported V")
    _, lg, _ = tk.prefill(0, dev(emb[:5]))
    assert tk.cur_len(0) == 5
    _, rl = oc.prefill(0, emb[:5])
    check_rows(host(lg), rl, bf16=False, what="second prefill logits")
    assert tk.sync_status() == 0
    tk.close()


@pytest.mark.parametrize("wdt", ["f32", "bf16"])
def test_fused_argmax_tie_goes_to_lowest_index(cuda, wdt):
    """Two codec_head rows made identical (in different CTAs of the head kernel) give bit-equal
    maximal logits; the fused argmax of prefill and decode must return the lower index."""
    from kv_cached_qwen3_gb300.talker import Talker
    g = inputs.Geometry(**{**inputs.TINY.__dict__, "weight_dtype": wdt, "kv_dtype": wdt})
    w = inputs.make_weights(g, 47)
    emb = inputs.make_embeddings(g, 47, 0, 20)
    hid, ref_logits = Oracle(g, w).forward_full(emb[:17])
    lo, hi = 3, 200
    # rows lo and hi both = a * y15 + b * y16 with y the final hidden rows of the prefill's last
    # row (15) and of the decode row (16), solved so that both logits are 3x the largest other
    # logit at both steps: the two rows win by a wide margin and are equal bit for bit
    y15, y16 = hid[15], hid[16]
    target = 3.0 * float(np.abs(ref_logits[15:17]).max())
    G = np.array([[y15 @ y15, y16 @ y15], [y15 @ y16, y16 @ y16]])
    a, b = np.linalg.solve(G, [target, target])
    big = (a * y15 + b * y16).astype(np.float32)
    if wdt == "bf16":
        big = inputs.round_to_bf16(big)
    head = np.array(w["codec_head"], copy=True)
    head[lo] = big
    head[hi] = big
    w2 = dict(w)
    w2["codec_head"] = head
    tk = Talker(g, w2)
    tk.kv_init_batched(1, 32)
    _, lg, am = tk.prefill(0, dev(emb[:16]))
    lgh = host(lg)
    assert lgh[lo] == lgh[hi] and lgh[lo] == lgh.max()
    assert int(host(am)[0]) == lo
    out_l = torch.empty(1, g.vocab, device="cuda")
    out_a = torch.empty(1, device="cuda", dtype=torch.int32)
    tk.decode(dev(emb[16:17]), out_l, None, out_a)
    d = host(out_l)[0]
    assert d[lo] == d[hi] and d[lo] == d.max()
    assert int(out_a.cpu()[0]) == lo
    assert tk.sync_status() == 0
    tk.close()
