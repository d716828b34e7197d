"""GPU parity: the CUDA library against the fp64 oracle on the same seeded inputs.

Every test calls the library through its C-ABI (ctypes binding) and compares
element by element with the oracle (tolerances in parity_util)."""
import numpy as np
import pytest

from kv_cached_qwen3_gb300 import inputs
from oracle import Oracle, OracleCache
from parity_util import assert_top1, check_rows, top1_agreement, TOL_TOP1

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


DECODE_MODES = [pytest.param(2, id="graph")]
BF16_DECODE_MODES = [pytest.param(2, id="graph"), pytest.param(3, id="tensor-core-graph")]


def run_prefill_decode(geom, weights, emb, T0, n_dec, max_seq, mode=0):
    from kv_cached_qwen3_gb300.talker import Talker
    tk = Talker(geom, weights)
    tk.set_decode_mode(mode)
    tk.kv_init_batched(1, max_seq)
    hid, lg, am = tk.prefill(0, dev(emb[:T0]))
    hids, lgs, ams = [host(hid)], [host(lg)], [int(host(am)[0])]
    assert tk.cur_len(0) == T0
    H, V = geom.hidden, geom.vocab
    out_l = torch.empty(1, V, device="cuda")
    out_h = torch.empty(1, H, device="cuda")
    out_a = torch.empty(1, device="cuda", dtype=torch.int32)
    e = torch.empty(1, H, device="cuda")
    for t in range(n_dec):
        e.copy_(dev(emb[T0 + t:T0 + t + 1]))
        tk.decode(e, out_l, out_h, out_a)
        hids.append(host(out_h)[0])
        lgs.append(host(out_l)[0])
        ams.append(int(host(out_a)[0]))
    assert tk.sync_status() == 0
    assert tk.cur_len(0) == T0 + n_dec
    tk.close()
    return np.stack(hids), np.stack(lgs), np.array(ams)


@pytest.mark.parametrize("mode", DECODE_MODES)
def test_tiny_prefill_and_decode_fp32(cuda, mode):
    wl = inputs.WORKLOADS["tiny"]
    g = wl.geometry
    w = inputs.make_weights(g, wl.seed)
    T0, n = wl.prefill_T, wl.decode_steps
    emb = inputs.make_embeddings(g, wl.seed, 0, T0 + n)
    hid, lg, am = run_prefill_decode(g, w, emb, T0, n, 64, mode)
    rh, rl = Oracle(g, w).forward_full(emb)
    check_rows(hid, rh[T0 - 1:], bf16=False, what="tiny hidden")
    check_rows(lg, rl[T0 - 1:], bf16=False, what="tiny logits")
    # the fused argmax equals the host argmax of the returned logits, bit for bit
    np.testing.assert_array_equal(am, np.argmax(lg, axis=-1))


def test_tiny_prefill_all_rows_and_ragged_lengths(cuda):
    from kv_cached_qwen3_gb300.talker import Talker
    wl = inputs.WORKLOADS["tiny"]
    g = wl.geometry
    w = inputs.make_weights(g, wl.seed)
    o = Oracle(g, w)
    tk = Talker(g, w)
    tk.kv_init_batched(1, 200)
    for T in (1, 7, 16, 17, 65, 130):     # several tiles, ragged tails, page boundaries
        emb = inputs.make_embeddings(g, 11, 0, T)
        hid, lg = tk.prefill_all_rows(0, dev(emb))
        rh, rl = o.forward_full(emb)
        check_rows(host(hid), rh, bf16=False, what="tiny all rows T=%d hidden" % T)
        check_rows(host(lg), rl, bf16=False, what="tiny all rows T=%d logits" % T)
        assert tk.cur_len(0) == T
    assert tk.sync_status() == 0


@pytest.fixture(scope="module")
def talker_b1_ref():
    wl = inputs.WORKLOADS["talker_b1"]
    g = wl.geometry
    w = inputs.make_weights(g, wl.seed)
    emb = inputs.make_embeddings(g, wl.seed, 0, wl.prefill_T + wl.decode_steps)
    rh, rl = Oracle(g, w).forward_full(emb)
    return w, emb, rh, rl


@pytest.mark.parametrize("mode", BF16_DECODE_MODES)
def test_talker_b1_prefill96_decode512_bf16(cuda, talker_b1_ref, mode):
    wl = inputs.WORKLOADS["talker_b1"]
    g = wl.geometry
    w, emb, rh, rl = talker_b1_ref
    T0, n = wl.prefill_T, wl.decode_steps
    hid, lg, am = run_prefill_decode(g, w, emb, T0, n, T0 + n, mode)
    check_rows(hid, rh[T0 - 1:], bf16=True, what="talker hidden")
    check_rows(lg, rl[T0 - 1:], bf16=True, what="talker logits")
    assert_top1(lg[1:], rl[T0:], "talker_b1 mode %d" % mode)
    np.testing.assert_array_equal(am, np.argmax(lg, axis=-1))


@pytest.mark.parametrize("T", [16, 100, 257])
def test_talker_prefill_all_rows_tensor_cores(cuda, T):
    """Tensor-core prefill (bf16 GEMMs) against the oracle on every row, ragged T across pages."""
    from kv_cached_qwen3_gb300.talker import Talker
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 4})
    w = inputs.make_weights(g, 21)
    emb = inputs.make_embeddings(g, 21, 0, T)
    tk = Talker(g, w)
    tk.kv_init_batched(1, 512)
    hid, lg = tk.prefill_all_rows(0, dev(emb))
    assert tk.sync_status() == 0
    rh, rl = Oracle(g, w).forward_full(emb)
    check_rows(host(hid), rh, bf16=True, what="tc prefill hidden T=%d" % T)
    check_rows(host(lg), rl, bf16=True, what="tc prefill logits T=%d" % T)
    # the GEMV path on the same inputs agrees as well
    tk.set_prefill_mode(2)
    hid2, lg2 = tk.prefill_all_rows(0, dev(emb))
    check_rows(host(lg2), rl, bf16=True, what="gemv prefill logits T=%d" % T)
    tk.close()


@pytest.mark.parametrize("mode", [pytest.param(2, id="gemv-graph"), pytest.param(3, id="tensor-core-graph"),
                                  pytest.param(0, id="auto")])
def test_batched16_ragged_decode(cuda, mode):
    """16 streams with ragged imported caches, 4 decode steps, against the oracle stream by stream."""
    from kv_cached_qwen3_gb300.talker import Talker
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 3})
    w = inputs.make_weights(g, 31)
    lens = inputs.make_start_lengths(31, 16, 60, 300)
    steps = 4
    max_seq = int(lens.max()) + steps + 1
    o = Oracle(g, w)
    oc = OracleCache(o, 16, max_seq)
    tk = Talker(g, w)
    tk.set_decode_mode(mode)
    tk.kv_init_batched(16, max_seq)
    for s in range(16):
        L = int(lens[s])
        ks, vs = [], []
        for l in range(g.n_layers):
            k, v = inputs.make_kv_layer(g, 31, l, L, stream=s)
            ks.append(k)
            vs.append(v)
        K = np.stack(ks)
        V = np.stack(vs)
        oc.kv_import(s, K, V, L)
        kt = torch.from_numpy(K).to(torch.bfloat16).cuda()
        vt = torch.from_numpy(V).to(torch.bfloat16).cuda()
        tk.kv_import(s, kt, vt, L)
    lg = torch.empty(16, g.vocab, device="cuda")
    hd = torch.empty(16, g.hidden, device="cuda")
    am = torch.empty(16, device="cuda", dtype=torch.int32)
    for t in range(steps):
        emb = np.stack([inputs.make_embeddings(g, 31, t, t + 1, stream=s)[0] for s in range(16)])
        tk.decode(dev(emb), lg, hd, am)
        rh, rl = oc.decode(emb)
        check_rows(host(hd), rh, bf16=True, what="batched hidden step %d" % t)
        check_rows(host(lg), rl, bf16=True, what="batched logits step %d" % t)
        np.testing.assert_array_equal(host(am).astype(np.int64), np.argmax(host(lg), axis=-1))
    assert tk.sync_status() == 0
    assert [tk.cur_len(s) for s in range(16)] == [int(L) + steps for L in lens]
    tk.close()
