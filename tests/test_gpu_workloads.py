"""GPU parity on the predictor loop and the long-context workloads, at their full sizes.

predictor_loop: the 5-layer predictor runs frames of prefill T=2 followed by 15 decode
steps; every frame starts again at position 0. long_context: the 28-layer Talker decodes
one row against caches of 8K, 16K and 32K imported positions, and prefills T=4096 rows on
the tensor-core path. The oracle runs every compared row in fp64.
"""
import numpy as np
import pytest

from kv_cached_qwen3_gb300 import inputs
from oracle import Oracle, decode_row_lazy_cache
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


def frame_embeddings(g, seed, frame, rows):
    """Frame f of the predictor loop reads embedding stream f, rows [0, rows)."""
    return inputs.make_embeddings(g, seed, 0, rows, stream=frame)


@pytest.fixture(scope="module")
def predictor():
    wl = inputs.WORKLOADS["predictor_loop"]
    g = wl.geometry
    w = inputs.make_weights(g, wl.seed)
    return wl, g, w, Oracle(g, w)


@pytest.mark.parametrize("mode", [pytest.param(2, id="graph"), pytest.param(3, id="tensor-core-graph")])
def test_predictor_loop_frames(cuda, predictor, mode):
    """Four frames of prefill T=2 + 15 decodes on one cache; each frame against a fresh oracle forward."""
    from kv_cached_qwen3_gb300.talker import Talker
    wl, g, w, o = predictor
    T0, n = wl.prefill_T, wl.decode_steps
    tk = Talker(g, w)
    tk.set_decode_mode(mode)
    tk.kv_init_batched(1, T0 + n)
    lg = torch.empty(1, g.vocab, device="cuda")
    hd = torch.empty(1, g.hidden, device="cuda")
    am = torch.empty(1, device="cuda", dtype=torch.int32)
    e = torch.empty(1, g.hidden, device="cuda")
    all_gpu, all_ref = [], []
    for f in range(4):
        emb = frame_embeddings(g, wl.seed, f, T0 + n)
        hid0, lg0, am0 = tk.prefill(0, dev(emb[:T0]))
        assert tk.cur_len(0) == T0
        hids, lgs, ams = [host(hid0)], [host(lg0)], [int(host(am0)[0])]
        for t in range(n):
            e.copy_(dev(emb[T0 + t:T0 + t + 1]))
            tk.decode(e, lg, hd, am)
            hids.append(host(hd)[0])
            lgs.append(host(lg)[0])
            ams.append(int(host(am)[0]))
        assert tk.cur_len(0) == T0 + n
        rh, rl = o.forward_full(emb)
        hids, lgs = np.stack(hids), np.stack(lgs)
        check_rows(hids, rh[T0 - 1:], bf16=True, what="predictor frame %d hidden" % f)
        check_rows(lgs, rl[T0 - 1:], bf16=True, what="predictor frame %d logits" % f)
        np.testing.assert_array_equal(np.array(ams), np.argmax(lgs, axis=-1))
        all_gpu.append(lgs)
        all_ref.append(rl[T0 - 1:])
    assert top1_agreement(np.concatenate(all_gpu), np.concatenate(all_ref)) >= TOL_TOP1
    assert tk.sync_status() == 0
    tk.close()


@pytest.fixture(scope="module")
def talker_long():
    wl = inputs.WORKLOADS["long_context"]
    g = wl.geometry
    w = inputs.make_weights(g, wl.seed)
    return wl, g, w, Oracle(g, w)


@pytest.mark.parametrize("L", [8192, 16384, 32768])
def test_long_context_decode(cuda, talker_long, L):
    """One decode row against an imported L-position cache on every decode path, 28 layers."""
    from kv_cached_qwen3_gb300.talker import Talker
    wl, g, w, o = talker_long
    nl, nkv, hd = g.n_layers, g.n_kv_heads, g.head_dim
    K = torch.empty(nl, nkv, L, hd, dtype=torch.bfloat16, device="cuda")
    V = torch.empty_like(K)
    host_kv = []
    for l in range(nl):
        k, v = inputs.make_kv_layer(g, wl.seed, l, L)
        kt, vt = torch.from_numpy(k).to(torch.bfloat16), torch.from_numpy(v).to(torch.bfloat16)
        K[l].copy_(kt)
        V[l].copy_(vt)
        host_kv.append((kt, vt))
    emb = inputs.make_embeddings(g, wl.seed, L, L + 1)
    rh, rl = decode_row_lazy_cache(
        o, emb[0], L, lambda l: (host_kv[l][0].float().numpy(), host_kv[l][1].float().numpy()))
    tk = Talker(g, w)
    tk.kv_init_batched(1, L + 1)
    tk.kv_import(0, K, V, L)
    del K, V
    lg = torch.empty(1, g.vocab, device="cuda")
    hdn = torch.empty(1, g.hidden, device="cuda")
    am = torch.empty(1, device="cuda", dtype=torch.int32)
    for mode in (2, 3):
        tk.set_decode_mode(mode)
        tk.rewind(0, L)
        tk.decode(dev(emb), lg, hdn, am)
        assert tk.sync_status() == 0
        assert tk.cur_len(0) == L + 1
        check_rows(host(hdn), rh[None], bf16=True, what="L=%d mode %d hidden" % (L, mode))
        check_rows(host(lg), rl[None], bf16=True, what="L=%d mode %d logits" % (L, mode))
        assert int(host(am)[0]) == int(np.argmax(host(lg)[0]))
    tk.close()


@pytest.mark.slow
def test_long_context_prefill_4096_tensor_cores(cuda, talker_long):
    """Prefill T=4096 on the 28-layer Talker (tensor-core path), every row against the oracle."""
    from kv_cached_qwen3_gb300.talker import Talker
    wl, g, w, o = talker_long
    T = wl.prefill_T
    emb = inputs.make_embeddings(g, wl.seed, 0, T)
    tk = Talker(g, w)
    tk.kv_init_batched(1, T + 1)
    hid, lg = tk.prefill_all_rows(0, dev(emb))
    assert tk.sync_status() == 0
    assert tk.cur_len(0) == T
    hid, lg = host(hid), host(lg)
    tk.close()
    rh, rl = o.forward_full(emb)
    check_rows(hid, rh, bf16=True, what="prefill 4096 hidden")
    check_rows(lg, rl, bf16=True, what="prefill 4096 logits")
    assert_top1(lg, rl, what="prefill 4096 rows")


def stream_cache(g, seed, s, L):
    """Stream s's pre-filled cache of L rows, fp32 [n_layers, n_kv, L, hd] (bf16-valued)."""
    ks, vs = zip(*(inputs.make_kv_layer(g, seed, l, L, stream=s) for l in range(g.n_layers)))
    return np.stack(ks), np.stack(vs)


@pytest.mark.slow
@pytest.mark.parametrize("mode", [pytest.param(0, id="auto"), pytest.param(2, id="gemv-graph")])
def test_batched16_full_size(cuda, mode):
    """The 16-stream batched decode at its own size: the 28-layer Talker, start lengths drawn
    U{128..2048} (the workload's seed), per-stream causal windows, 8 decode steps. Every stream
    against the oracle (its own cache and rows) at the bf16 tolerances; top-1 >= 99% over all
    stream-steps that the logits tolerance decides (the near-tie rule of parity_util);
    lengths advance exactly."""
    from kv_cached_qwen3_gb300.talker import Talker
    from oracle import OracleCache
    wl = inputs.WORKLOADS["batched16"]
    g, seed, B = wl.geometry, wl.seed, wl.n_streams
    w = inputs.make_weights(g, seed)
    lens = inputs.make_start_lengths(seed, B, *wl.start_len_range)
    steps = 8
    max_seq = int(lens.max()) + steps + 1
    tk = Talker(g, w)
    tk.set_decode_mode(mode)
    tk.kv_init_batched(B, max_seq)
    for s in range(B):
        K, V = stream_cache(g, seed, s, int(lens[s]))
        tk.kv_import(s, torch.from_numpy(K).to(torch.bfloat16).cuda(), torch.from_numpy(V).to(torch.bfloat16).cuda(),
                     int(lens[s]))
        del K, V
    embs = [inputs.make_embeddings(g, seed, int(lens[s]), int(lens[s]) + steps, stream=s) for s in range(B)]
    lg = torch.empty(B, g.vocab, device="cuda")
    hd = torch.empty(B, g.hidden, device="cuda")
    am = torch.empty(B, device="cuda", dtype=torch.int32)
    got_h, got_l = [], []
    for t in range(steps):
        tk.decode(dev(np.stack([embs[s][t] for s in range(B)])), lg, hd, am)
        got_h.append(host(hd))
        got_l.append(host(lg))
        np.testing.assert_array_equal(host(am).astype(np.int64), np.argmax(got_l[-1], axis=-1))
    assert tk.sync_status() == 0
    assert [tk.cur_len(s) for s in range(B)] == [int(L) + steps for L in lens]
    tk.close()
    got_h, got_l = np.stack(got_h), np.stack(got_l)      # [steps, B, *]
    o = Oracle(g, w)
    ref_l = np.empty_like(got_l, dtype=np.float64)
    for s in range(B):
        oc = OracleCache(o, 1, max_seq)
        K, V = stream_cache(g, seed, s, int(lens[s]))
        oc.kv_import(0, K, V, int(lens[s]))
        del K, V
        for t in range(steps):
            rh, rl = oc.decode(embs[s][t:t + 1])
            ref_l[t, s] = rl[0]
            check_rows(got_h[t, s], rh[0], bf16=True, what="stream %d (L=%d) step %d hidden" % (s, lens[s], t))
            check_rows(got_l[t, s], rl[0], bf16=True, what="stream %d (L=%d) step %d logits" % (s, lens[s], t))
    assert_top1(got_l.reshape(-1, g.vocab), ref_l.reshape(-1, g.vocab), "batched16 full size")
