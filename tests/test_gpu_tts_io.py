"""GPU parity of the TTS loop's input and output fusion.

Input: decode rows built from codebook ids (sum of the selected table rows plus an overlay
row) against the oracle's embed_codes. Output: codebook-0 logit suppression (vocabulary
tail to -inf except EOS) before the fused argmax, against the oracle's suppress_logits,
on the GEMV graph, the tensor-core graph and the prefill heads.
"""
import numpy as np
import pytest

from kv_cached_qwen3_gb300 import inputs
from oracle import Oracle, OracleCache, code_predictor_frame, embed_codes, suppress_logits
from parity_util import assert_top1, check_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ST_BAD_ARG = 1 << 3


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cached_qwen3_gb300 import talker
    talker.load_library()
    return torch.device("cuda", 0)


def dev(a, dtype=np.float32):
    return torch.from_numpy(np.ascontiguousarray(a, dtype)).cuda()


def host(t):
    return t.detach().float().cpu().numpy()


def check_suppressed(gpu, ref, bf16, what):
    """Same -inf pattern; the finite entries within tolerance."""
    gpu, ref = np.atleast_2d(gpu), np.atleast_2d(ref)
    np.testing.assert_array_equal(np.isneginf(gpu), np.isneginf(ref), err_msg=what)
    fin = ~np.isneginf(ref)
    for g, r, m in zip(gpu, ref, fin):
        check_rows(g[m], r[m], bf16=bf16, what=what)


@pytest.mark.parametrize("mode", [pytest.param(0, id="auto"), pytest.param(2, id="graph")])
def test_logit_suppression_prefill_and_decode_fp32(cuda, mode):
    from kv_cached_qwen3_gb300.talker import Talker
    g = inputs.TINY
    w = inputs.make_weights(g, 61)
    tail, eos = 100, 200
    emb = inputs.make_embeddings(g, 61, 0, 12)
    tk = Talker(g, w)
    tk.set_decode_mode(mode)
    tk.set_logit_suppression(tail, eos)
    tk.kv_init_batched(1, 16)
    oc = OracleCache(Oracle(g, w), 1, 16)
    _, lg, am = tk.prefill(0, dev(emb[:8]))
    _, rl = oc.prefill(0, emb[:8])
    check_suppressed(host(lg), suppress_logits(rl, tail, eos), False, "prefill")
    assert int(host(am)[0]) == int(np.argmax(host(lg)))
    out_l = torch.empty(1, g.vocab, device="cuda")
    out_a = torch.empty(1, device="cuda", dtype=torch.int32)
    for t in range(8, 12):
        tk.decode(dev(emb[t:t + 1]), out_l, None, out_a)
        _, rl = oc.decode(emb[t:t + 1])
        check_suppressed(host(out_l), suppress_logits(rl, tail, eos), False, "decode %d" % t)
        assert int(host(out_a)[0]) == int(np.argmax(host(out_l)[0]))
        assert int(host(out_a)[0]) < g.vocab - tail or int(host(out_a)[0]) == eos
    # off again: plain logits
    tk.set_logit_suppression(0, eos)
    tk.decode(dev(emb[:1]), out_l, None, out_a)
    assert np.all(np.isfinite(host(out_l)))
    assert tk.sync_status() == 0
    tk.close()


def test_logit_suppression_tensor_core_graph_bf16(cuda):
    from kv_cached_qwen3_gb300.talker import Talker
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 2})
    w = inputs.make_weights(g, 62)
    B, tail, eos = 4, 1024, 3000
    tk = Talker(g, w)
    tk.set_decode_mode(3)
    tk.set_logit_suppression(tail, eos)
    tk.kv_init_batched(B, 8)
    oc = OracleCache(Oracle(g, w), B, 8)
    emb = np.stack([inputs.make_embeddings(g, 62, 0, 1, stream=s)[0] for s in range(B)])
    lg = torch.empty(B, g.vocab, device="cuda")
    am = torch.empty(B, device="cuda", dtype=torch.int32)
    tk.decode(dev(emb), lg, None, am)
    _, rl = oc.decode(emb)
    check_suppressed(host(lg), suppress_logits(rl, tail, eos), True, "tensor-core decode")
    np.testing.assert_array_equal(host(am).astype(np.int64), np.argmax(host(lg), axis=-1))
    assert tk.sync_status() == 0
    tk.close()


@pytest.mark.parametrize("bf16", [False, True])
def test_decode_from_codebook_ids(cuda, bf16):
    from kv_cached_qwen3_gb300.talker import Talker
    if bf16:
        g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 2})
    else:
        g = inputs.TINY
    w = inputs.make_weights(g, 63)
    rng = np.random.Generator(np.random.PCG64(63))
    vocabs = [50, 30, 20, 17]
    tables = [rng.standard_normal((v, g.hidden)).astype(np.float32) for v in vocabs]
    if bf16:
        tables = [inputs.round_to_bf16(t) for t in tables]
    tdev = [dev(t).to(torch.bfloat16) if bf16 else dev(t) for t in tables]
    B, steps = 2, 3
    tk = Talker(g, w)
    tk.set_code_tables(tdev, bf16)
    tk.kv_init_batched(B, 8)
    oc = OracleCache(Oracle(g, w), B, 8)
    lg = torch.empty(B, g.vocab, device="cuda")
    hd = torch.empty(B, g.hidden, device="cuda")
    for t in range(steps):
        ids = np.stack([rng.integers(0, v, size=B) for v in vocabs]).astype(np.int32)   # [G, B]
        overlay = rng.standard_normal((B, g.hidden)).astype(np.float32) if t != 1 else None
        tk.decode_codes(dev(ids, np.int32), dev(overlay) if overlay is not None else None, lg, hd)
        x = embed_codes(tables, ids, overlay)
        rh, rl = oc.decode(x)
        check_rows(host(hd), rh, bf16=bf16, what="codes step %d hidden" % t)
        check_rows(host(lg), rl, bf16=bf16, what="codes step %d logits" % t)
    assert tk.sync_status() == 0
    # an id outside its table is reported through the device status word
    bad = np.zeros((len(vocabs), B), np.int32)
    bad[2, 1] = vocabs[2]
    tk.decode_codes(dev(bad, np.int32), None, lg, hd)
    assert tk.sync_status() & ST_BAD_ARG
    tk.close()


@pytest.mark.parametrize("suppress", [False, True])
def test_whole_frame_graph_predictor(cuda, suppress):
    """Prefill T=2 + 15 device-fed steps in one graph on the predictor geometry, replayed for
    8 frames, with a separate output head per code (head j mod 15 for code j: the predictor's
    per-codebook heads). The oracle follows the GPU's codes (teacher forcing): every step's
    logits against the oracle, every code = the argmax of the GPU's own logits, and top-1
    agreement >= 99% over the steps that the logits tolerance decides (the near-tie rule of
    parity_util: undecided steps are counted and the margin distribution is printed)."""
    from kv_cached_qwen3_gb300.talker import Talker
    pl = inputs.WORKLOADS["predictor_loop"]
    g = pl.geometry
    w = inputs.make_weights(g, pl.seed)
    rng = np.random.Generator(np.random.PCG64(64))
    n_tables = 15
    tables = [inputs.round_to_bf16(rng.standard_normal((g.vocab, g.hidden)).astype(np.float32))
              for _ in range(n_tables)]
    heads = [inputs.round_to_bf16((0.02 * rng.standard_normal((g.vocab, g.hidden))).astype(np.float32))
             for _ in range(15)]
    tdev = [dev(t).to(torch.bfloat16) for t in tables]
    hdev = [dev(h).to(torch.bfloat16) for h in heads]
    T0, n = pl.prefill_T, pl.decode_steps
    steps = list(range(n))                       # step i reads table i
    head_of = [j % 15 for j in range(n + 1)]     # code j through head j mod 15
    tk = Talker(g, w)
    tk.set_code_tables(tdev, True)
    if suppress:
        tk.set_logit_suppression(1024, 2047)
    tk.kv_init_batched(1, T0 + n + 1)
    emb_dev = torch.empty(T0, g.hidden, device="cuda")
    codes = torch.empty(n + 1, device="cuda", dtype=torch.int32)
    lg = torch.empty(n + 1, g.vocab, device="cuda")
    o = Oracle(g, w)
    all_l, all_r = [], []
    for frame in range(8):
        emb = inputs.make_embeddings(g, pl.seed, 0, T0, stream=frame)
        emb_dev.copy_(dev(emb))
        tk.frame(emb_dev, steps, codes, lg, heads=[hdev[j] for j in head_of])
        assert tk.cur_len(0) == T0 + n
        c, L = host(codes).astype(np.int64), host(lg)
        np.testing.assert_array_equal(c, np.argmax(L, axis=-1))
        ref, _ = code_predictor_frame(OracleCache(o, 1, T0 + n + 1), emb, tables, steps,
                                      [heads[j] for j in head_of], codes=c)
        if suppress:
            check_suppressed(L, suppress_logits(ref, 1024, 2047), True, "frame %d" % frame)
            ref = suppress_logits(ref, 1024, 2047)
        else:
            check_rows(L, ref, bf16=True, what="frame %d logits" % frame)
        all_l.append(L)
        all_r.append(ref)
    assert_top1(np.concatenate(all_l), np.concatenate(all_r), "frame graph")
    assert tk.sync_status() == 0
    tk.close()
