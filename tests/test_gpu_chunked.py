"""GPU parity of chunked prefill (talker_prefill_append): rows appended after cached rows.

The oracle appends the same chunks with n_past = cur_len (talker_forward_core); chunk
sizes cross page boundaries and switch between the GEMV path (T < 16) and the
tensor-core path (T >= 16, bf16 weights). Decode steps after the chunks read the cache
the chunks wrote. With Q8_0 storage every chunk takes the tensor-core path and attends the
earlier chunks' rows dequantized.
"""
import numpy as np
import pytest

from kv_cached_qwen3_gb300 import inputs
from oracle import Oracle, OracleCache
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


def run_chunks(g, w, chunks, n_dec, seed, bf16, prefill_mode=0):
    from kv_cached_qwen3_gb300.talker import Talker
    total = sum(chunks) + n_dec
    emb = inputs.make_embeddings(g, seed, 0, total)
    tk = Talker(g, w)
    tk.set_prefill_mode(prefill_mode)
    tk.kv_init_batched(1, total + 3)
    oc = OracleCache(Oracle(g, w), 1, total + 3, kv_q8=(g.kv_dtype == "q8_0"))
    at = 0
    for i, T in enumerate(chunks):
        part = emb[at:at + T]
        if i == 0:
            hd, lg, am = tk.prefill(0, dev(part))
            rh, rl = oc.prefill(0, part)
        else:
            hd, lg, am = tk.prefill_append(0, dev(part))
            rhs, rls = oc.append_rows(0, part)
            rh, rl = rhs[-1], rls[-1]
        at += T
        assert tk.cur_len(0) == at
        check_rows(host(hd), rh[None], bf16=bf16, what="chunk %d (T=%d) hidden" % (i, T))
        check_rows(host(lg), rl[None], bf16=bf16, what="chunk %d (T=%d) logits" % (i, T))
        assert int(host(am)[0]) == int(np.argmax(host(lg)))
    for t in range(n_dec):
        e = emb[at + t:at + t + 1]
        lg, hd = torch.empty(1, g.vocab, device="cuda"), torch.empty(1, g.hidden, device="cuda")
        tk.decode(dev(e), lg, hd)
        rh, rl = oc.decode(e)
        check_rows(host(hd), rh, bf16=bf16, what="decode %d hidden" % t)
        check_rows(host(lg), rl, bf16=bf16, what="decode %d logits" % t)
    assert tk.cur_len(0) == total
    assert tk.sync_status() == 0
    tk.close()


def test_chunked_prefill_fp32_gemv_path(cuda):
    g = inputs.TINY
    run_chunks(g, inputs.make_weights(g, 51), [20, 1, 7, 30, 40], 3, 52, bf16=False)


@pytest.mark.parametrize("mode", [pytest.param(0, id="auto"), pytest.param(3, id="mma-sync-attention"),
                                  pytest.param(4, id="tcgen05-attention")])
def test_chunked_prefill_bf16_both_paths(cuda, mode):
    """Chunks on the GEMV path (T < 16) and the tensor-core path; modes 3 / 4 pin the causal
    attention of the tensor-core chunks to the mma.sync / tcgen05 kernel (the latter reads the
    earlier keys of the stream through its dense copy and masks on positions pos0 + r)."""
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 4})
    run_chunks(g, inputs.make_weights(g, 53), [100, 70, 5, 16, 64], 2, 54, bf16=True, prefill_mode=mode)


@pytest.mark.parametrize("chunks", [pytest.param([100, 70, 5, 16, 64], id="short"),
                                    pytest.param([300, 260, 40], id="long")])
def test_chunked_prefill_q8_0(cuda, chunks):
    """Chunks over Q8_0 storage: each chunk attends the rows of the earlier chunks dequantized
    from the cache and its own rows exactly (the oracle's reading), on the tcgen05 attention
    whatever the chunk size, then decode steps over the quantized rows."""
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 2, "kv_dtype": "q8_0"})
    run_chunks(g, inputs.make_weights(g, 63), chunks, 2, 64, bf16=True)


@pytest.mark.parametrize("mode", [pytest.param(0, id="auto"), pytest.param(4, id="tcgen05-attention")])
def test_chunked_prefill_long_chunks(cuda, mode):
    """Chunks of several 128-row query tiles whose start positions are not multiples of the
    128-key block (300, then 260 after 300, then 40 after 560)."""
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 2})
    run_chunks(g, inputs.make_weights(g, 56), [300, 260, 40], 1, 58, bf16=True, prefill_mode=mode)


@pytest.mark.parametrize("kv", ["bf16", "f32"])
def test_chunked_prefill_tall_chunk(cuda, kv):
    """A 1000-row chunk appended after 300 cached rows: tall products on the CTA-pair GEMM, QK-norm,
    RoPE and the KV append at positions 300..1299 (bf16 and f32 caches)."""
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 2, "kv_dtype": kv})
    run_chunks(g, inputs.make_weights(g, 61), [300, 1000], 1, 62, bf16=True)


def test_append_overflow_changes_nothing(cuda):
    from kv_cached_qwen3_gb300.talker import Talker, TalkerError
    g = inputs.TINY
    w = inputs.make_weights(g, 55)
    tk = Talker(g, w)
    tk.kv_init_batched(1, 40)
    emb = inputs.make_embeddings(g, 55, 0, 41)
    tk.prefill(0, dev(emb[:30]))
    with pytest.raises(TalkerError) as ei:
        tk.prefill_append(0, dev(emb[30:41]))
    assert ei.value.status == 2   # EOVERFLOW
    assert tk.cur_len(0) == 30
    tk.prefill_append(0, dev(emb[30:40]))
    assert tk.cur_len(0) == 40
    assert tk.sync_status() == 0
    tk.close()


@pytest.mark.parametrize("mode", [pytest.param(3, id="mma-sync-attention"), pytest.param(4, id="tcgen05-attention")])
@pytest.mark.parametrize("kv,B,T", [("bf16", 3, 70), ("q8_0", 3, 70), ("bf16", 4, 240)])
def test_batched_prefill_streams(cuda, kv, B, T, mode):
    """Streams 0..B-1 prefilled in one call (T rows each, across page boundaries), then a decode
    step; the causal attention pinned to either kernel (tcgen05: one launch pair per stream). With
    4 x 240 rows the projections run on the CTA-pair GEMM and each row maps to its stream's position."""
    from kv_cached_qwen3_gb300.talker import Talker
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 2, "kv_dtype": kv})
    w = inputs.make_weights(g, 57)
    emb = np.stack([inputs.make_embeddings(g, 57, 0, T + 1, stream=s) for s in range(B)])   # [B, T+1, H]
    tk = Talker(g, w)
    tk.set_prefill_mode(mode)
    tk.kv_init_batched(B, T + 2)
    oc = OracleCache(Oracle(g, w), B, T + 2, kv_q8=(kv == "q8_0"))
    hd, lg, am = tk.prefill_batched(dev(emb[:, :T]))
    for s in range(B):
        rh, rl = oc.prefill(s, emb[s, :T])
        check_rows(host(hd)[s], rh[None], bf16=True, what="stream %d hidden" % s)
        check_rows(host(lg)[s], rl[None], bf16=True, what="stream %d logits" % s)
        assert int(host(am)[s]) == int(np.argmax(host(lg)[s]))
        assert tk.cur_len(s) == T
    lgd = torch.empty(B, g.vocab, device="cuda")
    tk.decode(dev(emb[:, T]), lgd)
    _, rl = oc.decode(emb[:, T])
    check_rows(host(lgd), rl, bf16=True, what="decode after batched prefill")
    assert tk.sync_status() == 0
    tk.close()
