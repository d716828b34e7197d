"""GPU parity of the two causal prefill attention kernels (tcgen05 tiles with dense K / V^T,
and mma.sync tiles over the paged cache) through every row of a prefill.

talker_prefill_all_rows returns the logits and final hidden state of every row, so a wrong
attention output of any query row (any 128-row tile, the diagonal block, the ragged last
tile, keys past the stream's length) shows in that row. Both kernels are checked against the
oracle's full-sequence forward (explicit causal mask), and against each other. Prefill modes
4 and 3 pin the kernel; mode 0 picks tcgen05 from 256 rows up.
"""
import numpy as np
import pytest

from kv_cached_qwen3_gb300 import inputs
from oracle import Oracle
from parity_util import check_rows, rel_l2

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cached_qwen3_gb300 import talker
    talker.load_library()
    return torch.device("cuda", 0)


def host(t):
    return t.detach().float().cpu().numpy()


def all_rows(g, w, emb, prefill_mode, max_seq):
    from kv_cached_qwen3_gb300.talker import Talker
    tk = Talker(g, w)
    tk.set_prefill_mode(prefill_mode)
    tk.kv_init_batched(1, max_seq)
    hd, lg = tk.prefill_all_rows(0, torch.from_numpy(emb).cuda())
    st = tk.sync_status()
    tk.close()
    assert st == 0, "device status word %d" % st
    return host(hd), host(lg)


@pytest.mark.parametrize("kv", ["bf16", "q8_0"])
@pytest.mark.parametrize("T", [16, 100, 128, 129, 300])
def test_prefill_attention_kernels_every_row(cuda, T, kv):
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 2, "kv_dtype": kv})
    w = inputs.make_weights(g, 70 + T)
    emb = inputs.make_embeddings(g, 70 + T, 0, T)
    ref_h, ref_l = Oracle(g, w).forward_full(emb)
    got = {}
    for mode in (4, 3):        # 4: tcgen05 attention, 3: mma.sync attention
        h, lg = all_rows(g, w, emb, mode, T + 5)
        check_rows(h, ref_h, bf16=True, what="T=%d %s mode %d hidden" % (T, kv, mode))
        check_rows(lg, ref_l, bf16=True, what="T=%d %s mode %d logits" % (T, kv, mode))
        got[mode] = lg
    # the two kernels differ only in summation order and P's rounding point
    worst = max(rel_l2(a, b) for a, b in zip(got[4], got[3]))
    assert worst <= 1e-2, worst


def test_prefill_attention_long_rows_sampled(cuda):
    """T = 1000 (8 query tiles, ragged): rows sampled across the tiles against the oracle's
    full-sequence forward; every row of the two kernels against each other."""
    g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 1})
    w = inputs.make_weights(g, 77)
    T = 1000
    emb = inputs.make_embeddings(g, 77, 0, T)
    h0, l0 = all_rows(g, w, emb, 4, T + 1)
    h3, l3 = all_rows(g, w, emb, 3, T + 1)
    rows = [0, 1, 127, 128, 255, 511, 640, 999]
    ref_h, ref_l = Oracle(g, w).forward_full(emb)
    check_rows(l0[rows], ref_l[rows], bf16=True, what="tcgen05 sampled rows")
    check_rows(l3[rows], ref_l[rows], bf16=True, what="mma.sync sampled rows")
    assert max(rel_l2(a, b) for a, b in zip(l0, l3)) <= 1e-2
