"""GPU: the allocation-free codec_head + argmax entry point against the library's own head.

Callers that cannot allocate device memory (a real-time audio thread where a
cudaMalloc would stall, a host that hands the library fixed buffers only, an
allocator owned by another framework) use talker_head_argmax_noalloc, whose
scratch is a fixed device array inside the library. This checks, through the
C-ABI, that two calls in a row reproduce the logits and argmax that the normal
entry points (talker_prefill and talker_decode) compute for the same final
hidden states, within the tolerance the parity tests use.
"""
import numpy as np
import pytest

from kv_cached_qwen3_gb300 import inputs
from parity_util import TOL_F32, rel_l2

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cached_qwen3_gb300 import talker
    talker.load_library()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("name", ["tiny", "talker4"])
def test_noalloc_head_matches_library_head(cuda, name):
    from kv_cached_qwen3_gb300.talker import Talker, head_argmax_noalloc
    if name == "tiny":
        g = inputs.TINY
    else:
        g = inputs.Geometry(**{**inputs.TALKER.__dict__, "n_layers": 4})
    w = inputs.make_weights(g, 41)
    wdt = torch.bfloat16 if g.weight_dtype == "bf16" else torch.float32
    W = torch.from_numpy(w["codec_head"]).to(wdt).cuda()
    tk = Talker(g, w)
    tk.kv_init_batched(4, 64)
    emb = torch.from_numpy(inputs.make_embeddings(g, 41, 0, 24)).cuda()
    # reference: the library's own head (prefill of stream 0, then a 4-stream decode)
    hid, lg, am = tk.prefill(0, emb[:16].contiguous())
    for s in range(1, 4):
        tk.prefill(s, emb[:8 + s].contiguous())
    dl = torch.empty(4, g.vocab, device="cuda")
    dh = torch.empty(4, g.hidden, device="cuda")
    da = torch.empty(4, device="cuda", dtype=torch.int32)
    tk.decode(emb[16:20].contiguous(), dl, dh, da)
    assert tk.sync_status() == 0
    cases = [(hid.view(1, -1), lg.view(1, -1), am.view(1)), (dh, dl, da)]
    for hidden, ref_logits, ref_argmax in cases:
        rows = hidden.shape[0]
        for _ in range(2):      # two calls in a row share the scratch
            out = torch.full((rows, g.vocab), float("nan"), device="cuda")
            arg = torch.full((rows,), -1, device="cuda", dtype=torch.int32)
            head_argmax_noalloc(hidden.contiguous(), W, out, arg, g.weight_dtype)
            torch.cuda.synchronize()
            got = out.cpu().numpy().astype(np.float64)
            ref = ref_logits.cpu().numpy().astype(np.float64)
            for r in range(rows):
                assert rel_l2(got[r], ref[r]) <= TOL_F32
            a = arg.cpu().numpy()
            np.testing.assert_array_equal(a, np.argmax(out.cpu().numpy(), axis=-1))
            np.testing.assert_array_equal(a, ref_argmax.cpu().numpy())
    tk.close()


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda):
    from kv_cached_qwen3_gb300.talker import TalkerError, head_argmax_noalloc
    hidden = torch.zeros(65, 64, device="cuda")
    W = torch.zeros(8, 64, device="cuda")
    with pytest.raises(TalkerError):
        head_argmax_noalloc(hidden, W, torch.empty(65, 8, device="cuda"), torch.empty(65, dtype=torch.int32,
                                                                                        device="cuda"), "f32")
    W2 = torch.zeros(8200, 64, device="cuda")
    with pytest.raises(TalkerError):
        head_argmax_noalloc(hidden[:1], W2, torch.empty(1, 8200, device="cuda"),
                            torch.empty(1, dtype=torch.int32, device="cuda"), "f32")


def _noalloc(hidden, W, wdt):
    from kv_cached_qwen3_gb300.talker import head_argmax_noalloc
    rows, V = hidden.shape[0], W.shape[0]
    out = torch.full((rows, V), float("nan"), device="cuda")
    arg = torch.full((rows,), -1, device="cuda", dtype=torch.int32)
    head_argmax_noalloc(hidden.contiguous(), W.contiguous(), out, arg, wdt)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64), arg.cpu().numpy()


@pytest.mark.parametrize("rows,H,V,wdt", [(64, 1024, 8192, "bf16"), (3, 37, 8189, "f32"), (1, 1024, 3072, "bf16"),
                                          (64, 37, 8, "f32")])
def test_noalloc_head_matches_fp64_product(cuda, rows, H, V, wdt):
    """logits against an fp64 hidden @ W.T of the same stored values, at the size limits
    (64 rows, vocab 8192), with a vocab that is not a multiple of 8 (idle warps in the
    last CTA) and a hidden size that is not a multiple of 32; calls of different grid
    sizes run back to back, so the arrival counter must be back at zero after each."""
    g = torch.Generator(device="cpu").manual_seed(rows * 1000 + V)
    hidden = torch.randn(rows, H, generator=g)
    W = 0.05 * torch.randn(V, H, generator=g)
    if wdt == "bf16":
        W = W.to(torch.bfloat16)
    ref = hidden.double() @ W.double().T
    for _ in range(2):
        got, arg = _noalloc(hidden.cuda(), W.cuda(), wdt)
        for r in range(rows):
            assert rel_l2(got[r], ref[r].numpy()) <= TOL_F32
        np.testing.assert_array_equal(arg, np.argmax(got, axis=-1))


def test_noalloc_small_grid_after_large_grid(cuda):
    """A one-CTA call right after a 1024-CTA call reduces only its own partials."""
    W_big = (0.05 * torch.randn(8192, 64)).cuda()
    W_small = (0.05 * torch.randn(8, 64)).cuda()
    x = torch.randn(4, 64).cuda()
    _noalloc(x, W_big, "f32")
    got, arg = _noalloc(x, W_small, "f32")
    ref = x.double().cpu() @ W_small.double().cpu().T
    np.testing.assert_array_equal(arg, np.argmax(ref.numpy(), axis=-1))
    _noalloc(x, W_big, "f32")
    got2, arg2 = _noalloc(x, W_small, "f32")
    np.testing.assert_array_equal(arg2, arg)


def test_noalloc_ties_and_nan_rows(cuda):
    """Equal maxima resolve to the lowest index (also when they sit in different CTAs);
    NaN logits rank as -inf, so an all-NaN row returns index 0, a valid index."""
    V, H = 64, 8
    W = torch.zeros(V, H)
    W[5, 0] = 1.0          # rows 5 and 40 give the same logit for hidden = e0
    W[40, 0] = 1.0
    W[50, 1] = 2.0         # the maximum for hidden = e1, unless that row is NaN
    hidden = torch.zeros(4, H)
    hidden[0, 0] = 1.0                      # tie between 5 and 40 (CTAs 0 and 5) -> 5
    hidden[1, :] = float("nan")             # every logit NaN -> 0
    hidden[2, 1] = 1.0                      # plain maximum -> 50
    # row 3 all zero: every logit 0.0, a 64-way tie -> 0
    got, arg = _noalloc(hidden.cuda(), W.cuda(), "f32")
    assert list(arg) == [5, 0, 50, 0]
    assert np.all(np.isnan(got[1]))
    W2 = W.clone()
    W2[50, 1] = float("nan")                # a NaN logit never wins: row 2 falls to the zeros -> 0
    W2[7, 1] = -1.0
    got, arg = _noalloc(hidden[2:3].cuda(), W2.cuda(), "f32")
    assert list(arg) == [0]
