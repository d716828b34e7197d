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
