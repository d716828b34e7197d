"""GPU: the tensor-core (tcgen05/TMEM) GEMM against a float64 matmul of the same bf16 inputs.

Shapes cover both tile widths (N % 256 == 0 or not), split-K, ragged M, and tall M (eight
or more row blocks, the wide-tile range) with a ragged last row block; products of at most
128 rows take the kernel with the weights as the MMA's M operand (rows rounded up to 16
columns), checked at 1, 15, 16, 17, 96 and 128 rows and just above at 129."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from kv_cached_qwen3_gb300 import talker
    talker.load_library()
    return torch.device("cuda", 0)


@pytest.mark.parametrize("M,N,K,splits", [(1, 128, 64, 1), (96, 4096, 1024, 1), (96, 1024, 3072, 12),
                                          (15, 4096, 1024, 4), (16, 1024, 2048, 16), (17, 6144, 1024, 3),
                                          (128, 1024, 3072, 5), (129, 1024, 1024, 2), (1, 1024, 3072, 48),
                                          (130, 256, 128, 1), (300, 384, 2048, 4), (4096, 1024, 1024, 1),
                                          (1100, 384, 256, 1), (1030, 768, 1024, 2), (2048, 6144, 1024, 1)])
def test_gemm_matches_fp64(cuda, M, N, K, splits):
    from kv_cached_qwen3_gb300.talker import test_gemm_bf16
    g = torch.Generator(device="cpu").manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (0.02 * torch.randn(N, K, generator=g)).to(torch.bfloat16)
    ref = A.double() @ B.double().T
    out = torch.zeros(M, N, device="cuda")
    test_gemm_bf16(A.cuda(), B.cuda(), out, splits=splits)
    got = out.cpu().double()
    err = (got - ref).norm() / ref.norm()
    assert float(err) < 1e-5, float(err)


@pytest.mark.parametrize("M,splits", [(64, 1), (16, 3), (300, 2)])
def test_gemm_accumulates_into_output(cuda, M, splits):
    from kv_cached_qwen3_gb300.talker import test_gemm_bf16
    A = torch.randn(M, 256).to(torch.bfloat16).cuda()
    B = (0.02 * torch.randn(128, 256)).to(torch.bfloat16).cuda()
    base = torch.randn(M, 128, device="cuda")
    out = base.clone()
    test_gemm_bf16(A, B, out, accumulate=True, splits=splits)
    ref = base.double().cpu() + A.double().cpu() @ B.double().cpu().T
    assert float((out.cpu().double() - ref).norm() / ref.norm()) < 1e-5


@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (16, 6144, 1024), (96, 6144, 1024), (33, 256, 3072),
                                   (130, 256, 128), (300, 6144, 1024), (1024, 384, 192),
                                   (1100, 6144, 1024)])
def test_gemm_swiglu_epilogue(cuda, M, N, K):
    """silu(gate) * up from interleaved gate/up rows, rounded to bf16 (both tile widths, ragged M)."""
    from kv_cached_qwen3_gb300.talker import test_gemm_swiglu_bf16
    g = torch.Generator(device="cpu").manual_seed(M + 3 * N + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (0.05 * torch.randn(N, K, generator=g)).to(torch.bfloat16)
    gu = A.double() @ B.double().T
    gate, up = gu[:, 0::2], gu[:, 1::2]
    ref = gate / (1.0 + torch.exp(-gate)) * up
    out = torch.zeros(M, N // 2, dtype=torch.bfloat16, device="cuda")
    test_gemm_swiglu_bf16(A.cuda(), B.cuda(), out)
    got = out.cpu().double()
    err = (got - ref).norm() / ref.norm()
    assert float(err) < 4e-3, float(err)          # bf16 output rounding (2^-9 relative per element)
    assert float((got - ref).abs().max()) <= float(ref.abs().max()) * 2 ** -7
