"""tcgen05 / TMA / tensor-memory building blocks in isolation (through the C ABI):
a 128 x N x K bf16 GEMM against an fp64 product of the same bf16 values."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import kimi_delta_attention_11_gb300 as k
    k.load_library()
    return k


@pytest.mark.parametrize("mode", [0, 1], ids=["tma", "swizzled_stores"])
@pytest.mark.parametrize("N", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("K", [16, 64, 128])
def test_umma_gemm(kda, mode, N, K):
    g = torch.Generator(device="cpu").manual_seed(N * 1000 + K + mode)
    A = torch.randn((128, K), generator=g).to(torch.bfloat16).cuda()
    B = torch.randn((N, K), generator=g).to(torch.bfloat16).cuda()
    D = kda.selftest_umma(A, B, mode)
    ref = A.double() @ B.double().T
    err = (D.double() - ref).abs().max().item()
    assert err <= 1e-3 * max(1.0, ref.abs().max().item()), f"max err {err}"


@pytest.mark.parametrize("N", [64, 128, 256])
@pytest.mark.parametrize("K", [16, 64, 128])
def test_umma_gemm_b_mn_major(kda, N, K):
    g = torch.Generator(device="cpu").manual_seed(7 * N + K)
    A = torch.randn((128, K), generator=g).to(torch.bfloat16).cuda()
    Bt = torch.randn((K, N), generator=g).to(torch.bfloat16).cuda()
    D = kda.selftest_umma(A, Bt.contiguous(), 2)
    ref = A.double() @ Bt.double()
    assert (D.double() - ref).abs().max().item() <= 1e-3 * max(1.0, ref.abs().max().item())


@pytest.mark.parametrize("N", [32, 64, 256])
@pytest.mark.parametrize("K", [16, 64, 128])
def test_umma_gemm_a_mn_major(kda, N, K):
    g = torch.Generator(device="cpu").manual_seed(11 * N + K)
    At = torch.randn((K, 128), generator=g).to(torch.bfloat16).cuda()
    B = torch.randn((N, K), generator=g).to(torch.bfloat16).cuda()
    D = kda.selftest_umma(At.contiguous(), B, 3)
    ref = At.double().T @ B.double().T
    assert (D.double() - ref).abs().max().item() <= 1e-3 * max(1.0, ref.abs().max().item())


@pytest.mark.parametrize("N", [16, 64, 128, 256])
@pytest.mark.parametrize("K", [16, 64, 128])
def test_umma_gemm_a_in_tmem(kda, N, K):
    """A written to tensor memory with tcgen05.st (row m in lane m, two bf16 per 32-bit
    column), B in shared memory: the operand form of the recurrence kernel's chained
    products."""
    g = torch.Generator(device="cpu").manual_seed(13 * N + K)
    A = torch.randn((128, K), generator=g).to(torch.bfloat16).cuda()
    B = torch.randn((N, K), generator=g).to(torch.bfloat16).cuda()
    D = kda.selftest_umma(A, B, 4)
    ref = A.double() @ B.double().T
    assert (D.double() - ref).abs().max().item() <= 1e-3 * max(1.0, ref.abs().max().item())
