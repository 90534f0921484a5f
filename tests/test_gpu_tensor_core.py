"""The tensor-core building blocks (swizzled shared tiles, descriptors,
tcgen05.mma, TMEM loads/stores) against torch's GEMM."""
import pytest
import torch

from continuous_linear_attention_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N", [64, 128, 192, 256])
@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("acc", [False, True])
@pytest.mark.parametrize("f16", [False, True])
def test_umma_gemm_matches_torch(N, K, acc, f16):
    g = torch.Generator(device="cuda").manual_seed(N * 1000 + K + acc)
    A = torch.randn(128, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    C = torch.randn(128, N, device="cuda", generator=g) if acc else None
    D = torch.full((128, N), float("nan"), device="cuda")
    binding.diag_umma_gemm(A, B, C, D, operand_f16=f16)
    torch.cuda.synchronize()
    ref = A.float() @ B.float().T + (C if acc else 0)
    torch.testing.assert_close(D, ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("N", [64, 128, 256])
@pytest.mark.parametrize("major", ["a_mn", "b_mn", "both"])
@pytest.mark.parametrize("f16", [False, True])
def test_umma_gemm_mn_major_matches_torch(N, major, f16):
    """MN-major operands (the layout of a token-major TMA tile) give the same
    product as K-major ones."""
    K = 64
    g = torch.Generator(device="cuda").manual_seed(7 * N + len(major))
    A = torch.randn(128, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    C = torch.randn(128, N, device="cuda", generator=g)
    D = torch.full((128, N), float("nan"), device="cuda")
    binding.diag_umma_gemm_ex(A, B, C, D, operand_f16=f16, a_mn=major in ("a_mn", "both"),
                              b_mn=major in ("b_mn", "both"))
    torch.cuda.synchronize()
    ref = A.float() @ B.float().T + C
    torch.testing.assert_close(D, ref, rtol=1e-5, atol=1e-4)


@pytest.mark.parametrize("N", [64, 128])
# an MN-major shared B operand of the helper holds K = 64
@pytest.mark.parametrize("K,b_mn", [(64, False), (128, False), (64, True)])
@pytest.mark.parametrize("f16", [False, True])
def test_umma_gemm_a_in_tensor_memory_matches_torch(N, K, b_mn, f16):
    """A read by the MMA from tensor memory (two 16-bit elements per column)
    gives the same product as A from shared memory."""
    g = torch.Generator(device="cuda").manual_seed(11 * N + K + 3 * b_mn + f16)
    A = torch.randn(128, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
    C = torch.randn(128, N, device="cuda", generator=g)
    D = torch.full((128, N), float("nan"), device="cuda")
    binding.diag_umma_gemm_ex(A, B, C, D, operand_f16=f16, a_mn=2, b_mn=b_mn)
    torch.cuda.synchronize()
    ref = A.float() @ B.float().T + C
    torch.testing.assert_close(D, ref, rtol=1e-5, atol=1e-4)


def test_bounded_wait_times_out_and_reports_the_flag():
    """A wait on an mbarrier that nothing arrives on (nothing in flight) gives
    up after the library's limit, raises GDN_FLAG_TIMEOUT, and the context
    stays usable: a forward afterwards still matches the oracle."""
    import time
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    binding.diag_wait_timeout(flags)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(flags.item()) == binding.FLAG_TIMEOUT
    assert 1.5 <= waited <= 30.0, waited
    from gpu_check import check_against_oracle
    from continuous_linear_attention_gb300 import synth
    check_against_oracle(synth.tiny_packed(0))
