"""The backward pass's tcgen05 GEMM engine with K-major and M/N-major operands, against a
plain fp32 matmul of the same bf16 values (tolerance: fp32 accumulation of exact bf16 products,
1e-5 relative to the largest |C|)."""
import pytest
import torch

from sparse_conditional_moe_b300 import moe

pytestmark = pytest.mark.gpu

SHAPES = [(128, 128, 64), (256, 384, 192), (200, 136, 104), (64, 72, 8), (384, 256, 1000)]


@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_majorness(a_mn, b_mn, shape):
    M, N, K = shape
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + K)
    Am = torch.randn((M, K), generator=g, device="cuda").to(torch.bfloat16)   # A(m, k)
    Bn = torch.randn((N, K), generator=g, device="cuda").to(torch.bfloat16)   # B(n, k)
    A = Am.t().contiguous() if a_mn else Am
    B = Bn.t().contiguous() if b_mn else Bn
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    C = moe.moe_selftest_gemm(A, B, M, N, K, a_mn, b_mn, ws)
    torch.cuda.synchronize()
    assert moe.moe_device_error(ws) == 0
    ref = Am.float() @ Bn.float().t()
    err = (C - ref).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item() + 1e-6, err
