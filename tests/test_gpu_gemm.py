"""The tcgen05 GEMM engine through moe_gemm_bf16, in all four operand
layouts, against a plain PyTorch fp32 matmul of the same bf16 values."""

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_kmajor", [True, False])
@pytest.mark.parametrize("b_kmajor", [True, False])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (296, 512, 200), (1000, 768, 1032)])
def test_dense_gemm_layouts(a_kmajor, b_kmajor, M, N, K):
    from mixture_experts_layer_17_gb300 import moe_gemm_bf16
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N + K)
    A = torch.randn(M, K, device="cuda", generator=g).bfloat16()
    B = torch.randn(N, K, device="cuda", generator=g).bfloat16()
    a_in = A if a_kmajor else A.t().contiguous()
    b_in = B if b_kmajor else B.t().contiguous()
    D = torch.full((M, N), float("nan"), device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    moe_gemm_bf16(a_in, a_kmajor, b_in, b_kmajor, D, ws)
    ref = A.float() @ B.float().t()
    torch.cuda.synchronize()
    err = ((D - ref).norm() / ref.norm()).item()
    assert err < 1e-5, err
    assert (D - ref).abs().max().item() < 1e-3 * ref.abs().max().item()
