"""The tcgen05 / TMA GEMM engine on its own (diagnostic entry point), every
operand major-ness the head uses, against an fp32 matmul of the same bf16 data."""

import pytest
import torch

import orpo_preference_loss_gb300 as orpo
from gpu_helpers import dev, status_tensor

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 320), (200, 296, 72), (1000, 776, 1032)])
def test_debug_gemm_matches_matmul(a_mn, b_mn, M, N, K):
    g = torch.Generator(device="cpu").manual_seed(M * 7 + N * 3 + K + 11 * a_mn + 13 * b_mn)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    ref = A.float() @ B.float().T
    A_st = (A.T.contiguous() if a_mn else A).to(dev())
    B_st = (B.T.contiguous() if b_mn else B).to(dev())
    C = torch.full((M, N), float("nan"), device=dev())
    st = status_tensor()
    orpo.orpo_debug_gemm(A_st, B_st, C, M, N, K, a_mn, b_mn, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    err = (C.cpu() - ref).abs().max().item()
    assert err <= 1e-4 * max(1.0, ref.abs().max().item()), err
