"""The tcgen05/TMEM/TMA tile kernel in isolation: the one-CTA tile kernel (test
hook ttt_dbg_gemm_bf16) in every operand orientation, against an fp64 product
of the same bf16 values."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_mn", [False, True])
@pytest.mark.parametrize("b_mn", [False, True])
@pytest.mark.parametrize("Z,M,N,K", [(1, 128, 128, 64), (2, 256, 384, 320), (3, 192, 64, 128)])
def test_tile_kernel_matches_fp64(a_mn, b_mn, Z, M, N, K):
    from long_seq_models_chunked_b300 import abi
    g = torch.Generator(device="cpu").manual_seed(M * 7 + N * 3 + K + 11 * a_mn + 5 * b_mn)
    A = torch.randn(Z, M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(Z, N, K, generator=g).to(torch.bfloat16)
    ref = torch.bmm(A.double(), B.double().transpose(1, 2))
    Ad = (A.transpose(1, 2) if a_mn else A).contiguous().cuda()
    Bd = (B.transpose(1, 2) if b_mn else B).contiguous().cuda()
    D = torch.full((Z, M, N), float("nan"), dtype=torch.float32, device="cuda")
    assert abi.ttt_dbg_gemm_bf16(Ad, a_mn, Bd, b_mn, D, Z, M, N, K) == 0
    torch.cuda.synchronize()
    err = (D.double().cpu() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err
