"""Op-level parity of the tcgen05/TMEM GEMM (cac_op_gemm_bf16) against fp64
matmul of the same bf16 operands: ragged M (partial row tiles, TMA zero fill),
every K split the cluster reduction supports, and the shapes of the encoder."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (130, 128, 192), (512, 2048, 512), (512, 512, 2048),
                                   (777, 640, 512), (3840, 512, 384), (129, 1536, 512)])
@pytest.mark.parametrize("splits", [0, 1, 2, 4])
def test_gemm_matches_fp64(M, N, K, splits):
    from cache_aware_conformer_gb300 import native
    if splits > K // 64:
        pytest.skip("more splits than K slices")
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) / 8).to(torch.bfloat16)
    bias = torch.randn(N, generator=g)
    C = native.gemm_bf16(A.cuda(), B.cuda(), bias.cuda(), splits=splits)
    torch.cuda.synchronize()
    ref = A.double() @ B.double().T + bias.double()
    err = (C.cpu().double() - ref).abs().max().item()
    # fp32 accumulation of exact bf16 products: error grows like sqrt(K) ulp of |C|
    assert err <= 2e-6 * np.sqrt(K) * ref.abs().max().item() + 1e-6, err


def test_gemm_splits_are_deterministic():
    from cache_aware_conformer_gb300 import native
    A = torch.randn(512, 2048, device="cuda").to(torch.bfloat16)
    B = torch.randn(512, 2048, device="cuda").to(torch.bfloat16)
    c1 = native.gemm_bf16(A, B, splits=4)
    c2 = native.gemm_bf16(A, B, splits=4)
    assert torch.equal(c1, c2)


def test_gemm_rejects_bad_shapes():
    from cache_aware_conformer_gb300 import native
    A = torch.zeros(4, 96, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(native.CacError):
        native.gemm_bf16(A, torch.zeros(64, 96, device="cuda", dtype=torch.bfloat16))   # K % 64


@pytest.mark.parametrize("M,N,K", [(130, 128, 192), (512, 2048, 512), (512, 512, 2048)])
@pytest.mark.parametrize("splits", [1, 2])
def test_split_operand_gemm(M, N, K, splits):
    """A split operand [hi | lo] enters the product as hi + lo: exact against
    fp64 of (hi + lo), and far closer to the fp32 activation than hi alone."""
    from cache_aware_conformer_gb300 import native
    g = torch.Generator().manual_seed(M + 5 * N + 11 * K)
    X = torch.randn(M, K, generator=g)
    hi = X.to(torch.bfloat16)
    lo = (X - hi.float()).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) / 8).to(torch.bfloat16)
    Bd = B.cuda()
    C = native.gemm_bf16(torch.cat([hi, lo], dim=1).cuda(), Bd, splits=splits, split=True).cpu().double()
    C1 = native.gemm_bf16(hi.cuda(), Bd, splits=splits).cpu().double()
    ref_pair = (hi.double() + lo.double()) @ B.double().T
    assert (C - ref_pair).abs().max().item() <= 2e-6 * np.sqrt(K) * ref_pair.abs().max().item() + 1e-6
    ref_x = X.double() @ B.double().T
    assert (C - ref_x).abs().max().item() < (C1 - ref_x).abs().max().item() / 20
