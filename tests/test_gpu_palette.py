"""GPU parity of the palette-weight GEMM (cac_op_gemm_palette) against the fp64
product with the compression oracle's decoded weights ("Fast Accuracy-Preserving
RNNT Beam Search on Apple Silicon", §1.3: 64-entry tables, 6-bit palettes).

The weights are palettized and packed by oracle/compress.py; the kernel decodes
the packed rows on the GPU.  A and the table values are bf16, so every product
is exact in fp32 and the only error is the fp32 accumulation: |C - ref| <=
K * 2^-24 * sum_k |a_k w_k| for any summation order.  Shapes cover M not a
multiple of 128 (TMA zero fill), K > 4 * 64 (the 4-stage ring wraps), N > 64,
and the encoder's projection shapes; with and without bias; the status word
stays 0."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import compress as OC  # noqa: E402

pytestmark = pytest.mark.gpu


def _case(M, N, K, seed):
    r = np.random.default_rng(seed)
    W = r.normal(size=(N, K)) * np.sqrt(2.0 / (N + K))
    table, idx = OC.palettize(W, table_dtype="bf16")
    packed = OC.pack6(idx)
    A = torch.from_numpy(r.normal(size=(M, K)).astype(np.float32)).to(torch.bfloat16)
    bias = torch.from_numpy(r.normal(size=N).astype(np.float32) * 0.02)
    return table, idx, packed, A, bias


def _bf16_table(table):
    return torch.from_numpy(np.asarray(table, np.float32)).to(torch.bfloat16)


@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (200, 128, 512), (300, 192, 320), (512, 2048, 512),
                                   (128, 512, 2048), (777, 640, 512)])
@pytest.mark.parametrize("with_bias", [True, False])
def test_palette_gemm_matches_fp64_of_decoded_weights(M, N, K, with_bias):
    from cache_aware_conformer_gb300 import native
    table, idx, packed, A, bias = _case(M, N, K, M + 3 * N + 7 * K)
    tab = _bf16_table(table)
    # the table rounded to bf16 by the oracle is exactly representable
    assert np.array_equal(tab.double().numpy(), np.asarray(table, np.float64))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = native.gemm_palette(A.cuda(), torch.from_numpy(packed).cuda(), tab.cuda(),
                            bias.cuda() if with_bias else None, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    Wd = OC.depalettize(table, idx)                       # fp64 decoded weights
    Ad = A.double().numpy()
    ref = Ad @ Wd.T + (bias.double().numpy() if with_bias else 0.0)
    bound = K * 2.0 ** -24 * (np.abs(Ad) @ np.abs(Wd).T) + 1e-7
    err = np.abs(C.cpu().double().numpy() - ref)
    assert (err <= bound).all(), float((err - bound).max())


def test_palette_gemm_equals_dense_gemm_of_decoded_weights():
    """The same product through the dense tcgen05 GEMM with the decoded bf16
    weights: both accumulate exact products in fp32, so they agree to within
    the accumulation bound (the palette path only changes how B reaches
    shared memory)."""
    from cache_aware_conformer_gb300 import native
    M, N, K = 384, 512, 1024
    table, idx, packed, A, _ = _case(M, N, K, 11)
    Wb = torch.from_numpy(OC.depalettize(table, idx).astype(np.float32)).to(torch.bfloat16)
    Ac = A.cuda()
    Cp = native.gemm_palette(Ac, torch.from_numpy(packed).cuda(), _bf16_table(table).cuda())
    Cd = native.gemm_bf16(Ac, Wb.cuda(), splits=1)
    torch.cuda.synchronize()
    bound = 2 * K * 2.0 ** -24 * (A.double().abs() @ Wb.double().abs().T) + 1e-7
    assert ((Cp.cpu().double() - Cd.cpu().double()).abs() <= bound).all()


def test_palette_gemm_rejects_bad_arguments():
    from cache_aware_conformer_gb300 import native
    A = torch.zeros(4, 96, device="cuda", dtype=torch.bfloat16)
    packed = torch.zeros(64, 72, device="cuda", dtype=torch.uint8)
    tab = torch.zeros(64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(native.CacError):
        native.gemm_palette(A, packed, tab)                 # K % 64
