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


# ---------------------------------------------------------------------------
# the encoder with palette weights (cac_model_create_palette)
# ---------------------------------------------------------------------------
def _palette_model_inputs(cfg, seed=0):
    """Weights of cfg palettized by the compression oracle (bf16 tables): the
    decoded weight dict and the tables in the library's order."""
    from cache_aware_conformer_gb300 import synth
    W = synth.make_weights(cfg, seed)
    Wd = dict(W)
    tables = []
    for name in OC.compressed_names(cfg.n_layers):
        table, idx = OC.palettize(W[name], table_dtype="bf16")
        Wd[name] = OC.depalettize(table, idx)
        tables.append(table)
    return Wd, np.stack(tables).astype(np.float32)


def test_palette_encoder_matches_dense_and_oracle():
    """A two-layer bf16 encoder whose projections run on 6-bit palettes, pushed
    160 ms at a time: bit-identical to the dense model on the decoded weights
    (the kernel must decode exactly their bf16 values), and within the bf16
    bars of the fp64 oracle on the decoded weights (the compressed encoder)."""
    from dataclasses import replace
    from cache_aware_conformer_gb300 import native, synth
    from cache_aware_conformer_gb300.config import EOU_120M
    from oracle import conformer as O
    from _util import assert_close
    cfg = replace(EOU_120M, n_layers=2, d_model=128, n_heads=2, ff_dim=512)
    Wd, tables = _palette_model_inputs(cfg)
    blob = synth.pack_weights(cfg, Wd)
    pal = native.Model(cfg, blob, tables=tables)
    dense = native.Model(cfg, blob)
    S = 8
    pools = [native.Pool(m, S, 2) for m in (pal, dense)]
    ids = [[p.create_stream() for _ in range(S)] for p in pools]
    refs = [O.StreamingEncoder(Wd, cfg) for _ in range(2)]  # streams 0 and S - 1
    mels = [synth.make_mel(96, 40 + s) for s in range(S)]
    for k in range(6):
        chunk = np.stack([m[16 * k: 16 * (k + 1)] for m in mels])
        outs = [p.push(i, torch.from_numpy(chunk).cuda()) for p, i in zip(pools, ids)]
        e_pal, j_pal = outs[0][0].cpu().numpy(), outs[0][1].cpu().numpy()
        e_den, j_den = outs[1][0].cpu().numpy(), outs[1][1].cpu().numpy()
        assert np.array_equal(e_pal, e_den) and np.array_equal(j_pal, j_den), k
        for r, s in zip(refs, (0, S - 1)):
            e_ref, j_ref = r.push(mels[s][16 * k: 16 * (k + 1)])
            assert_close(e_pal[s], e_ref, cfg, f"palette enc step {k} stream {s}")
            assert_close(j_pal[s], j_ref, cfg, f"palette joint step {k} stream {s}")
    for p in pools:
        p.check()
    pal.check()


def test_palette_model_rejects_a_weight_missing_from_its_table():
    from dataclasses import replace
    from cache_aware_conformer_gb300 import native, synth
    from cache_aware_conformer_gb300.config import EOU_120M
    cfg = replace(EOU_120M, n_layers=1, d_model=128, n_heads=2, ff_dim=512)
    Wd, tables = _palette_model_inputs(cfg)
    blob = synth.pack_weights(cfg, Wd)
    bad = tables.copy()
    # an entry of the pw2 table (layer 0: 5 + 8) that some weight uses, moved off its value
    t = 5 + 8
    used = np.unique(Wd["l0.conv.w_pw2"])
    i = int(np.flatnonzero(np.isin(bad[t], used))[0])
    bad[t, i] = np.float32(bad[t, i] * 1.5 + 0.25)
    with pytest.raises(native.CacError) as e:
        native.Model(cfg, blob, tables=bad)
    assert e.value.code == -1  # CAC_E_INVAL
    with pytest.raises(native.CacError):
        native.Model(cfg, blob, tables=tables[:-1])  # one table short
