"""Host replay of the palette GEMM's in-kernel decode: the steps the kernel
takes per weight row and 64-wide K slice (six packed bytes -> eight 6-bit
indices -> eight table values -> one 16-byte chunk written at the 128-byte
swizzle position (c ^ (r & 7)) of the row), restated in numpy, against the
compression oracle's packing and decoding.  The kernel's format contract is
the one include/cac_ops.h states: index k of row n in bits [6k, 6k + 6) of
the row's little-endian bit stream."""
import numpy as np

from oracle import compress as OC


def _decode_tile_as_kernel(packed_rows, table_u16):
    """packed_rows [64][48] bytes of one K slice -> the 8 KB swizzled smem tile
    the kernel builds (uint16 table values, 64 rows x 64 columns, 128-byte rows)."""
    tile = np.zeros((64, 64), np.uint16)      # [row][16-byte chunk position * 8 + element]
    for r in range(64):
        for c in range(8):
            v = 0
            for q in range(6):
                v |= int(packed_rows[r, c * 6 + q]) << (8 * q)
            vals = [table_u16[(v >> (6 * j)) & 63] for j in range(8)]
            pos = c ^ (r & 7)
            tile[r, pos * 8:(pos + 1) * 8] = vals
    return tile


def _unswizzle(tile):
    out = np.zeros_like(tile)
    for r in range(tile.shape[0]):
        for c in range(8):
            pos = c ^ (r & 7)
            out[r, c * 8:(c + 1) * 8] = tile[r, pos * 8:(pos + 1) * 8]
    return out


def test_kernel_decode_order_matches_oracle_packing():
    rng = np.random.default_rng(5)
    N, K = 64, 256
    W = rng.normal(size=(N, K)) * 0.05
    table, idx = OC.palettize(W, table_dtype="bf16")
    packed = OC.pack6(idx)
    assert packed.shape == (N, 3 * K // 4)
    # table values as the bit patterns the kernel holds (bf16 = top half of fp32)
    t32 = np.asarray(table, np.float32).view(np.uint32)
    assert ((t32 & 0xFFFF) == 0).all()
    t16 = (t32 >> 16).astype(np.uint16)
    dec = OC.depalettize(table, idx)
    for kb in range(K // 64):
        tile = _decode_tile_as_kernel(packed[:, kb * 48:(kb + 1) * 48], t16)
        got = (_unswizzle(tile).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        np.testing.assert_array_equal(got, dec[:, kb * 64:(kb + 1) * 64])
        np.testing.assert_array_equal(OC.unpack6(packed, K)[:, kb * 64:(kb + 1) * 64], idx[:, kb * 64:(kb + 1) * 64])


def test_library_palettiser_tables_and_nearest_entries():
    """cache_aware_conformer_gb300.palette (the users' compression tool): 64
    sorted bf16 table values per matrix, every decoded weight its entry's
    nearest table value (ties to the lower entry), one table per matrix in the
    order cac_model_create_palette documents."""
    from dataclasses import replace
    import torch
    from cache_aware_conformer_gb300 import palette, synth
    from cache_aware_conformer_gb300.config import EOU_120M
    r = np.random.default_rng(3)
    w = (r.normal(size=(96, 128)) * 0.05).astype(np.float32)
    table, dec = palette.palettize(w)
    assert table.shape == (64,) and np.all(np.diff(table) >= 0)
    assert np.array_equal(torch.from_numpy(table).to(torch.bfloat16).float().numpy(), table)
    d = np.abs(w.astype(np.float64)[..., None] - table.astype(np.float64)[None, None, :])
    best = np.argmin(d, axis=-1)                      # first (lowest) index among the nearest
    assert np.array_equal(dec, table[best])
    # bf16 rounding: ties to even, as torch rounds
    x = np.float32([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5e-3, 123.456])
    assert np.array_equal(palette.to_bf16(x), torch.from_numpy(x).to(torch.bfloat16).float().numpy())
    cfg = replace(EOU_120M, n_layers=2, d_model=128, n_heads=2, ff_dim=512)
    W = synth.make_weights(cfg, 0)
    Wd, tables = palette.palettize_model(cfg, W)
    names = palette.matrix_names(cfg.n_layers)
    assert tables.shape == (5 + 11 * cfg.n_layers, 64) and len(names) == tables.shape[0]
    for t, n in zip(tables, names):
        assert np.all(np.isin(np.asarray(Wd[n], dtype=np.float32), t)), n
    assert all(np.array_equal(Wd[k], W[k]) for k in W if k not in names)
    from oracle import compress as OC
    assert names == OC.compressed_names(cfg.n_layers)  # the oracle's order, the library's table order
