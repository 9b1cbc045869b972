"""Pins of the compressed-weight oracle (oracle/compress.py) to things other
than itself: a hand-packed byte fixture, exact reproduction of a matrix with at
most 64 distinct values, brute-force nearest entries, the uniform
distribution's optimal quantiser, scikit-learn's k-means objective, torch's
bf16 rounding, and int8 bounds and ties ("Fast Accuracy-Preserving RNNT Beam
Search on Apple Silicon", §1.3: 64-entry tables, i.e. 6-bit palettes)."""
import numpy as np
import pytest

from cache_aware_conformer_gb300 import synth
from cache_aware_conformer_gb300.config import TINY
from oracle import compress as C


def test_packed_bytes_fixture_and_round_trip():
    # indices 1, 2, 3, 4 -> bit stream 000001 000010 000011 000100 (LSB first) = 0x103081
    assert C.pack6(np.array([[1, 2, 3, 4]])).tolist() == [[0x81, 0x30, 0x10]]
    assert C.pack6(np.array([[63] * 4])).tolist() == [[0xFF, 0xFF, 0xFF]]
    assert C.pack6(np.array([[0, 0, 0, 63, 1]])).shape == (1, 4)     # 30 bits -> 4 bytes
    rng = np.random.default_rng(0)
    for K in (4, 5, 64, 67):
        idx = rng.integers(0, 64, size=(3, K))
        assert np.array_equal(C.unpack6(C.pack6(idx), K), idx)


def test_at_most_64_distinct_values_are_reproduced_exactly():
    rng = np.random.default_rng(1)
    values = np.float16(rng.standard_normal(50) * 0.05).astype(np.float64)
    w = rng.choice(values, size=(40, 30))
    table, idx = C.palettize(w, "fp16")
    assert np.array_equal(C.depalettize(table, idx), w)


def test_indices_are_the_nearest_entry_by_brute_force():
    rng = np.random.default_rng(2)
    w = rng.standard_normal((16, 48)) * 0.1
    table, idx = C.palettize(w, "bf16")
    for v, i in zip(w.reshape(-1), idx.reshape(-1)):
        d = [abs(v - t) for t in table]
        best = min(range(len(table)), key=lambda j: (d[j], j))
        assert i == best


def test_tables_hold_values_of_the_stored_type():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    w = rng.standard_normal((32, 32)) * 0.07
    t16, _ = C.palettize(w, "fp16")
    assert np.array_equal(t16, t16.astype(np.float16).astype(np.float64))
    v = rng.standard_normal(1000) * np.exp(rng.uniform(-10, 10, 1000))
    ref = torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(C._round_to(v, "bf16"), ref)


def test_kmeans_objective_never_increases():
    rng = np.random.default_rng(4)
    for x in (rng.standard_normal(20000), rng.laplace(size=20000), rng.random(20000) ** 3):
        _, hist = C.lloyd_1d(x)
        assert all(b <= a * (1 + 1e-12) for a, b in zip(hist, hist[1:]))


def test_uniform_data_gives_the_optimal_uniform_quantiser():
    """For U[0, 1) the optimal 64-level quantiser has centres (i + 1/2)/64 and
    mean squared error 1/(12 * 64^2)."""
    x = np.random.default_rng(5).random(50000)
    c, hist = C.lloyd_1d(x)
    assert np.max(np.abs(np.sort(c) - (np.arange(64) + 0.5) / 64)) < 0.25 / 64
    assert abs(hist[-1] / (1.0 / (12 * 64 * 64)) - 1.0) < 0.02


def test_objective_close_to_scikit_learn_kmeans():
    KMeans = pytest.importorskip("sklearn.cluster").KMeans
    x = np.random.default_rng(6).standard_normal(20000) * 0.03      # Xavier-scaled bell-shaped weights
    _, hist = C.lloyd_1d(x)
    km = KMeans(64, n_init=4, random_state=0).fit(x.reshape(-1, 1))
    assert hist[-1] <= 1.02 * km.inertia_ / x.size


def test_int8_bounds_extremes_and_half_even_ties():
    s = 0.01
    w = np.array([[0.5 * s, 1.5 * s, 2.5 * s, -2.5 * s, 127 * s], [0.0] * 5])
    q, scale = C.int8_quantize(w)
    assert abs(scale[0] - s) < 1e-18 and scale[1] == 1.0
    assert q[0].tolist() == [0, 2, 2, -2, 127] and q[1].tolist() == [0] * 5
    rng = np.random.default_rng(7)
    w = rng.standard_normal((20, 33)) * rng.uniform(0.01, 1, (20, 1))
    q, scale = C.int8_quantize(w)
    assert np.all(np.abs(q.astype(int)) <= 127)
    assert np.all(np.max(np.abs(q.astype(int)), axis=1) == 127)      # each row's extreme maps to +-127
    assert np.all(np.abs(C.int8_dequantize(q, scale) - w) <= scale[:, None] / 2 * (1 + 1e-12))


def test_only_the_encoder_matrices_change():
    W = synth.make_weights(TINY, 0)
    for scheme in ("palette6", "int8"):
        Wc = C.compress_weights(W, TINY.n_layers, scheme)
        changed = {k for k in W if not np.array_equal(np.asarray(W[k], np.float64), Wc[k])}
        assert changed == set(C.compressed_names(TINY.n_layers))
        assert all(np.asarray(W[k]).ndim >= 2 for k in changed)
        for k in changed:
            levels = np.unique(Wc[k])
            if scheme == "palette6":
                assert levels.size <= 64
            else:
                rows = Wc[k].reshape(Wc[k].shape[0], -1)
                assert all(np.unique(r).size <= 255 for r in rows)
