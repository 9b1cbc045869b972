"""Host logic of the log-mel front end (include/cac_frontend.h) without a GPU:
the frame schedule of cac_frontend_schedule against the oracle's streaming
front end (oracle/frontend.py), push by push and at flush — integer
bookkeeping, compared exactly."""
import os

import numpy as np
import pytest

from oracle import frontend as F


@pytest.fixture(scope="module")
def native():
    from cache_aware_conformer_gb300 import native as nat
    if not os.path.exists(nat.LIB_PATH):
        from cache_aware_conformer_gb300 import build
        build.build()
    return nat


@pytest.mark.parametrize("sizes", [[2560] * 6, [1, 254, 1, 159, 1, 160, 3000, 0, 17], [255, 256, 257, 96, 64],
                                   [0, 0, 40000], [7] * 120])
def test_schedule_matches_the_oracle_stream(native, sizes):
    sm = F.StreamingMel()
    n = t = 0
    for k in sizes:
        got = native.frontend_schedule(n, t, k, False)
        assert got == sm.push(np.zeros(k)).shape[0], (n, k)
        n, t = n + k, t + got
    last = native.frontend_schedule(n, t, 0, True)
    assert last == sm.flush().shape[0]
    assert t + last == F.n_frames(n)


def test_schedule_one_shot_and_the_pages_window(native):
    assert native.frontend_schedule(0, 0, 240000, True) == 1501      # 15 s window -> 1,501 frames
    assert native.frontend_schedule(0, 0, 0, True) == 1              # an empty stream still has frame 0
    assert native.frontend_schedule(0, 0, 255, False) == 0
    assert native.frontend_schedule(0, 0, 256, False) == 1
    assert native.frontend_schedule(-1, 0, 1, False) == -1                # CAC_E_INVAL


def test_schedule_flush_after_a_ragged_stream(native):
    rng = np.random.default_rng(5)
    for _ in range(50):
        sizes = rng.integers(0, 4000, size=int(rng.integers(1, 8)))
        n = t = 0
        for k in sizes:
            f = native.frontend_schedule(n, t, int(k), False)
            n, t = n + int(k), t + f
        tail = int(rng.integers(0, 500))
        assert t + native.frontend_schedule(n, t, tail, True) == F.n_frames(n + tail)


def test_kernel_tables_match_the_oracle(native):
    """The window, twiddles and sparse mel rows the kernel reads equal the
    oracle's fp64 definitions rounded once to fp32, and the 16-bin rows hold
    every nonzero weight of each filter."""
    win, tw, st, mw = native.frontend_tables()
    np.testing.assert_array_equal(win, F.frame_window().astype(np.float32))
    k = np.arange(256)
    np.testing.assert_array_equal(tw[:, 0], np.cos(2 * np.pi * k / 512).astype(np.float32))
    np.testing.assert_array_equal(tw[:, 1], (-np.sin(2 * np.pi * k / 512)).astype(np.float32))
    fb = F.mel_filterbank()
    dense = np.zeros_like(fb)
    for m in range(F.N_MELS):
        assert 0 <= st[m] <= fb.shape[1] - 16
        dense[m, st[m]:st[m] + 16] = mw[m]
    np.testing.assert_allclose(dense, fb.astype(np.float32), rtol=0, atol=1e-9)
    assert np.array_equal(dense != 0, fb != 0)


def test_frames_per_call_stay_within_the_bindings_capacity(native):
    """A push emits at most n/160 + 1 frames and a flush at most n/160 + 3
    (the binding sizes its default output by these bounds)."""
    rng = np.random.default_rng(8)
    for _ in range(3000):
        n = int(rng.integers(0, 200000))
        t = native.frontend_schedule(0, 0, n, False)
        ns = int(rng.integers(0, 6000))
        assert native.frontend_schedule(n, t, ns, False) <= ns // 160 + 1
        assert native.frontend_schedule(n, t, ns, True) <= ns // 160 + 3
