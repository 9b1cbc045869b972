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
