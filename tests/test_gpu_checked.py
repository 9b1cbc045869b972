"""Memory checks that stand in for a memory checker (compute-sanitizer is not
available on this pool): guard zones around every per-stream device pool —
K/V rings, conv ring, provisional x0 ring — in both builds, and the CAC_CHECKED
build's index checks (libcac_checked.so, selected with CAC_LIB=checked), under
which the whole GPU suite can run: every stream id, position and ring slot is
checked before use, an out-of-range one latches CAC_E_BOUNDS (which each
test's pool.check() would raise) and the access is skipped — no trap, no
wait."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import EOU_120M, EOU_RC3  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _pool(cfg, S, nmax=2):
    from cache_aware_conformer_gb300 import native
    model = native.Model(cfg, synth.pack_weights(cfg, synth.make_weights(cfg, 0)))
    pool = native.Pool(model, S, nmax)
    return model, pool, [pool.create_stream() for _ in range(S)]


def test_guard_zones_intact_after_pushes_resets_wraps_and_flushes():
    """Every K/V ring slot (positions well past the 72-row ring), the conv ring
    and the stream ids up to the pool's last one are written; nothing lands in
    a guard zone."""
    cfg = replace(EOU_120M, n_layers=2)
    S = 70
    model, pool, ids = _pool(cfg, S)
    pool.check_guards()
    mel = torch.from_numpy(np.stack([synth.make_mel(16 * 40 + 8, 700 + s) for s in range(S)])).to(DEV)
    for t in range(40):
        if t in (7, 23):
            pool.reset([ids[0], ids[S - 1]])
        pool.push(ids, mel[:, 16 * t:16 * (t + 1)].contiguous())
    pool.flush(ids, mel[:, 640:648].contiguous(), [8] * S)
    pool.check()
    pool.check_guards()


def test_guard_zones_intact_in_a_provisional_pool():
    cfg = replace(EOU_RC3, n_layers=2)
    S = 9
    model, pool, ids = _pool(cfg, S, nmax=4)
    mel = torch.from_numpy(np.stack([synth.make_mel(32 * 12 + 24, 900 + s) for s in range(S)])).to(DEV)
    for t in range(12):
        if t == 5:
            pool.reset([ids[3]])
        pool.push(ids, mel[:, 32 * t:32 * (t + 1)].contiguous())
    pool.flush(ids, mel[:, 384:408].contiguous(), [24] * S)
    pool.check()
    pool.check_guards()


def test_index_check_of_the_checked_build():
    """In the checked build an out-of-range index is caught, the access skipped
    and CAC_E_BOUNDS latched; the default build has no checks to exercise."""
    from cache_aware_conformer_gb300 import native
    if native.build_checked():
        assert native.bounds_selftest() == -11
    else:
        assert native.bounds_selftest() == -9
