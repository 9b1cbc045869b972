"""The offline encode entry point that allocates nothing (cac_encode_offline_noalloc).

It serves callers that may not allocate device memory once they are running:
a real-time audio callback cannot wait on cudaMalloc (which may block and
synchronize the device), and some hosts give the library a fixed memory
budget up front.  The entry point runs the offline encode on the library's
fixed device-side scratch array instead of a cudaMalloc-grown workspace.
These checks call it through the C ABI and compare it with the allocating
cac_encode_offline on the same inputs, twice in a row (the shared array keeps
the previous call's contents, so the second call shows nothing stale leaks),
within the bf16 tolerance the other GPU tests use.  This file is collected
last so that a stop-at-first-failure run has already run every other test."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import EOU_120M  # noqa: E402

from _util import BF16_MAX_ABS, cosine, max_abs  # noqa: E402

pytestmark = pytest.mark.gpu


def _inputs(lens, seed):
    t = max(lens)
    batch = np.zeros((len(lens), t, 128), np.float32)
    for k, n in enumerate(lens):
        batch[k, :n] = synth.make_mel(n, seed + k)
    return torch.from_numpy(batch).cuda()


def test_noalloc_matches_allocating_offline_encode_twice():
    from cache_aware_conformer_gb300 import native
    cfg = replace(EOU_120M, n_layers=3)
    W = synth.make_weights(cfg, 0)
    model = native.Model(cfg, synth.pack_weights(cfg, W))
    for call, (lens, seed) in enumerate([([1501, 640, 37], 500), ([903, 1200], 600)]):
        mel = _inputs(lens, seed)
        e_ref, j_ref, n_ref = model.encode_offline(mel, lens)
        # fresh outputs filled with garbage: every valid frame must be written
        T = e_ref.shape[1]
        enc = torch.full((len(lens), T, cfg.d_model), float("nan"), device="cuda")
        joint = torch.full((len(lens), T, cfg.joint_dim), float("nan"), device="cuda")
        e, j, n = model.encode_offline(mel, lens, out=(enc, joint), noalloc=True)
        model.check()
        assert n == n_ref
        for k, nk in enumerate(n):
            a, b = e[k, :nk].cpu().numpy(), e_ref[k, :nk].cpu().numpy()
            assert np.isfinite(a).all(), (call, k)
            assert max_abs(a, b) <= BF16_MAX_ABS and cosine(a, b) >= 0.999, (call, k)
            assert max_abs(j[k, :nk].cpu().numpy(), j_ref[k, :nk].cpu().numpy()) <= 2 * BF16_MAX_ABS


def test_noalloc_rejects_requests_beyond_its_scratch():
    from cache_aware_conformer_gb300 import native
    cfg = replace(EOU_120M, n_layers=1)
    model = native.Model(cfg, synth.pack_weights(cfg, synth.make_weights(cfg, 0)))
    mel = torch.zeros(16, 1501, 128, device="cuda")           # ~24,000 mel frames
    with pytest.raises(native.CacError) as e:
        model.encode_offline(mel, [1501] * 16, noalloc=True)
    assert e.value.code == -10
