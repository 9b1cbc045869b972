"""GPU parity of the streaming log-mel front end (include/cac_frontend.h)
against the fp64 oracle (oracle/frontend.py).

Frames: 16 kHz, 160-sample hop, 128 bins ("Parakeet-EOU-120M — Streaming ASR
Model", §Config), 240,000 samples -> 1,501 frames ("Fast Accuracy-Preserving
RNNT Beam Search on Apple Silicon", §1.3), padding only at the stream's top
and at flush, streamed == one-shot ("True streaming encode — implementation
spec", §Status).  Every stream's streamed GPU frames are compared with the
oracle's one-shot transform of the same audio (the oracle's own streamed ==
one-shot equality is pinned on the CPU).

Tolerance (fp32 kernel vs fp64 oracle): a 512-point fp32 FFT is accurate to a
few 1e-7 of the frame's spectral norm, so a filter energy E_m carries an
absolute error of about 1e-6 of the frame's largest filter energy E_max.
Filters with E_m >= 1e-3 E_max therefore get |delta log| <= 1e-3; weaker
filters are compared in the energy domain, |exp(gpu) - exp(ref)| <= 1e-6 E_max.
Integer bookkeeping (frames per call, counters) is compared exactly."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from cache_aware_conformer_gb300 import synth  # noqa: E402
from oracle import frontend as F  # noqa: E402

pytestmark = pytest.mark.gpu


def _assert_logmel_close(gpu, ref, what):
    gpu, ref = np.asarray(gpu, np.float64), np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    if not gpu.size:
        return
    assert np.isfinite(gpu).all(), what
    E = np.exp(ref)
    Emax = E.max(axis=1, keepdims=True)
    strong = E >= 1e-3 * Emax
    dlog = np.abs(gpu - ref)
    dE = np.abs(np.exp(gpu) - E)
    assert (dlog[strong] <= 1e-3).all(), (what, float(dlog[strong].max()))
    assert (dE[~strong] <= 1e-6 * np.broadcast_to(Emax, E.shape)[~strong]).all(), what
    print(f"[parity] {what}: max|dlog| strong {dlog[strong].max():.2e}, all {dlog.max():.2e}")


def _run(fe, ids, audio, sizes, flush_each):
    """Push audio[:, ...] in pieces of `sizes` (same size for every slot per call),
    then flush the per-slot remainders; returns per-slot frame arrays."""
    n = len(ids)
    got = [[] for _ in range(n)]
    pos = 0
    for k in sizes:
        chunk = torch.from_numpy(np.ascontiguousarray(audio[:, pos:pos + k])).cuda() if k else None
        counts_before = [fe.state(i)[1] for i in ids]
        outs = fe.push(ids, chunk) if k else fe.push(ids, None, max_frames=1)
        for b in range(n):
            got[b].append(outs[b].cpu().numpy())
            s, f, fin = fe.state(ids[b])
            assert s == pos + k and f == counts_before[b] + outs[b].shape[0] and fin == 0
        pos += k
    rest = max(flush_each)
    tail = torch.from_numpy(np.ascontiguousarray(audio[:, pos:pos + rest])).cuda() if rest else None
    outs = fe.push(ids, tail, flush=True, n_samples_each=list(flush_each))
    for b in range(n):
        got[b].append(outs[b].cpu().numpy())
    return [np.concatenate(g) for g in got]


@pytest.mark.parametrize("sizes", [
    [1, 254, 1, 159, 1, 160, 3000, 0, 17, 2560],
    [2560] * 8,
    [255, 256, 257, 96, 64, 7, 7, 7],
    [40000],
])
def test_streamed_frames_match_the_oracle(sizes):
    from cache_aware_conformer_gb300 import native
    ids = [5, 2, 7]                                   # non-contiguous slots
    fe = native.Frontend(max_streams=8)
    flush_each = [0, 333, 1700]
    n_total = sum(sizes) + max(flush_each)
    audio = np.stack([synth.make_audio(n_total, sid) for sid in ids])
    got = _run(fe, ids, audio, sizes, flush_each)
    for b, sid in enumerate(ids):
        n_b = sum(sizes) + flush_each[b]
        ref = F.logmel(audio[b, :n_b].astype(np.float64))
        assert got[b].shape[0] == F.n_frames(n_b)
        _assert_logmel_close(got[b], ref, f"stream {sid}, pushes {sizes[:4]}...")
        s, f, fin = fe.state(sid)
        assert (s, f, fin) == (n_b, F.n_frames(n_b), 1)
    fe.close()


def test_the_pages_window_gives_1501_frames():
    from cache_aware_conformer_gb300 import native
    fe = native.Frontend(max_streams=1)
    audio = synth.make_audio(240000, 0)
    outs = fe.push([0], torch.from_numpy(audio[None]).cuda(), flush=True, n_samples_each=[240000])
    assert outs[0].shape == (1501, 128)
    _assert_logmel_close(outs[0].cpu().numpy(), F.logmel(audio.astype(np.float64)), "15 s window")


def test_reset_starts_a_fresh_stream():
    from cache_aware_conformer_gb300 import native
    fe = native.Frontend(max_streams=4)
    a_old = synth.make_audio(5000, 11)
    fe.push([1], torch.from_numpy(a_old[None, :3333]).cuda())
    fe.reset([1])
    assert fe.state(1) == (0, 0, 0)
    a_new = synth.make_audio(6000, 12)
    got = _run(fe, [1], a_new[None], [2000, 1, 1999], [2000])
    _assert_logmel_close(got[0], F.logmel(a_new.astype(np.float64)), "after reset")
    # a flushed stream refuses pushes until its reset
    with pytest.raises(native.CacError):
        fe.push([1], torch.zeros(1, 160, device="cuda"))
    fe.close()


def test_silence_and_an_empty_stream():
    from cache_aware_conformer_gb300 import native
    fe = native.Frontend(max_streams=2)
    z = np.zeros((2, 4000), np.float32)
    got = _run(fe, [0, 1], z, [1600, 1600], [800, 0])
    guard = np.log(2.0 ** -24)
    for b, n_b in enumerate((4000, 3200)):
        assert got[b].shape == (F.n_frames(n_b), 128)
        np.testing.assert_allclose(got[b], guard, rtol=0, atol=1e-6)
    fe2 = native.Frontend(max_streams=1)
    outs = fe2.push([0], None, flush=True, n_samples_each=[0])
    assert outs[0].shape == (1, 128)


def test_many_streams_160ms_pushes():
    """The bench's shape: 256 streams pushed 2,560 samples (160 ms) at a time;
    streams 0, 100 and 255 compared after 1 s and a flush."""
    from cache_aware_conformer_gb300 import native
    S = 256
    fe = native.Frontend(max_streams=S)
    ids = list(range(S))
    n = 6 * 2560 + 900
    audio = np.stack([synth.make_audio(n, sid) for sid in ids])
    got = _run(fe, ids, audio, [2560] * 6, [900] * S)
    for sid in (0, 100, 255):
        _assert_logmel_close(got[sid], F.logmel(audio[sid].astype(np.float64)), f"stream {sid} of 256")
    fe.close()


def test_push_beyond_capacity_is_rejected_without_state_change():
    from cache_aware_conformer_gb300 import native
    fe = native.Frontend(max_streams=1)
    mel = torch.empty(1, 2, 128, device="cuda")
    with pytest.raises(native.CacError) as e:
        fe.push_into([0], torch.zeros(1, 2560, device="cuda"), mel)    # 15 frames > 2
    assert e.value.code == -10
    assert fe.state(0) == (0, 0, 0)
