"""Pins of the log-mel front-end oracle (oracle/frontend.py) to things other
than itself: torch.stft and scipy's lfilter as library references, closed
forms of the Slaney mel scale, the triangles' partition of unity, pure tones,
silence, the pages' frame count, and streamed == one-shot output ("True
streaming encode — implementation spec", §Status)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import frontend as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_facts.json")


def _audio(n, seed=3):
    return np.random.default_rng(seed).standard_normal(n) * 0.1


def test_frame_count_is_the_pages():
    facts = json.load(open(GOLDEN))["mel_frontend"]
    assert F.SAMPLE_RATE == facts["sample_rate"] and F.HOP == facts["hop"] and F.N_MELS == facts["mel_bins"]
    assert F.n_frames(facts["samples"]) == facts["mel_frames"]          # 240,000 -> 1,501
    x = np.zeros(facts["samples"])
    assert F.logmel(x).shape == (facts["mel_frames"], facts["mel_bins"])


def test_slaney_scale_closed_forms():
    assert F.hz_to_mel(0.0) == 0.0
    assert abs(F.hz_to_mel(1000.0) - 15.0) < 1e-12                    # 1 kHz = 15 mels
    assert abs(F.hz_to_mel(500.0) - 7.5) < 1e-12                      # linear region: 200/3 Hz per mel
    assert abs(F.hz_to_mel(6400.0) - 42.0) < 1e-9                     # factor 6.4 per 27 mels above 1 kHz
    m = np.linspace(0, 45, 91)
    np.testing.assert_allclose(F.hz_to_mel(F.mel_to_hz(m)), m, atol=1e-9)


def test_preemphasis_matches_lfilter():
    signal = pytest.importorskip("scipy.signal")
    x = _audio(1000)
    np.testing.assert_allclose(F.preemphasis(x), signal.lfilter([1.0, -F.PREEMPH], [1.0], x), atol=1e-12)


def test_power_spectrum_matches_torch_stft():
    torch = pytest.importorskip("torch")
    y = F.preemphasis(_audio(16000))
    win = torch.hann_window(F.WIN, periodic=False, dtype=torch.float64)
    X = torch.stft(torch.from_numpy(y), n_fft=F.NFFT, hop_length=F.HOP, win_length=F.WIN, window=win,
                   center=True, pad_mode="constant", return_complex=True)
    ref = (X.abs() ** 2).numpy().T                                    # [frames][257]
    yp = np.concatenate([np.zeros(F.NFFT // 2), y, np.zeros(F.NFFT // 2)])
    w = F.frame_window()
    ours = np.stack([np.abs(np.fft.rfft(yp[t * F.HOP:t * F.HOP + F.NFFT] * w)) ** 2
                     for t in range(F.n_frames(len(y)))])
    assert ours.shape == ref.shape
    np.testing.assert_allclose(ours, ref, rtol=1e-9, atol=1e-12)
    # the whole chain: natural log of the filter energies of torch's power spectrum
    full = np.log(ref @ F.mel_filterbank().T + F.LOG_GUARD)
    np.testing.assert_allclose(F.logmel(_audio(16000)), full, rtol=0, atol=1e-9)


def test_triangles_partition_unity_and_edges():
    """Without the area scaling the triangles sum to 1 between the first and
    last centres; each filter is zero outside its two neighbouring edges."""
    fb, edges = F.mel_filterbank(), F.mel_edges()
    freqs = np.linspace(0.0, F.SAMPLE_RATE / 2, F.NFFT // 2 + 1)
    unscaled = fb * ((edges[2:] - edges[:-2]) / 2.0)[:, None]
    inside = (freqs >= edges[1]) & (freqs <= edges[-2])
    np.testing.assert_allclose(unscaled.sum(0)[inside], 1.0, atol=1e-9)
    for m in range(F.N_MELS):
        outside = (freqs <= edges[m]) | (freqs >= edges[m + 2])
        assert np.all(fb[m][outside] == 0.0)
    assert np.all(fb >= 0.0)


def test_pure_tone_lands_in_its_filter():
    """A tone at a filter's centre frequency gives that filter the most energy
    (above ~1.5 kHz: lower down the filters are ~23 Hz apart, closer than the
    31.25 Hz transform bins, and the window's leakage decides)."""
    edges = F.mel_edges()
    t = np.arange(16000) / F.SAMPLE_RATE
    for m in (60, 90, 110):
        x = np.sin(2 * math.pi * edges[m + 1] * t)
        lm = F.logmel(x)[10:-10]
        assert np.all(np.argmax(lm, axis=1) == m), m


def test_silence_is_the_log_guard():
    lm = F.logmel(np.zeros(3200))
    assert lm.shape == (21, F.N_MELS)
    assert np.all(lm == math.log(F.LOG_GUARD))


@pytest.mark.parametrize("sizes", [[2560] * 10 + [1234], [1000, 3333, 17, 1, 160, 255, 256, 4000], [1] * 700])
def test_streamed_equals_one_shot(sizes):
    x = _audio(sum(sizes), seed=len(sizes))
    ref = F.logmel(x)
    sm = F.StreamingMel()
    parts, off = [], 0
    for n in sizes:
        parts.append(sm.push(x[off:off + n]))
        off += n
    parts.append(sm.flush())
    got = np.concatenate(parts)
    assert got.shape == ref.shape
    np.testing.assert_array_equal(got, ref)


def test_streaming_emits_only_complete_windows():
    sm = F.StreamingMel()
    assert sm.push(np.zeros(255)).shape[0] == 0        # frame 0 needs samples up to 255
    assert sm.push(np.zeros(1)).shape[0] == 1
    assert sm.push(np.zeros(159)).shape[0] == 0
    assert sm.push(np.zeros(1)).shape[0] == 1          # frame 1 needs samples up to 415
    assert sm.flush().shape[0] == F.n_frames(416) - 2
