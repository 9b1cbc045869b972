"""Oracle: the log-mel front end (16 kHz audio -> 128-bin log-mel frames), fp64.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module.  It shares no code with the CUDA library
and never imports it.

Sources ("the pages"):
  * "Parakeet-EOU-120M — Streaming ASR Model", §Config: 16 kHz audio, 10 ms hop
    (160 samples), 128-bin mel frames.
  * "Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon", §1.3: a
    15-second window of 240,000 samples gives 1,501 mel frames of 128 bins, i.e.
    one frame per hop plus one — frames centred on every hop, the signal padded
    by half a transform on both sides.
  * "True streaming encode — implementation spec", §Status: the streaming front
    end pads only at the top of the first chunk and at the bottom on flush, and
    the streamed mel equals the one-shot mel exactly.

Readings where the pages are silent (each is listed in the design notes): the
usual NeMo-style filterbank front end —
  * pre-emphasis y[n] = x[n] - 0.97 x[n-1] (y[0] = x[0]);
  * a 512-point transform of 400-sample (25 ms) frames weighted by a symmetric
    Hann window centred in the 512 points; frame t centred on sample 160 t, the
    pre-emphasised signal padded with 256 zeros on both sides;
  * power spectrum |X|^2 of the 257 non-negative frequencies;
  * 128 triangular mel filters from 0 to 8 kHz on the Slaney mel scale (linear
    below 1 kHz at 200/3 Hz per mel, logarithmic above with a factor 6.4 per 27
    mels), each scaled by 2 / (its bandwidth in Hz) (Slaney area
    normalisation);
  * natural log of (filter energy + 2^-24); no dither and no per-utterance
    normalisation (a stream has no utterance statistics to normalise with).

Parity pins: tests/test_oracle_frontend_pins.py (torch.stft and scipy's lfilter
as library references, the Slaney scale's closed forms, the triangles'
partition of unity, pure tones, silence, the pages' 240,000 -> 1,501 frame
count, and streamed == one-shot output).  Readings that no page fixes (every
function is still pinned): the window, transform size, filter shape, log
guard and pre-emphasis above; the pins show they are stated correctly.
"""
from __future__ import annotations

import math

import numpy as np

SAMPLE_RATE = 16000
HOP = 160
WIN = 400
NFFT = 512
N_MELS = 128
F_MAX = SAMPLE_RATE / 2
PREEMPH = 0.97
LOG_GUARD = 2.0 ** -24

# Slaney mel scale
_F_SP = 200.0 / 3.0                 # Hz per mel below 1 kHz
_MIN_LOG_HZ = 1000.0
_MIN_LOG_MEL = _MIN_LOG_HZ / _F_SP  # 15
_LOGSTEP = math.log(6.4) / 27.0


def hz_to_mel(f):
    f = np.asarray(f, dtype=np.float64)
    lin = f / _F_SP
    return np.where(f >= _MIN_LOG_HZ, _MIN_LOG_MEL + np.log(np.maximum(f, 1e-300) / _MIN_LOG_HZ) / _LOGSTEP, lin)


def mel_to_hz(m):
    m = np.asarray(m, dtype=np.float64)
    return np.where(m >= _MIN_LOG_MEL, _MIN_LOG_HZ * np.exp(_LOGSTEP * (m - _MIN_LOG_MEL)), _F_SP * m)


def mel_edges():
    """Hz of the N_MELS + 2 filter edges, equally spaced in mel from 0 to F_MAX."""
    return mel_to_hz(np.linspace(hz_to_mel(0.0), hz_to_mel(F_MAX), N_MELS + 2))


def mel_filterbank():
    """[N_MELS][NFFT/2 + 1]: filter m rises linearly from edge m to edge m + 1 and
    falls to edge m + 2, times 2 / (edge m+2 - edge m)."""
    edges = mel_edges()
    freqs = np.linspace(0.0, SAMPLE_RATE / 2, NFFT // 2 + 1)
    fb = np.zeros((N_MELS, freqs.size))
    for m in range(N_MELS):
        lo, mid, hi = edges[m], edges[m + 1], edges[m + 2]
        rise = (freqs - lo) / (mid - lo)
        fall = (hi - freqs) / (hi - mid)
        fb[m] = np.maximum(0.0, np.minimum(rise, fall)) * (2.0 / (hi - lo))
    return fb


def hann_symmetric(n):
    k = np.arange(n, dtype=np.float64)
    return 0.5 - 0.5 * np.cos(2.0 * math.pi * k / (n - 1))


def frame_window():
    """The 400-point Hann window centred in the 512-point transform."""
    w = np.zeros(NFFT)
    off = (NFFT - WIN) // 2
    w[off:off + WIN] = hann_symmetric(WIN)
    return w


def preemphasis(x, prev=0.0):
    """y[n] = x[n] - 0.97 x[n-1], with x[-1] = prev (0 at a stream start)."""
    x = np.asarray(x, dtype=np.float64)
    y = x.copy()
    if x.size:
        y[0] = x[0] - PREEMPH * prev
        y[1:] = x[1:] - PREEMPH * x[:-1]
    return y


def n_frames(n_samples: int) -> int:
    """Frames of a signal of n_samples: one per hop, plus one."""
    return 1 + n_samples // HOP


def frame_logmel(seg, fb=None, win=None):
    """Log-mel of one 512-sample frame of the (padded) pre-emphasised signal."""
    fb = mel_filterbank() if fb is None else fb
    win = frame_window() if win is None else win
    spec = np.fft.rfft(np.asarray(seg, dtype=np.float64) * win)
    power = spec.real ** 2 + spec.imag ** 2
    return np.log(fb @ power + LOG_GUARD)


def logmel(x):
    """One-shot front end: [n_frames(len(x))][128] log-mel of 16 kHz audio x."""
    y = preemphasis(x)
    yp = np.concatenate([np.zeros(NFFT // 2), y, np.zeros(NFFT // 2)])
    fb, win = mel_filterbank(), frame_window()
    T = n_frames(len(y))
    return np.stack([frame_logmel(yp[t * HOP:t * HOP + NFFT], fb, win) for t in range(T)]) if T else \
        np.zeros((0, N_MELS))


class StreamingMel:
    """The same frames from audio pushed in pieces: frame t (centred on sample
    160 t) is emitted once samples up to 160 t + 255 have arrived; flush()
    treats the rest of its window as the bottom padding and emits the frames
    a one-shot call would still produce."""

    def __init__(self):
        self.prev = 0.0                      # last raw sample (pre-emphasis)
        self.buf = np.zeros(NFFT // 2)       # pre-emphasised samples from index base on (top padding first)
        self.base = -(NFFT // 2)             # signal index of buf[0]
        self.n = 0                           # samples received
        self.t = 0                           # next frame to emit
        self.fb, self.win = mel_filterbank(), frame_window()

    def _emit(self, limit_frames, padded):
        out = []
        while self.t < limit_frames:
            start = self.t * HOP - NFFT // 2            # signal index of the frame's first sample
            a = start - self.base
            seg = self.buf[a:a + NFFT]
            if seg.size < NFFT:
                if not padded:
                    break
                seg = np.concatenate([seg, np.zeros(NFFT - seg.size)])
            out.append(frame_logmel(seg, self.fb, self.win))
            self.t += 1
        # drop samples no later frame needs
        keep_from = self.t * HOP - NFFT // 2
        if keep_from > self.base:
            self.buf = self.buf[keep_from - self.base:]
            self.base = keep_from
        return np.stack(out) if out else np.zeros((0, N_MELS))

    def push(self, x):
        x = np.asarray(x, dtype=np.float64)
        y = preemphasis(x, self.prev)
        if x.size:
            self.prev = float(x[-1])
        self.buf = np.concatenate([self.buf, y])
        self.n += x.size
        complete = (self.n - NFFT // 2) // HOP + 1 if self.n >= NFFT // 2 else 0  # frames whose window is in
        return self._emit(complete, padded=False)

    def flush(self):
        return self._emit(n_frames(self.n), padded=True)
