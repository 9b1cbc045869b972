"""Seeded synthetic inputs: model weights, log-mel streams, start offsets, resets.

This module is the only code shared by the oracle's tests and the CUDA path's
tests; it holds none of the encoder's arithmetic.  Every value comes from one
counter-based generator so that any tensor element can be regenerated alone:

    splitmix64(z):  z += 0x9E3779B97F4A7C15
                    z  = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
                    z  = (z ^ (z >> 27)) * 0x94D049BB133111EB
                    return z ^ (z >> 31)                       (all mod 2^64)
    key(seed, tid)  = splitmix64(splitmix64(seed) ^ tid)
    bits(key, i)    = splitmix64(key + i)
    uniform(key, i) = (bits(key, i) >> 11) * 2^-53             in [0, 1)
    normal(key, i)  = sqrt(-2 ln(1 - uniform(key, 2i))) * cos(2 pi uniform(key, 2i + 1))

Weights (seed 0 by default) follow the synthetic init of the workloads:
Xavier-normal linears and convolutions (std = sqrt(2 / (fan_in + fan_out)),
fan = channels x taps for convolutions, 9 / 9 for the depthwise kernel), LayerNorm
and folded-BatchNorm gains uniform on [0.9, 1.1], every bias, LayerNorm/BatchNorm
shift and the positional biases pos_bias_u / pos_bias_v ~ N(0, 0.02^2).  In bf16
configurations every parameter is rounded to the nearest bf16 value (ties to
even) here, so the device copy is exact and the oracle sees the same numbers.

Log-mel (seed 1000 + stream id) is N(0, 1) with near-silence spans N(-4, 0.3^2);
span lengths are uniform on 30..200 mel frames and spans are placed until they
cover the requested fraction of frames.
"""
from __future__ import annotations

import numpy as np

from .config import ModelConfig, DTYPE_BF16

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLD = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)

TID_MEL = 1 << 20
TID_SPANS = (1 << 20) + 1
TID_OFFSETS = (1 << 20) + 2
TID_RESETS = (1 << 20) + 3


def splitmix64(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = z + _GOLD
        z = (z ^ (z >> np.uint64(30))) * _C1
        z = (z ^ (z >> np.uint64(27))) * _C2
    return z ^ (z >> np.uint64(31))


def key(seed: int, tid: int) -> np.uint64:
    return splitmix64(splitmix64(np.uint64(seed)) ^ np.uint64(tid))


def uniform(k: np.uint64, idx: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        b = splitmix64(np.uint64(k) + np.asarray(idx, dtype=np.uint64))
    return (b >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(k: np.uint64, n: int, start: int = 0) -> np.ndarray:
    i = np.arange(start, start + n, dtype=np.uint64)
    u1 = uniform(k, 2 * i)
    u2 = uniform(k, 2 * i + np.uint64(1))
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even), kept as float32."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return (b << np.uint64(16)).astype(np.uint32).view(np.float32)


# ---------------------------------------------------------------------------
# Weight layout.  All linears are stored [out, in]; the subsampling
# convolutions [out, tap, in]; the depthwise kernel [channel, tap].
# ---------------------------------------------------------------------------

def weight_layout(cfg: ModelConfig):
    """Ordered (name, shape, kind) list; the flat blob is their concatenation.

    kind: ("xavier", fan_in, fan_out) | "gain" | "bias".
    """
    D, F, M, J, K, H = cfg.d_model, cfg.ff_dim, cfg.mel_bins, cfg.joint_dim, cfg.dw_kernel, cfg.n_heads
    HD = D // H
    L = []
    L += [("sub.w1", (D, 3, M), ("xavier", 3 * M, 3 * D)), ("sub.b1", (D,), "bias"),
          ("sub.w2", (D, 3, D), ("xavier", 3 * D, 3 * D)), ("sub.b2", (D,), "bias"),
          ("sub.w3", (D, 3, D), ("xavier", 3 * D, 3 * D)), ("sub.b3", (D,), "bias"),
          ("sub.wo", (D, D), ("xavier", D, D)), ("sub.bo", (D,), "bias")]
    for l in range(cfg.n_layers):
        p = f"l{l}."
        L += [(p + "ff1.ln_g", (D,), "gain"), (p + "ff1.ln_b", (D,), "bias"),
              (p + "ff1.w1", (F, D), ("xavier", D, F)), (p + "ff1.b1", (F,), "bias"),
              (p + "ff1.w2", (D, F), ("xavier", F, D)), (p + "ff1.b2", (D,), "bias")]
        L += [(p + "att.ln_g", (D,), "gain"), (p + "att.ln_b", (D,), "bias"),
              (p + "att.wq", (D, D), ("xavier", D, D)), (p + "att.bq", (D,), "bias"),
              (p + "att.wk", (D, D), ("xavier", D, D)), (p + "att.bk", (D,), "bias"),
              (p + "att.wv", (D, D), ("xavier", D, D)), (p + "att.bv", (D,), "bias"),
              (p + "att.wo", (D, D), ("xavier", D, D)), (p + "att.bo", (D,), "bias"),
              (p + "att.wpos", (D, D), ("xavier", D, D)),
              (p + "att.pbu", (H, HD), "bias"), (p + "att.pbv", (H, HD), "bias")]
        L += [(p + "conv.ln_g", (D,), "gain"), (p + "conv.ln_b", (D,), "bias"),
              (p + "conv.w_pw1", (2 * D, D), ("xavier", D, 2 * D)), (p + "conv.b_pw1", (2 * D,), "bias"),
              (p + "conv.w_dw", (D, K), ("xavier", K, K)), (p + "conv.b_dw", (D,), "bias"),
              (p + "conv.bn_g", (D,), "gain"), (p + "conv.bn_b", (D,), "bias"),
              (p + "conv.w_pw2", (D, D), ("xavier", D, D)), (p + "conv.b_pw2", (D,), "bias")]
        L += [(p + "ff2.ln_g", (D,), "gain"), (p + "ff2.ln_b", (D,), "bias"),
              (p + "ff2.w1", (F, D), ("xavier", D, F)), (p + "ff2.b1", (F,), "bias"),
              (p + "ff2.w2", (D, F), ("xavier", F, D)), (p + "ff2.b2", (D,), "bias")]
        L += [(p + "out.ln_g", (D,), "gain"), (p + "out.ln_b", (D,), "bias")]
    L += [("joint.w", (J, D), ("xavier", D, J)), ("joint.b", (J,), "bias")]
    return L


def weights_size(cfg: ModelConfig) -> int:
    return int(sum(np.prod(s) for _, s, _ in weight_layout(cfg)))


def make_weights(cfg: ModelConfig, seed: int = 0) -> dict:
    """Named float32 parameter arrays (bf16-representable in bf16 configurations)."""
    return dict(_make_tensor((cfg, seed, tid)) for tid in range(len(weight_layout(cfg))))


def pack_weights(cfg: ModelConfig, w: dict) -> np.ndarray:
    """Flat float32 blob in weight_layout order (the C library's input format)."""
    parts = []
    for name, shape, _ in weight_layout(cfg):
        a = np.asarray(w[name], dtype=np.float32)
        assert a.shape == tuple(shape), (name, a.shape, shape)
        parts.append(a.reshape(-1))
    return np.ascontiguousarray(np.concatenate(parts))


def make_mel(n_frames: int, stream_id: int, mel_bins: int = 128, silence_frac: float = 0.2,
             seed_base: int = 1000) -> np.ndarray:
    """[n_frames, mel_bins] float32 synthetic log-mel with near-silence spans."""
    seed = seed_base + stream_id
    x = normal(key(seed, TID_MEL), n_frames * mel_bins).reshape(n_frames, mel_bins)
    silent = np.zeros(n_frames, dtype=bool)
    target = int(round(silence_frac * n_frames))
    ks = key(seed, TID_SPANS)
    draw = 0
    while silent.sum() < target and draw < 4 * n_frames + 8:
        u = uniform(ks, np.array([draw, draw + 1], dtype=np.uint64))
        draw += 2
        length = 30 + int(u[0] * 171)
        start = int(u[1] * max(1, n_frames - length + 1))
        silent[start:start + length] = True
    ksil = key(seed, TID_MEL + 7)
    quiet = -4.0 + 0.3 * normal(ksil, n_frames * mel_bins).reshape(n_frames, mel_bins)
    x = np.where(silent[:, None], quiet, x)
    return x.astype(np.float32)


def start_offsets(n_streams: int, max_offset: int, seed: int = 7) -> np.ndarray:
    """Even start offsets in subsampled frames: 2 * floor(u / 2), u uniform on 0..max_offset-1."""
    if max_offset <= 0:
        return np.zeros(n_streams, dtype=np.int64)
    u = uniform(key(seed, TID_OFFSETS), np.arange(n_streams, dtype=np.uint64))
    raw = np.floor(u * max_offset).astype(np.int64)
    return 2 * (raw // 2)


def reset_mask(n_streams: int, step: int, prob: float, seed: int = 11) -> np.ndarray:
    """Streams that reset before push `step` (independent Bernoulli(prob) per stream and step)."""
    if prob <= 0:
        return np.zeros(n_streams, dtype=bool)
    idx = np.arange(n_streams, dtype=np.uint64) * np.uint64(1 << 32) + np.uint64(step)
    return uniform(key(seed, TID_RESETS), idx) < prob


def unpack_weights(cfg: ModelConfig, blob: np.ndarray) -> dict:
    """Inverse of pack_weights: named views into a flat float32 blob."""
    out, off = {}, 0
    for name, shape, _ in weight_layout(cfg):
        n = int(np.prod(shape))
        out[name] = np.asarray(blob[off:off + n]).reshape(shape)
        off += n
    assert off == blob.size
    return out


def _make_tensor(args):
    cfg, seed, tid = args
    name, shape, kind = weight_layout(cfg)[tid]
    n = int(np.prod(shape))
    k = key(seed, tid)
    if kind == "gain":
        v = 0.9 + 0.2 * uniform(k, np.arange(n, dtype=np.uint64))
    elif kind == "bias":
        v = 0.02 * normal(k, n)
    else:
        _, fi, fo = kind
        v = np.sqrt(2.0 / (fi + fo)) * normal(k, n)
    v = v.astype(np.float32).reshape(shape)
    if cfg.dtype == DTYPE_BF16:
        v = round_bf16(v).reshape(shape)
    return name, v


def make_weights_parallel(cfg: ModelConfig, seed: int = 0, workers: int = 8) -> dict:
    """Same values as make_weights, generated by a spawn process pool."""
    import multiprocessing as mp
    tids = list(range(len(weight_layout(cfg))))
    with mp.get_context("spawn").Pool(workers) as pool:
        items = pool.map(_make_tensor, [(cfg, seed, t) for t in tids], chunksize=4)
    return dict(items)


# ---------------------------------------------------------------------------
# Greedy RNN-T decoder (fp32): weights and projected encoder frames
# ---------------------------------------------------------------------------

TID_DEC = 1 << 21          # decoder weights: TID_DEC + index in decoder_layout
TID_JOINT_FRAMES = (1 << 21) + 1000


def decoder_layout(dcfg):
    """Ordered (name, shape, kind) of the decoder parameters; linears [out, in],
    LSTM gate rows in the order input, forget, cell, output."""
    C, P, J = dcfg.classes, dcfg.pred_dim, dcfg.joint_dim
    return [("emb", (C, P), "embed"),
            ("lstm.w_ih", (4 * P, P), ("xavier", P, 4 * P)), ("lstm.w_hh", (4 * P, P), ("xavier", P, 4 * P)),
            ("lstm.b_ih", (4 * P,), "bias"), ("lstm.b_hh", (4 * P,), "bias"),
            ("pred.w", (J, P), ("xavier", P, J)), ("pred.b", (J,), "bias"),
            ("out.w", (C, J), ("xavier", J, C)), ("out.b", (C,), "out_bias")]


def make_decoder_weights(dcfg, seed: int = 0) -> dict:
    """Named float32 decoder parameters: Xavier-normal linears, N(0, 1)
    embedding rows, N(0, 0.02^2) biases; the output bias of the blank class is
    raised by dcfg.blank_bias so that most decisions are blank, as in speech."""
    out = {}
    for tid, (name, shape, kind) in enumerate(decoder_layout(dcfg)):
        n = int(np.prod(shape))
        k = key(seed, TID_DEC + tid)
        if kind == "embed":
            v = normal(k, n)
        elif kind in ("bias", "out_bias"):
            v = 0.02 * normal(k, n)
            if kind == "out_bias":
                v[dcfg.blank] += dcfg.blank_bias
        else:
            _, fi, fo = kind
            v = np.sqrt(2.0 / (fi + fo)) * normal(k, n)
        out[name] = v.astype(np.float32).reshape(shape)
    return out


def pack_decoder_weights(dcfg, w: dict) -> np.ndarray:
    """Flat float32 blob in decoder_layout order (the C library's input format)."""
    parts = []
    for name, shape, _ in decoder_layout(dcfg):
        a = np.asarray(w[name], dtype=np.float32)
        assert a.shape == tuple(shape), (name, a.shape, shape)
        parts.append(a.reshape(-1))
    return np.ascontiguousarray(np.concatenate(parts))


def make_joint_frames(n_frames: int, stream_id: int, joint_dim: int = 640, seed_base: int = 3000) -> np.ndarray:
    """[n_frames, joint_dim] float32 stand-in for projected encoder frames: N(0, 1)."""
    k = key(seed_base + stream_id, TID_JOINT_FRAMES)
    return normal(k, n_frames * joint_dim).reshape(n_frames, joint_dim).astype(np.float32)


def _mel_job(args):
    n_frames, sid, silence_frac = args
    return make_mel(n_frames, sid, silence_frac=silence_frac)


def make_mels_parallel(n_frames: int, stream_ids, silence_frac: float = 0.2, workers: int = 8) -> np.ndarray:
    """[len(stream_ids), n_frames, 128] synthetic mel, generated by a spawn process pool."""
    import multiprocessing as mp
    with mp.get_context("spawn").Pool(workers) as pool:
        return np.stack(pool.map(_mel_job, [(n_frames, int(s), silence_frac) for s in stream_ids]))


TID_AUDIO = (1 << 21) + 2000


def make_audio(n_samples: int, stream_id: int, silence_frac: float = 0.2, seed_base: int = 5000) -> np.ndarray:
    """[n_samples] float32 speech-like 16 kHz audio: a voiced source (five
    harmonics of a pitch gliding between 100 and 250 Hz, amplitude 0.2) plus
    white noise (0.02), with silent spans (exact zeros) covering about
    silence_frac of the signal."""
    k = key(seed_base + stream_id, TID_AUDIO)
    u = uniform(k, np.arange(4, dtype=np.uint64))
    t = np.arange(n_samples) / 16000.0
    f0 = 100.0 + 150.0 * (0.5 + 0.5 * np.sin(2 * np.pi * (0.3 + 0.4 * u[0]) * t + 6.283 * u[1]))
    phase = 2 * np.pi * np.cumsum(f0) / 16000.0
    x = sum((0.2 / h) * np.sin(h * phase) for h in range(1, 6))
    x = x + 0.02 * normal(k, n_samples, start=2)
    span = 4800                                      # 0.3 s silent spans
    n_span = int(round(silence_frac * n_samples / span))
    ks = key(seed_base + stream_id, TID_AUDIO + 1)
    starts = (uniform(ks, np.arange(n_span, dtype=np.uint64)) * max(1, n_samples - span)).astype(np.int64)
    for s0 in starts:
        x[s0:s0 + span] = 0.0
    return x.astype(np.float32)
