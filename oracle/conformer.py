"""Oracle: a plain, slow, fp64 CPU statement of the cache-aware Conformer encoder.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module.  It shares no code with the CUDA library
and never imports it; inputs (weights, mel) arrive as plain arrays.

Sources ("the pages"):
  * "True streaming encode — implementation spec" (fluidaudio-web STREAMING.md):
    §Why this is provably correct (chunked-causal mask, chunk 2 / left 70, offline
    encode already emulates streaming), §State (14-frame mel tail, K/V caches of
    at most 70 rows taken after projection, conv cache = last 8 GLU outputs, subT),
    §Per-chunk flow steps 1-4 (subsample with causal pad only at stream start,
    FF1, xln -> K/V, rectangular rel-pos score with rel(i,j) = (Lc + i) - j on
    absolute positions, softmax, probs@V, pw1+GLU, causal depthwise over
    [convCache | glu_new], pw2, FF2, ln_out, cache update, joint projection),
    §Status (relShift trick offline; Nemotron right-context-3 provisional tail).
  * "Parakeet-EOU-120M — Streaming ASR Model", §Architecture / §Config (17 layers,
    hidden 512, attention context 70, explicit state passed in and out).
  * "Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon", §1.3
    (1501 mel frames -> 188 encoder frames, encoder-side 640-wide projection
    computed once per frame).

Readings where the pages are silent (each is listed in the design notes):
  * subsampling = three 1-D convolutions over time (kernel 3, stride 2, ReLU), mel
    bins as input channels, each output t reading inputs 2t-2 .. 2t, zero for
    negative time, then a D -> D linear;
  * the block is the standard macaron Conformer: pre-LayerNorm (eps 1e-5) on every
    module, half-weighted FF residuals with SiLU, GLU = first half * sigmoid(second
    half), depthwise conv followed by a per-channel affine (folded BatchNorm) and
    SiLU, every linear with a bias except the positional projection;
  * score scale 1/sqrt(head_dim) on the sum of the content and position terms;
  * sinusoidal encoding pe[r][2m] = sin(r * 10000^(-2m/D)), pe[r][2m+1] = cos(.),
    rel = query position - key position;
  * right-context variant: window mask p_k in [p_q - 70, p_q + right_context].

Parity pins: every function here is checked by tests/test_oracle_pins.py against
library routines (torch layer_norm / conv1d / glu / scaled-dot-product attention),
closed forms, the relShift cross-check and the streaming == offline invariant.
Readings that no page fixes (every function is still pinned above): the
subsampling form, block internals, score scale, positional encoding and the
synthetic initialisation; the pins show that this module states them
correctly, not that the pages' model used them.
"""
from __future__ import annotations

import math

import numpy as np

LN_EPS = 1e-5
MEL_TAIL = 14          # conv1 needs 2, conv2 2*2, conv3 4*2 input frames


# ---------------------------------------------------------------------------
# elementary pieces
# ---------------------------------------------------------------------------

def f64(a):
    return np.asarray(a, dtype=np.float64)


def weights_f64(W):
    """Widen every parameter to float64 once (bf16-representable values stay exact)."""
    return {k: f64(v) for k, v in W.items()}


def layer_norm(x, g, b):
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + LN_EPS) * g + b


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def silu(x):
    return x * sigmoid(x)


def linear(x, w, b=None):
    y = x @ w.T
    return y if b is None else y + b


def glu(a):
    d = a.shape[-1] // 2
    return a[..., :d] * sigmoid(a[..., d:])


# ---------------------------------------------------------------------------
# causal subsampling (8x): three stride-2, kernel-3 convolutions over time
# ---------------------------------------------------------------------------

def conv_stage(x, w, b, pad_left):
    """y[t] = ReLU(b + sum_k w[:, k, :] @ xp[2t + k]), xp = [pad_left zeros | x].

    With pad_left = 2 this is the causal stage (output t reads x[2t-2 .. 2t],
    zero before the start); with pad_left = 0 it is the valid convolution used
    on a continuation window [melTail | new mel].
    """
    C = x.shape[1]
    xp = np.concatenate([np.zeros((pad_left, C)), x], axis=0)
    t_out = (xp.shape[0] - 3) // 2 + 1
    if t_out <= 0:
        return np.zeros((0, w.shape[0]))
    cols = np.stack([np.concatenate([xp[2 * t], xp[2 * t + 1], xp[2 * t + 2]])
                     for t in range(t_out)])                         # [t_out, 3C]
    y = cols @ w.reshape(w.shape[0], 3 * C).T + b
    return np.maximum(y, 0.0)


def subsample(mel, W, pad_left):
    y = f64(mel)
    for s in (1, 2, 3):
        y = conv_stage(y, f64(W[f"sub.w{s}"]), f64(W[f"sub.b{s}"]), pad_left)
    return linear(y, f64(W["sub.wo"]), f64(W["sub.bo"]))


def subsampled_len(t_mel):
    t = t_mel
    for _ in range(3):
        t = (t + 2 - 3) // 2 + 1 if t > 0 else 0
    return t


# ---------------------------------------------------------------------------
# relative-position multi-head attention
# ---------------------------------------------------------------------------

def sinusoid(r, d):
    r = f64(r).reshape(-1, 1)
    inv = 10000.0 ** (-2.0 * np.arange(d // 2) / d)
    pe = np.zeros((r.shape[0], d))
    pe[:, 0::2] = np.sin(r * inv)
    pe[:, 1::2] = np.cos(r * inv)
    return pe


def chunk_mask(pq, pk, chunk, left):
    """Chunked-causal on absolute positions: key allowed iff it exists (p_k >= 0)
    and lies in [c - left, c + chunk - 1], c = floor(p_q / chunk) * chunk."""
    c = (pq // chunk) * chunk
    pk = pk[None, :]
    return (pk >= 0) & (pk >= c[:, None] - left) & (pk <= c[:, None] + chunk - 1)


def window_mask(pq, pk, left, right):
    pk = pk[None, :]
    return (pk >= 0) & (pk >= pq[:, None] - left) & (pk <= pq[:, None] + right)


def make_mask(cfg, pq, pk):
    if cfg.right_context > 0:
        return window_mask(pq, pk, cfg.att_left, cfg.right_context)
    return chunk_mask(pq, pk, cfg.att_chunk, cfg.att_left)


def softmax_rows(s, mask):
    s = np.where(mask, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.where(mask, np.exp(s - m), 0.0)
    return e / e.sum(axis=-1, keepdims=True)


def rel_pos_attention(q, k, v, pq, pk, wpos, pbu, pbv, n_heads, mask):
    """score[i,j] = ((q_i + u) . k_j + (q_i + v) . P[p_q(i) - p_k(j)]) / sqrt(HD),
    P[r] = pe(r) @ wpos^T split into heads, then masked softmax and probs @ V.

    The position term is gathered by direct rel indexing over the distinct rel
    values present."""
    nq, D = q.shape
    hd = D // n_heads
    rel = pq[:, None] - pk[None, :]
    rvals = np.arange(rel.min(), rel.max() + 1) if rel.size else np.arange(0)
    P = linear(sinusoid(rvals, D), wpos)                      # [n_rel, D]
    ridx = rel - (rvals[0] if rvals.size else 0)
    out = np.zeros((nq, D))
    for h in range(n_heads):
        sl = slice(h * hd, (h + 1) * hd)
        ac = (q[:, sl] + pbu[h]) @ k[:, sl].T                 # [nq, nk]
        bd_all = (q[:, sl] + pbv[h]) @ P[:, sl].T             # [nq, n_rel]
        bd = np.take_along_axis(bd_all, ridx, axis=1)
        s = (ac + bd) / math.sqrt(hd)
        out[:, sl] = softmax_rows(s, mask) @ v[:, sl]
    return out


def rel_shift(bd):
    """Transformer-XL shift of a [T, 2T-1] score whose column c holds rel (T-1) - c:
    left-pad one zero column, view as [2T, T], drop the first row, view as
    [T, 2T-1], keep the first T columns."""
    T = bd.shape[0]
    padded = np.concatenate([np.zeros((T, 1)), bd], axis=1)
    return padded.reshape(2 * T, T)[1:].reshape(T, 2 * T - 1)[:, :T]


def bd_term_rel_shift(qv, wpos_head_rows):
    """Offline square position term (q + v) . P[i - j] via the relShift trick.

    qv: [T, hd] (query + pos_bias_v of one head); wpos_head_rows: callable r -> P rows."""
    T = qv.shape[0]
    rvals = np.arange(T - 1, -T, -1)                          # T-1 .. -(T-1)
    return rel_shift(qv @ wpos_head_rows(rvals).T)


# ---------------------------------------------------------------------------
# Conformer layer with explicit caches
# ---------------------------------------------------------------------------

def feed_forward(x, W, p):
    h = silu(linear(layer_norm(x, W[p + "ln_g"], W[p + "ln_b"]), W[p + "w1"], W[p + "b1"]))
    return x + 0.5 * linear(h, W[p + "w2"], W[p + "b2"])


def conv_module(x, W, p, glu_prev):
    """pw1 + GLU -> glu_new; causal depthwise over [glu_prev | glu_new] (exactly
    len(glu_new) outputs); affine + SiLU; pw2 + residual.  Returns (x, glu_all)."""
    kk = W[p + "w_dw"].shape[1]
    g = glu(linear(layer_norm(x, W[p + "ln_g"], W[p + "ln_b"]), W[p + "w_pw1"], W[p + "b_pw1"]))
    full = np.concatenate([glu_prev, g], axis=0)
    n = g.shape[0]
    dw = np.zeros_like(g)
    for t in range(n):
        win = full[t: t + kk]                                  # glu_{t-8} .. glu_t
        dw[t] = W[p + "b_dw"] + (win * W[p + "w_dw"].T).sum(axis=0)
    y = silu(W[p + "bn_g"] * dw + W[p + "bn_b"])
    return x + linear(y, W[p + "w_pw2"], W[p + "b_pw2"]), full, (g, y)


def layer_step(x, W, l, cfg, k_prev, v_prev, glu_prev, pos0, trace=None):
    """One Conformer layer over n new frames at absolute positions pos0 .. pos0+n-1.

    k_prev / v_prev hold the projected keys / values of the Lc frames just before
    pos0 (oldest first); glu_prev the last dw_kernel-1 GLU outputs (zeros at the
    stream start).  Returns x and the full K, V, GLU sequences for cache update."""
    p = f"l{l}."
    Wl = {k[len(p):]: v for k, v in W.items() if k.startswith(p)}
    n = x.shape[0]
    x = feed_forward(x, Wl, "ff1.")
    if trace is not None:
        trace.setdefault("ff1", []).append(x.copy())
    xln = layer_norm(x, Wl["att.ln_g"], Wl["att.ln_b"])
    q = linear(xln, Wl["att.wq"], Wl["att.bq"])
    K = np.concatenate([k_prev, linear(xln, Wl["att.wk"], Wl["att.bk"])], axis=0)
    V = np.concatenate([v_prev, linear(xln, Wl["att.wv"], Wl["att.bv"])], axis=0)
    Lc = k_prev.shape[0]
    pq = pos0 + np.arange(n)
    pk = pos0 - Lc + np.arange(Lc + n)
    att = rel_pos_attention(q, K, V, pq, pk, Wl["att.wpos"], Wl["att.pbu"], Wl["att.pbv"],
                            cfg.n_heads, make_mask(cfg, pq, pk))
    x = x + linear(att, Wl["att.wo"], Wl["att.bo"])
    if trace is not None:
        trace.setdefault("att", []).append(att.copy())
        trace.setdefault("x_att", []).append(x.copy())
    x, glu_all, (g, y) = conv_module(x, Wl, "conv.", glu_prev)
    if trace is not None:
        trace.setdefault("glu", []).append(g.copy())
        trace.setdefault("conv", []).append(y.copy())
        trace.setdefault("x_conv", []).append(x.copy())
    x = feed_forward(x, Wl, "ff2.")
    x = layer_norm(x, Wl["out.ln_g"], Wl["out.ln_b"])
    if trace is not None:
        trace.setdefault("out", []).append(x.copy())
    return x, K, V, glu_all


def joint_projection(enc, W):
    return linear(enc, f64(W["joint.w"]), f64(W["joint.b"]))


# ---------------------------------------------------------------------------
# offline chunked-causal encode (brute-force T x T masked attention)
# ---------------------------------------------------------------------------

def encode_offline(mel, W, cfg, trace=None):
    """Full-sequence encode; frames at positions 0..T-1 attend through the mask."""
    D = cfg.d_model
    W = weights_f64(W)
    x = subsample(mel, W, pad_left=2)
    if trace is not None:
        trace["sub"] = x.copy()
    empty = np.zeros((0, D))
    for l in range(cfg.n_layers):
        x, _, _, _ = layer_step(x, W, l, cfg, empty, empty, np.zeros((cfg.dw_kernel - 1, D)), 0, trace)
    return x, joint_projection(x, W)


# ---------------------------------------------------------------------------
# cache-aware streaming (chunked-causal, exact)
# ---------------------------------------------------------------------------

class StreamingEncoder:
    """Per-stream state of the streaming encoder: subT, melTail, per-layer K/V
    caches (<= att_left rows, oldest first) and conv caches (dw_kernel-1 rows)."""

    def __init__(self, W, cfg):
        self.W, self.cfg = weights_f64(W), cfg
        self.reset()

    def reset(self):
        cfg = self.cfg
        D = cfg.d_model
        self.subT = 0
        self.mel_tail = np.zeros((0, cfg.mel_bins))
        self.k = [np.zeros((0, D)) for _ in range(cfg.n_layers)]
        self.v = [np.zeros((0, D)) for _ in range(cfg.n_layers)]
        self.conv = [np.zeros((cfg.dw_kernel - 1, D)) for _ in range(cfg.n_layers)]
        self.finished = False

    @property
    def Lc(self):
        return self.k[0].shape[0]

    def _subsample(self, mel):
        if self.subT == 0:
            x0 = subsample(mel, self.W, pad_left=2)          # causal pads at stream start only
            window = f64(mel)
        else:
            window = np.concatenate([self.mel_tail, f64(mel)], axis=0)
            x0 = subsample(window, self.W, pad_left=0)       # continuation: no left pad
        self.mel_tail = window[-MEL_TAIL:]
        return x0

    def _encode(self, x, trace=None):
        cfg = self.cfg
        for l in range(cfg.n_layers):
            x, K, V, glu_all = layer_step(x, self.W, l, cfg, self.k[l], self.v[l], self.conv[l],
                                          self.subT, trace)
            self.k[l] = K[-cfg.att_left:]
            self.v[l] = V[-cfg.att_left:]
            self.conv[l] = glu_all[-(cfg.dw_kernel - 1):]
        return x

    def push(self, mel, trace=None):
        """Push a multiple of att_chunk * 8 mel frames (160 ms for chunk 2)."""
        cfg = self.cfg
        assert not self.finished, "push after flush needs a reset"
        mel = f64(mel)
        assert mel.shape[0] % (8 * cfg.att_chunk) == 0 and mel.shape[0] > 0
        x = self._subsample(mel)
        if trace is not None:
            trace["sub"] = x.copy()
        x = self._encode(x, trace)
        self.subT += x.shape[0]
        return x, joint_projection(x, self.W)

    def flush(self, mel, trace=None):
        """Final partial chunk: any number of mel frames; ceil(r / 8) new frames."""
        mel = f64(mel)
        self.finished = True
        if mel.shape[0] == 0:
            D = self.cfg.d_model
            return np.zeros((0, D)), np.zeros((0, self.cfg.joint_dim))
        x = self._subsample(mel)
        x = self._encode(x, trace)
        self.subT += x.shape[0]
        return x, joint_projection(x, self.W)


# ---------------------------------------------------------------------------
# right-context provisional tail (Nemotron variant)
# ---------------------------------------------------------------------------

class ProvisionalTailEncoder:
    """Each pass computes emit + lookahead frames, emits `emit`, commits K/V and
    the conv tail of the emitted frames only, and recomputes the tail next pass.

    The subsampled (layer-0) inputs of not-yet-emitted frames are exact because
    subsampling is causal; they wait in x0 until emitted."""

    def __init__(self, W, cfg):
        self.W, self.cfg = weights_f64(W), cfg
        self.reset()

    def reset(self):
        cfg = self.cfg
        D = cfg.d_model
        self.sub = StreamingEncoder(self.W, cfg)   # only its subsampling state is used
        self.emitted = 0
        self.x0 = np.zeros((0, D))
        self.k = [np.zeros((0, D)) for _ in range(cfg.n_layers)]
        self.v = [np.zeros((0, D)) for _ in range(cfg.n_layers)]
        self.conv = [np.zeros((cfg.dw_kernel - 1, D)) for _ in range(cfg.n_layers)]
        self.finished = False

    def _pass(self, n_frames, n_emit):
        cfg = self.cfg
        x = self.x0[:n_frames]
        for l in range(cfg.n_layers):
            x, K, V, glu_all = layer_step(x, self.W, l, cfg, self.k[l], self.v[l], self.conv[l],
                                          self.emitted)
            Lc = self.k[l].shape[0]
            self.k[l] = K[: Lc + n_emit][-cfg.att_left:]
            self.v[l] = V[: Lc + n_emit][-cfg.att_left:]
            kk = cfg.dw_kernel - 1
            self.conv[l] = glu_all[: kk + n_emit][-kk:]
        out = x[:n_emit]
        self.x0 = self.x0[n_emit:]
        self.emitted += n_emit
        return out

    def _drain(self, final):
        cfg = self.cfg
        outs = []
        need = cfg.emit_frames + cfg.lookahead_frames
        while self.x0.shape[0] >= need or (final and self.x0.shape[0] > 0):
            n = min(need, self.x0.shape[0])
            outs.append(self._pass(n, min(cfg.emit_frames, n)))
        x = np.concatenate(outs, axis=0) if outs else np.zeros((0, cfg.d_model))
        return x, joint_projection(x, self.W)

    def push(self, mel):
        assert not self.finished
        mel = f64(mel)
        assert mel.shape[0] % (8 * self.cfg.att_chunk) == 0 and mel.shape[0] > 0
        self.x0 = np.concatenate([self.x0, self.sub._subsample(mel)], axis=0)
        self.sub.subT += mel.shape[0] // 8
        return self._drain(final=False)

    def flush(self, mel):
        mel = f64(mel)
        self.finished = True
        if mel.shape[0]:
            x0 = self.sub._subsample(mel)
            self.sub.subT += x0.shape[0]
            self.x0 = np.concatenate([self.x0, x0], axis=0)
        return self._drain(final=True)
