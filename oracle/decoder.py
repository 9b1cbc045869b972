"""Oracle: greedy RNN-T decoding with an end-of-utterance class, fp32 on the CPU.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module.  It shares no code with the CUDA library
and never imports it; weights and projected encoder frames arrive as arrays.

Sources ("the pages"):
  * "Parakeet-EOU-120M — Streaming ASR Model", §Architecture: the decoder is a
    single-step fp32 LSTM that consumes the previous non-blank token and returns
    a decoder output plus new (h, c); the joint fuses one encoder frame with the
    decoder output into logits over vocabulary + blank + EOU; greedy decoding
    loops per encoder frame and advances the decoder only on non-blank
    emissions.  §Vocabulary: blank and EOU are the two classes after the
    vocabulary.
  * "True streaming encode — implementation spec", §Decoder state carry: the
    loop continues across calls with the predictor state kept (no reset, no
    re-prediction from blank); a separate reset starts a stream, from blank.
  * "Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon", §2.5 (test
    the decision loop against a prefix-aware toy scorer, not a fixed logit
    table) and §3 (the encoder frame is projected once, the predictor output
    once per prefix; the joint is add -> ReLU -> final linear).

Readings where the pages are silent (each is listed in the design notes):
  * predictor = embedding row of the last emitted token -> one LSTM layer
    (gate rows input, forget, cell, output; bias b_ih + b_hh) -> its h, then the
    640-wide predictor projection; at stream start h = c = 0 and the predictor
    runs once on the blank token;
  * EOU is a non-blank emission: it is output and the predictor advances on it;
  * argmax ties go to the lowest class index; after max_symbols emissions on
    one frame the loop moves to the next frame (a forced blank);
  * every operation is fp32 (the pages fix fp32 for the decoder), so both this
    oracle and the GPU take each argmax in fp32.

Parity pins: tests/test_oracle_decoder_pins.py checks the LSTM step against
torch.nn.LSTMCell and a closed form, the decision loop against hand-built toy
scorers, and the state-carry invariant (chunked decode == one-call decode).
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def sigmoid(x):
    x = np.asarray(x, dtype=F32)
    return (F32(1.0) / (F32(1.0) + np.exp(-x))).astype(F32)


def lstm_cell(x, h, c, W):
    """One LSTM step: gates = W_ih x + b_ih + W_hh h + b_hh, rows [i | f | g | o];
    c' = sigmoid(f) c + sigmoid(i) tanh(g); h' = sigmoid(o) tanh(c')."""
    P = h.shape[0]
    gates = (W["lstm.w_ih"] @ x + W["lstm.b_ih"] + W["lstm.w_hh"] @ h + W["lstm.b_hh"]).astype(F32)
    i, f, g, o = gates[:P], gates[P:2 * P], gates[2 * P:3 * P], gates[3 * P:]
    c2 = (sigmoid(f) * c + sigmoid(i) * np.tanh(g)).astype(F32)
    h2 = (sigmoid(o) * np.tanh(c2)).astype(F32)
    return h2, c2


def pred_project(h, W):
    """Predictor projection into the joint: W_pred h + b_pred."""
    return (W["pred.w"] @ h + W["pred.b"]).astype(F32)


def joint_logits(z_t, p, W):
    """Joint after both projections: W_out ReLU(z_t + p) + b_out."""
    a = np.maximum(np.asarray(z_t, dtype=F32) + p, F32(0.0)).astype(F32)
    return (W["out.w"] @ a + W["out.b"]).astype(F32)


def greedy_rnnt(n_frames, scorer, blank: int, max_symbols: int):
    """The greedy decision loop: per frame, take the argmax (lowest index on
    ties); blank moves to the next frame, anything else is emitted and the
    scorer advances on it; after max_symbols emissions the frame ends.
    Returns the emissions as (frame, class) pairs in order."""
    out = []
    for t in range(n_frames):
        for _ in range(max_symbols):
            k = int(np.argmax(scorer.logits(t)))
            if k == blank:
                break
            out.append((t, k))
            scorer.advance(k)
    return out


class DecoderState:
    """Per-stream predictor state carried across calls: LSTM (h, c) and the
    predictor projection p of h."""

    def __init__(self, h, c, p):
        self.h, self.c, self.p = h, c, p

    @classmethod
    def fresh(cls, W, dcfg):
        """Stream start: zero (h, c), then one predictor step on the blank token."""
        P = dcfg.pred_dim
        h, c = lstm_cell(W["emb"][dcfg.blank], np.zeros(P, F32), np.zeros(P, F32), W)
        return cls(h, c, pred_project(h, W))

    def copy(self):
        return DecoderState(self.h.copy(), self.c.copy(), self.p.copy())


class PredictorScorer:
    """Joint logits of the projected encoder frames z against the predictor
    state; advance(k) runs the predictor on token k."""

    def __init__(self, z, state: DecoderState, W):
        self.z, self.s, self.W = np.asarray(z, dtype=F32), state, W

    def logits(self, t):
        return joint_logits(self.z[t], self.s.p, self.W)

    def advance(self, k):
        h, c = lstm_cell(self.W["emb"][k], self.s.h, self.s.c, self.W)
        self.s = DecoderState(h, c, pred_project(h, self.W))


def decode_chunk(z, state: DecoderState, W, dcfg):
    """Greedy decode of the frames z [T, joint_dim] from `state`; returns the
    emissions [(frame, class)] and the state after the last frame."""
    sc = PredictorScorer(z, state.copy(), W)
    em = greedy_rnnt(len(sc.z), sc, dcfg.blank, dcfg.max_symbols)
    return em, sc.s


def decision_margins(z, state: DecoderState, W, dcfg):
    """The same loop, recording per decision (frame, class, top-1 minus top-2
    logit): where the margin is within fp32 rounding, another correct fp32
    evaluation order may take the other class."""
    sc = PredictorScorer(z, state.copy(), W)
    rec = []
    for t in range(len(sc.z)):
        for _ in range(dcfg.max_symbols):
            lg = sc.logits(t)
            k = int(np.argmax(lg))
            srt = np.sort(lg)
            rec.append((t, k, float(srt[-1] - srt[-2])))
            if k == dcfg.blank:
                break
            sc.advance(k)
    return rec
