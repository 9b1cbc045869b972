"""Pins of the greedy RNN-T decoder oracle (oracle/decoder.py) to things other
than itself: torch's LSTM cell and linear layer, closed forms, hand-built
prefix-aware toy scorers ("Fast Accuracy-Preserving RNNT Beam Search on Apple
Silicon", §2.5) and the state-carry invariant of "True streaming encode —
implementation spec", §Decoder state carry."""
import math
from dataclasses import replace

import numpy as np
import pytest

from cache_aware_conformer_gb300 import synth
from cache_aware_conformer_gb300.config import TINY_DECODER
from oracle import decoder as O

torch = pytest.importorskip("torch")


def _weights(dc=TINY_DECODER, seed=0):
    return synth.make_decoder_weights(dc, seed)


def test_lstm_cell_matches_torch_lstmcell():
    dc = TINY_DECODER
    W = _weights(dc)
    P = dc.pred_dim
    cell = torch.nn.LSTMCell(P, P)
    with torch.no_grad():
        cell.weight_ih.copy_(torch.from_numpy(W["lstm.w_ih"]))
        cell.weight_hh.copy_(torch.from_numpy(W["lstm.w_hh"]))
        cell.bias_ih.copy_(torch.from_numpy(W["lstm.b_ih"]))
        cell.bias_hh.copy_(torch.from_numpy(W["lstm.b_hh"]))
    rng = np.random.default_rng(5)
    x = rng.standard_normal(P).astype(np.float32)
    h = (0.5 * rng.standard_normal(P)).astype(np.float32)
    c = rng.standard_normal(P).astype(np.float32)
    h2, c2 = O.lstm_cell(x, h, c, W)
    with torch.no_grad():
        th, tc = cell(torch.from_numpy(x)[None], (torch.from_numpy(h)[None], torch.from_numpy(c)[None]))
    np.testing.assert_allclose(h2, th[0].numpy(), rtol=0, atol=2e-6)
    np.testing.assert_allclose(c2, tc[0].numpy(), rtol=0, atol=2e-6)


class TorchScorer:
    """The predictor + joint as torch modules in fp64: embedding, LSTM cell,
    predictor projection, ReLU joint, primed by one step on the blank token from
    zero state; the oracle's greedy loop drives it."""

    def __init__(self, z, W, dc):
        P, J, C = dc.pred_dim, dc.joint_dim, W["out.w"].shape[0]
        t = {k: torch.from_numpy(np.asarray(v, np.float64)) for k, v in W.items()}
        self.emb = torch.nn.Embedding.from_pretrained(t["emb"])
        self.cell = torch.nn.LSTMCell(P, P, dtype=torch.float64)
        self.pred = torch.nn.Linear(P, J, dtype=torch.float64)
        self.out = torch.nn.Linear(J, C, dtype=torch.float64)
        with torch.no_grad():
            for mod, pairs in ((self.cell, (("weight_ih", "lstm.w_ih"), ("weight_hh", "lstm.w_hh"),
                                            ("bias_ih", "lstm.b_ih"), ("bias_hh", "lstm.b_hh"))),
                               (self.pred, (("weight", "pred.w"), ("bias", "pred.b"))),
                               (self.out, (("weight", "out.w"), ("bias", "out.b")))):
                for attr, name in pairs:
                    getattr(mod, attr).copy_(t[name])
        self.z = torch.from_numpy(np.asarray(z, np.float64))
        zero = torch.zeros(1, P, dtype=torch.float64)
        self.hc = (zero, zero)
        self.advance(dc.blank)

    @torch.no_grad()
    def logits(self, t):
        return self.out(torch.relu(self.z[t] + self.p[0])).numpy()

    @torch.no_grad()
    def advance(self, k):
        self.hc = self.cell(self.emb(torch.tensor([k])), self.hc)
        self.p = self.pred(self.hc[0])


def test_predictor_and_joint_match_torch_modules():
    """The oracle's scorer (primed state, token embedding, LSTM step, predictor
    projection, joint) decides like the same network built from torch modules
    in fp64, emission for emission, and ends in the same LSTM state."""
    dc = replace(TINY_DECODER, blank_bias=2.0)  # a few dozen emissions over 24 frames
    W = _weights(dc, seed=4)
    z = synth.make_joint_frames(24, 7, dc.joint_dim)
    em, st = O.decode_chunk(z, O.DecoderState.fresh(W, dc), W, dc)
    ref = TorchScorer(z, W, dc)
    em_ref = O.greedy_rnnt(24, ref, dc.blank, dc.max_symbols)
    assert len(em) > 20 and len({k for _, k in em}) > 2 and em == em_ref
    np.testing.assert_allclose(st.h, ref.hc[0][0].numpy(), rtol=0, atol=1e-5)
    np.testing.assert_allclose(st.c, ref.hc[1][0].numpy(), rtol=0, atol=1e-5)


def test_lstm_cell_closed_form_with_zero_weights():
    """With zero matrices the gates are the biases: c' = s(b_f) c + s(b_i) tanh(b_g),
    h' = s(b_o) tanh(c'), s the logistic function (written out in float64 here)."""
    P = 4
    W = {"lstm.w_ih": np.zeros((4 * P, P), np.float32), "lstm.w_hh": np.zeros((4 * P, P), np.float32),
         "lstm.b_ih": np.array([0.3, -1, 2, 0, 0.5, 1.5, -2, 0, 1, -0.7, 0.2, 3, -1, 0.1, 0.4, 2], np.float32),
         "lstm.b_hh": np.zeros(4 * P, np.float32)}
    c = np.array([1.0, -2.0, 0.5, 0.0], np.float32)
    h2, c2 = O.lstm_cell(np.ones(P, np.float32), np.ones(P, np.float32), c, W)
    s = lambda v: 1.0 / (1.0 + math.exp(-v))
    b = W["lstm.b_ih"].astype(np.float64)
    for j in range(P):
        cj = s(b[P + j]) * c[j] + s(b[j]) * math.tanh(b[2 * P + j])
        hj = s(b[3 * P + j]) * math.tanh(cj)
        assert abs(c2[j] - cj) < 1e-6 and abs(h2[j] - hj) < 1e-6


def test_joint_matches_torch_linear_relu():
    dc = TINY_DECODER
    W = _weights(dc)
    rng = np.random.default_rng(2)
    z = rng.standard_normal(dc.joint_dim).astype(np.float32)
    p = rng.standard_normal(dc.joint_dim).astype(np.float32)
    ref = torch.nn.functional.linear(torch.relu(torch.from_numpy(z + p)), torch.from_numpy(W["out.w"]),
                                     torch.from_numpy(W["out.b"])).numpy()
    np.testing.assert_allclose(O.joint_logits(z, p, W), ref, rtol=0, atol=2e-6)
    # the predictor projection is a plain linear layer too
    h = rng.standard_normal(dc.pred_dim).astype(np.float32)
    ref = torch.nn.functional.linear(torch.from_numpy(h), torch.from_numpy(W["pred.w"]),
                                     torch.from_numpy(W["pred.b"])).numpy()
    np.testing.assert_allclose(O.pred_project(h, W), ref, rtol=0, atol=2e-6)


class ToyScorer:
    """Logits looked up by (frame, emitted prefix); classes 0, 1, 2 = tokens,
    3 = blank, 4 = EOU.  A missing key scores blank highest."""

    def __init__(self, table, classes=5, blank=3):
        self.table, self.prefix, self.C, self.blank = table, (), classes, blank

    def logits(self, t):
        if (t, self.prefix) in self.table:
            return np.asarray(self.table[(t, self.prefix)], np.float32)
        v = np.zeros(self.C, np.float32)
        v[self.blank] = 1.0
        return v

    def advance(self, k):
        self.prefix = self.prefix + (k,)


def test_toy_all_blank():
    assert O.greedy_rnnt(5, ToyScorer({}), blank=3, max_symbols=4) == []


def test_toy_tie_goes_to_lowest_index():
    # frame 0: token 1 and blank tie at the top -> token 1 (lower index) is emitted
    table = {(0, ()): [0, 2, 0, 2, 0]}
    assert O.greedy_rnnt(2, ToyScorer(table), blank=3, max_symbols=4) == [(0, 1)]
    # token 2 and EOU tie below a blank: blank wins, nothing is emitted
    table = {(0, ()): [0, 0, 1, 1.5, 1]}
    assert O.greedy_rnnt(1, ToyScorer(table), blank=3, max_symbols=4) == []


def test_toy_max_symbols_forces_the_next_frame():
    class Always2(ToyScorer):
        def logits(self, t):
            return np.array([0, 0, 5, 1, 0], np.float32)
    out = O.greedy_rnnt(3, Always2({}), blank=3, max_symbols=4)
    assert out == [(t, 2) for t in range(3) for _ in range(4)]


def test_toy_prefix_dependent_with_eou():
    """The logits depend on the emitted prefix; EOU (4) is emitted and the
    prefix advances on it, so the next lookup sees it."""
    table = {(0, ()): [3, 0, 0, 1, 0],
             (0, (0,)): [0, 0, 3, 1, 0],
             (0, (0, 2)): [0, 0, 0, 1, 0],
             (1, (0, 2)): [0, 0, 0, 1, 2],
             (1, (0, 2, 4)): [0, 2, 0, 1, 0],
             (1, (0, 2, 4, 1)): [0, 0, 0, 1, 0]}
    out = O.greedy_rnnt(3, ToyScorer(table), blank=3, max_symbols=5)
    assert out == [(0, 0), (0, 2), (1, 4), (1, 1)]


def test_state_carry_chunked_equals_one_call():
    """Decoding 24 frames in one call equals decoding them 2 at a time with the
    predictor state carried between calls."""
    dc = TINY_DECODER
    W = _weights(dc)
    z = synth.make_joint_frames(24, 3, dc.joint_dim)
    em_all, s_all = O.decode_chunk(z, O.DecoderState.fresh(W, dc), W, dc)
    st = O.DecoderState.fresh(W, dc)
    em = []
    for t0 in range(0, 24, 2):
        e, st = O.decode_chunk(z[t0:t0 + 2], st, W, dc)
        em += [(t0 + t, k) for t, k in e]
    assert em == em_all and len(em_all) > 0
    np.testing.assert_array_equal(st.h, s_all.h)
    np.testing.assert_array_equal(st.c, s_all.c)


def test_fresh_state_and_all_blank_decode():
    """A blank that always wins leaves the primed state untouched; the primed
    state is one LSTM step on the blank embedding from zeros."""
    dc = replace(TINY_DECODER, blank_bias=1e4)
    W = _weights(dc)
    st = O.DecoderState.fresh(W, dc)
    h, c = O.lstm_cell(W["emb"][dc.blank], np.zeros(dc.pred_dim, np.float32), np.zeros(dc.pred_dim, np.float32), W)
    np.testing.assert_array_equal(st.h, h)
    em, st2 = O.decode_chunk(synth.make_joint_frames(10, 0, dc.joint_dim), st, W, dc)
    assert em == []
    np.testing.assert_array_equal(st2.p, st.p)


def test_blank_never_wins_gives_max_symbols_per_frame():
    dc = replace(TINY_DECODER, blank_bias=-1e4)
    W = _weights(dc)
    em, _ = O.decode_chunk(synth.make_joint_frames(4, 1, dc.joint_dim), O.DecoderState.fresh(W, dc), W, dc)
    assert [t for t, _ in em] == [t for t in range(4) for _ in range(dc.max_symbols)]
    assert all(k != dc.blank for _, k in em)
