"""Oracle: batched-style modified-ALSD RNN-T beam search (the `malsd_batch`
state machine), one utterance, fp32 scores.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module.  It shares no code with the CUDA library.

Source: "Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon":
  * §2.2 (one iteration): every active hypothesis takes the joint at its own
    frame, log-softmax, its top K labels, adds its score; blank is forced where
    the per-frame symbol limit fired; the global top K of the K*K candidates
    survive (pruning first), then identical survivors are recombined by
    log-sum-exp into the best-scoring one (the vacated slots are not refilled);
    the predictor advances on the selected labels and keeps the parent's
    state on blank; acoustic time advances only on blank.
  * §2.3: survivors are equal when transcript, last label and non-blank length
    match (compared here on the token sequences themselves, which §2.3 allows
    instead of a hash); the merged score is the log-sum-exp, kept in the slot
    that held the highest score.
  * §2.4: max_symbols (10 by default) forces blank; score normalisation
    changes the final ordering.
  * §2.5: the machine is driven by a prefix-aware scorer
    log_probs(time, prefix), so that it can be tested against a toy table.
  * §4.1 (state per slot: score, time index, last label, non-blank length,
    symbols at the current time, predictor state, history).

Readings where the pages are silent (each is listed in the design notes):
  * the beam starts as one hypothesis (slot 0, score 0, empty transcript, last
    label = blank) and K - 1 empty slots (score -inf);
  * a hypothesis whose time has reached T is final: it stays in the beam as a
    single "keep" candidate with its unchanged score, competing in every later
    pruning (so a final hypothesis can stay in slot 0 and win);
  * ties in every top-K choose the lower index (label, then candidate position
    parent * K + j);
  * a hypothesis at the symbol limit offers only its blank candidate;
  * a merged hypothesis keeps everything but the score from its best member,
    including the count of symbols at the current frame (alignments of one
    transcript at one frame may differ in it, so a binding limit can cut a
    path that the alignment sum would have counted);
  * the final choice maximises score / (non-blank length + 1) when score_norm,
    else the raw score (ties: lower slot);
  * scores are accumulated in fp32 (the pages fix fp32), log-sum-exp in fp32;
  * streaming (frames in chunks): an iteration that a running hypothesis
    cannot take because its frame has not arrived waits for the next push,
    and only the end of the utterance makes hypotheses final, so the chunked
    search runs the very iterations of the one-shot search.

Parity pins: tests/test_oracle_beam_pins.py (toy-table fixtures of §2.5,
beam 1 == the greedy decoder of oracle/decoder.py, and with a beam wide enough
never to prune and a symbol limit that never binds, every final score equals
the brute-force log-sum-exp over all alignments of its transcript; chunked
pushes equal the one-shot search).
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32
NEG = F32(-np.inf)


def logsumexp32(xs):
    xs = np.asarray(xs, dtype=F32)
    m = xs.max()
    if not np.isfinite(m):
        return m
    return F32(m + np.log(np.sum(np.exp(xs - m), dtype=F32)))


def topk_lowest_index(v, k):
    """Indices of the k largest values, ties to the lower index, best first."""
    v = np.asarray(v)
    order = sorted(range(len(v)), key=lambda i: (-float(v[i]), i))
    return order[:k]


class Hyp:
    __slots__ = ("score", "time", "last", "tokens", "sym_t", "state")

    def __init__(self, score, time, last, tokens, sym_t, state):
        self.score, self.time, self.last, self.tokens, self.sym_t, self.state = \
            score, time, last, tokens, sym_t, state


def initial_beam(scorer, beam, blank):
    """Slot 0: score 0, empty transcript, last label blank; K - 1 empty slots."""
    return [Hyp(F32(0.0), 0, blank, (), 0, scorer.init_state())] + [None] * (beam - 1)


def _cut_gap(values, k):
    """Gap between the k-th and (k+1)-th largest finite values (inf if none)."""
    v = np.sort(np.asarray([x for x in values if np.isfinite(x)], dtype=np.float64))[::-1]
    return float(v[k - 1] - v[k]) if v.size > k else float("inf")


def malsd_iteration(hyps, scorer, n_frames, blank, max_symbols, margins=None):
    """One alignment iteration over the beam `hyps` (K slots, None = empty):
    candidates, pruning to K, labels applied, recombination.  A hypothesis
    whose time has reached n_frames is final and offers one keep candidate.
    margins: a list that, when given, receives the gaps at every top-K cut
    and within every recombined group (diagnostics for comparisons with a
    differently rounded implementation; the search itself is unchanged)."""
    K = len(hyps)
    cands = []  # (score, parent slot, label or None for "keep"), in candidate-position order
    for k, h in enumerate(hyps):
        if h is None:
            cands += [(NEG, k, None)] * K
            continue
        if h.time >= n_frames:  # final: one keep candidate
            cands += [(h.score, k, None)] + [(NEG, k, None)] * (K - 1)
            continue
        lp = np.asarray(scorer.log_probs(h.time, h.state), dtype=F32)
        if h.sym_t >= max_symbols:  # forced blank
            cands += [(F32(h.score + lp[blank]), k, blank)] + [(NEG, k, None)] * (K - 1)
            continue
        for lab in topk_lowest_index(lp, K):
            cands.append((F32(h.score + lp[lab]), k, lab))
        cands += [(NEG, k, None)] * (K - min(K, len(lp)))  # fewer classes than K
        if margins is not None:
            margins.append(_cut_gap(lp, K))
    keep = topk_lowest_index([c[0] for c in cands], K)
    if margins is not None:
        margins.append(_cut_gap([c[0] for c in cands], K))
    new = []
    for pos in keep:
        s, k, lab = cands[pos]
        h = hyps[k]
        if not np.isfinite(s):
            new.append(None)
        elif lab is None:
            new.append(Hyp(s, h.time, h.last, h.tokens, h.sym_t, h.state))
        elif lab == blank:
            new.append(Hyp(s, h.time + 1, h.last, h.tokens, 0, h.state))
        else:
            new.append(Hyp(s, h.time, lab, h.tokens + (lab,), h.sym_t + 1, scorer.advance(h.state, lab)))
    # recombination of identical survivors (transcript, last label, length)
    groups = {}
    for i, h in enumerate(new):
        if h is not None:
            groups.setdefault((h.tokens, h.last, len(h.tokens)), []).append(i)
    for members in groups.values():
        if len(members) < 2:
            continue
        best = min(members, key=lambda i: (-float(new[i].score), i))
        if margins is not None:
            sc = sorted((float(new[i].score) for i in members), reverse=True)
            margins.append(sc[0] - sc[1])
        merged = logsumexp32([new[i].score for i in members])
        for i in members:
            if i != best:
                new[i] = None
        new[best].score = merged
    return new


def best_hypothesis(hyps, score_norm=True):
    """Slot of the winner: the highest score, or score / (length + 1) when
    score_norm; ties to the lower slot."""
    live = [i for i, h in enumerate(hyps) if h is not None]
    key = (lambda i: float(hyps[i].score) / (len(hyps[i].tokens) + 1)) if score_norm else \
        (lambda i: float(hyps[i].score))
    return min(live, key=lambda i: (-key(i), i))


def _finals(hyps):
    return [(h.tokens, h.score) if h is not None else None for h in hyps]


def malsd_beam(n_frames, scorer, beam, blank, max_symbols=10, score_norm=True):
    """Beam search over n_frames with a scorer providing
         init_state(), log_probs(time, state) -> [V+1] fp32 log-probabilities,
         advance(state, label) -> new state.
    Returns (best token tuple, final hypotheses as (tokens, score) per slot)."""
    hyps = initial_beam(scorer, beam, blank)
    for _ in range(n_frames * (max_symbols + 1) + 1):
        if not any(h is not None and h.time < n_frames for h in hyps):
            break
        hyps = malsd_iteration(hyps, scorer, n_frames, blank, max_symbols)
    return hyps[best_hypothesis(hyps, score_norm)].tokens, _finals(hyps)


class StreamingMalsd:
    """The same search over frames that arrive in chunks.  Iterations keep
    every hypothesis at one alignment length, so an iteration whose running
    hypotheses need a frame that has not arrived waits for the next push;
    flush() marks the utterance's end (hypotheses at the last frame become
    final) and finishes.  The result equals malsd_beam over all frames.
    The scorer is asked only for frames already pushed."""

    def __init__(self, scorer, beam, blank, max_symbols=10, score_norm=True, margins=None):
        self.scorer, self.blank, self.max_symbols, self.score_norm = scorer, blank, max_symbols, score_norm
        self.hyps = initial_beam(scorer, beam, blank)
        self.available = 0
        self.iterations = 0
        self.margins = margins

    def _run(self, n_frames):
        while any(h is not None and h.time < n_frames for h in self.hyps):
            if any(h is not None and self.available <= h.time < n_frames for h in self.hyps):
                break  # a running hypothesis needs a frame that has not arrived
            self.hyps = malsd_iteration(self.hyps, self.scorer, n_frames, self.blank, self.max_symbols,
                                        self.margins)
            self.iterations += 1

    def push(self, n_new):
        self.available += n_new
        self._run(n_frames=1 << 62)  # the end is unknown: nothing is final yet

    def flush(self):
        self._run(n_frames=self.available)
        return self.hyps[best_hypothesis(self.hyps, self.score_norm)].tokens, _finals(self.hyps)


class TableScorer:
    """§2.5's toy scorer: log-probabilities looked up by (time, prefix); the
    predictor state is the emitted prefix.  A missing key gives blank 0 and
    every label -inf (fp32)."""

    def __init__(self, table, n_classes, blank):
        self.table, self.C, self.blank = table, n_classes, blank

    def init_state(self):
        return ()

    def log_probs(self, t, prefix):
        if (t, prefix) in self.table:
            return np.asarray(self.table[(t, prefix)], dtype=F32)
        v = np.full(self.C, -np.inf, dtype=F32)
        v[self.blank] = 0.0
        return v

    def advance(self, prefix, label):
        return prefix + (label,)


def brute_force_transcripts(n_frames, scorer, blank, max_symbols):
    """Every alignment (labels and blanks, at most max_symbols labels per frame,
    blank forced at the limit, ending with the blank of frame T-1): the
    log-sum-exp of its path scores per transcript, in fp64."""
    out = {}

    def walk(t, state, tokens, sym, logp):
        if t == n_frames:
            prev = out.get(tokens)
            out[tokens] = logp if prev is None else float(np.logaddexp(prev, logp))
            return
        lp = np.asarray(scorer.log_probs(t, state), dtype=np.float64)
        if np.isfinite(lp[blank]):
            walk(t + 1, state, tokens, 0, logp + lp[blank])
        if sym < max_symbols:
            for lab in range(len(lp)):
                if lab != blank and np.isfinite(lp[lab]):
                    walk(t, scorer.advance(state, lab), tokens + (lab,), sym + 1, logp + lp[lab])

    walk(0, scorer.init_state(), (), 0, 0.0)
    return out


class PredictorScorer:
    """The LSTM predictor and joint of oracle/decoder.py as a beam scorer over
    projected frames z: log-softmax of the joint logits (fp32)."""

    def __init__(self, z, W, dcfg):
        from . import decoder as D
        self.D, self.z, self.W, self.dcfg = D, np.asarray(z, dtype=F32), W, dcfg

    def init_state(self):
        return self.D.DecoderState.fresh(self.W, self.dcfg)

    def log_probs(self, t, state):
        lg = self.D.joint_logits(self.z[t], state.p, self.W).astype(F32)
        m = lg.max()
        return (lg - m - np.log(np.sum(np.exp(lg - m), dtype=F32))).astype(F32)

    def advance(self, state, label):
        h, c = self.D.lstm_cell(self.W["emb"][label], state.h, state.c, self.W)
        return self.D.DecoderState(h, c, self.D.pred_project(h, self.W))
