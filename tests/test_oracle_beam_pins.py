"""Pins of the MALSD beam-search oracle (oracle/beam.py): the toy-scorer
fixtures "Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon" §2.5
asks for, beam 1 against the independently written greedy decoder, and the
unpruned beam against brute-force sums over all alignments."""
import math

import numpy as np
import pytest

from cache_aware_conformer_gb300 import synth
from cache_aware_conformer_gb300.config import EOU_DECODER, TINY_DECODER
from oracle import beam as B
from oracle import decoder as D

NEG = -np.inf
BLANK = 2  # toy vocabulary: tokens 0 and 1, blank 2


def _lp(p0, p1, pb):
    """log-probabilities from probabilities (fp32); a zero gives -inf"""
    with np.errstate(divide="ignore"):
        return np.log(np.array([p0, p1, pb], dtype=np.float64)).astype(np.float32)


def test_blank_versus_label_tie_goes_to_the_lower_index():
    # frame 0: token 1 and blank tie at the top; beam 1 keeps the lower index (token 1)
    table = {(0, ()): _lp(0.2, 0.4, 0.4)}
    best, _ = B.malsd_beam(1, B.TableScorer(table, 3, BLANK), beam=1, blank=BLANK, max_symbols=3)
    assert best == (1,)


def test_two_alignments_of_one_transcript_are_recombined():
    """T = 2: 'a' emitted at frame 0 or at frame 1 gives the same transcript;
    the surviving hypothesis carries the log-sum-exp of both paths."""
    table = {(0, ()): _lp(0.5, 0.0, 0.5), (0, (0,)): _lp(0.0, 0.0, 1.0),
             (1, ()): _lp(0.5, 0.0, 0.5), (1, (0,)): _lp(0.0, 0.0, 1.0)}
    sc = B.TableScorer(table, 3, BLANK)
    best, finals = B.malsd_beam(2, sc, beam=4, blank=BLANK, max_symbols=3, score_norm=False)
    got = {tok: float(s) for f in finals if f is not None for tok, s in [f]}
    # paths: a@0 then blanks: .5*1*1 ; blank, a@1, blank: .5*.5*1 ; blank, blank: .5*.5
    assert abs(got[(0,)] - math.log(0.5 + 0.25)) < 1e-6
    assert abs(got[()] - math.log(0.25)) < 1e-6
    assert best == (0,)


def test_pruning_happens_before_recombination():
    """Three candidates for two slots: the two alignments of 'a' are pruned to
    one (the beam keeps 'a'-path-1 and 'b'); recombining first would have merged
    both 'a' paths into one slot and kept a third hypothesis."""
    table = {(0, ()): _lp(0.40, 0.35, 0.25),
             (0, (0,)): _lp(0.0, 0.0, 1.0), (0, (1,)): _lp(0.0, 0.0, 1.0),
             (1, ()): _lp(0.30, 0.0, 0.70), (1, (0,)): _lp(0.0, 0.0, 1.0), (1, (1,)): _lp(0.0, 0.0, 1.0)}
    sc = B.TableScorer(table, 3, BLANK)
    _, finals = B.malsd_beam(2, sc, beam=2, blank=BLANK, max_symbols=3, score_norm=False)
    got = {tok: float(s) for f in finals if f is not None for tok, s in [f]}
    # iteration 1 candidates: a(.40), b(.35), blank(.25) -> keep a, b; the blank path (and its later
    # 'a' at frame 1) is gone, so 'a' carries only its first alignment
    assert set(got) == {(0,), (1,)}
    assert abs(got[(0,)] - math.log(0.40)) < 1e-6 and abs(got[(1,)] - math.log(0.35)) < 1e-6


def test_max_symbols_forces_blank():
    table = {(t, (0,) * u): _lp(0.9, 0.05, 0.05) for t in range(2) for u in range(8)}
    best, _ = B.malsd_beam(2, B.TableScorer(table, 3, BLANK), beam=1, blank=BLANK, max_symbols=2)
    assert best == (0, 0, 0, 0)  # two per frame, then the forced blank


def test_final_hypothesis_kept_in_the_beam():
    """A hypothesis that reaches the last frame early stays as a candidate and
    wins over the ones still running."""
    table = {(0, ()): _lp(0.3, 0.0, 0.7), (0, (0,)): _lp(0.0, 0.0, 1.0),
             (1, ()): _lp(0.0, 0.0, 1.0), (1, (0,)): _lp(0.0, 0.99, 0.01),
             (1, (0, 1)): _lp(0.0, 0.0, 1.0)}
    sc = B.TableScorer(table, 3, BLANK)
    best, finals = B.malsd_beam(2, sc, beam=2, blank=BLANK, max_symbols=3, score_norm=False)
    assert best == ()                     # log 0.7 beats log(0.3 * 0.99)
    assert finals[0][0] == ()             # and it holds slot 0


def test_score_normalisation_changes_the_winner():
    table = {(0, ()): _lp(0.45, 0.0, 0.55), (0, (0,)): _lp(0.0, 0.9, 0.1),
             (0, (0, 1)): _lp(0.0, 0.0, 1.0)}
    sc = B.TableScorer(table, 3, BLANK)
    raw, _ = B.malsd_beam(1, sc, beam=3, blank=BLANK, max_symbols=3, score_norm=False)
    norm, _ = B.malsd_beam(1, sc, beam=3, blank=BLANK, max_symbols=3, score_norm=True)
    # () : log .55 = -0.598 ; (0,1): log(.45*.9) = -0.904, / 3 = -0.301 > -0.598
    assert raw == () and norm == (0, 1)


@pytest.mark.parametrize("dc,n", [(TINY_DECODER, 16), (EOU_DECODER, 6)])
def test_beam_one_is_the_greedy_decoder(dc, n):
    """Beam 1 takes the argmax of the log-softmax at every step: the greedy
    loop of oracle/decoder.py on the same predictor and frames."""
    W = synth.make_decoder_weights(dc, 0)
    for s in range(4 if dc is TINY_DECODER else 2):
        z = synth.make_joint_frames(n, s, dc.joint_dim)
        em, _ = D.decode_chunk(z, D.DecoderState.fresh(W, dc), W, dc)
        best, _ = B.malsd_beam(n, B.PredictorScorer(z, W, dc), beam=1, blank=dc.blank,
                               max_symbols=dc.max_symbols)
        assert best == tuple(k for _, k in em)


def test_unpruned_beam_sums_every_alignment():
    """With a beam wide enough that nothing is pruned, and a symbol limit that
    never binds (the table gives labels only to prefixes of up to 3 tokens, the
    limit is 4), each final hypothesis holds the log-sum-exp over all
    alignments of its transcript."""
    rng = np.random.default_rng(4)
    T = 2
    table = {}
    for t in range(T):
        for u in range(4):
            for code in range(2 ** u):
                table[(t, tuple((code >> i) & 1 for i in range(u)))] = \
                    np.log(rng.dirichlet([1.0, 1.0, 1.5])).astype(np.float32)
    sc = B.TableScorer(table, 3, BLANK)
    ref = B.brute_force_transcripts(T, sc, BLANK, 4)
    assert len(ref) == 31                                    # every transcript of up to 4 tokens over {0, 1}
    _, finals = B.malsd_beam(T, sc, beam=64, blank=BLANK, max_symbols=4, score_norm=False)
    got = {tok: float(s) for f in finals if f is not None for tok, s in [f]}
    assert set(got) == set(ref)
    for tok, s in ref.items():
        assert abs(got[tok] - s) < 1e-5, (tok, got[tok], s)


def test_merged_hypothesis_keeps_the_symbol_count_of_the_best_member():
    """Two alignments of 'aa' reach frame 1 together: 'a a | ' (no symbol yet at
    frame 1) and 'a | a' (one symbol at frame 1, the likelier).  The merged
    hypothesis takes the second one's count, so with max_symbols 2 only one more
    'a' fits at frame 1 and 'aaaa' (reachable through the first alignment) is
    gone; every other transcript still carries its full alignment sum."""
    table = {(0, ()): _lp(0.6, 0.0, 0.4), (0, (0,)): _lp(0.2, 0.0, 0.8), (0, (0, 0)): _lp(0.0, 0.0, 1.0),
             (1, ()): _lp(0.0, 0.0, 1.0), (1, (0,)): _lp(0.5, 0.0, 0.5), (1, (0, 0)): _lp(0.5, 0.0, 0.5),
             (1, (0, 0, 0)): _lp(0.5, 0.0, 0.5), (1, (0, 0, 0, 0)): _lp(0.0, 0.0, 1.0)}
    sc = B.TableScorer(table, 3, BLANK)
    ref = B.brute_force_transcripts(2, sc, BLANK, 2)
    _, finals = B.malsd_beam(2, sc, beam=8, blank=BLANK, max_symbols=2, score_norm=False)
    got = {tok: float(s) for f in finals if f is not None for tok, s in [f]}
    assert abs(ref[(0, 0, 0, 0)] - math.log(0.6 * 0.2 * 0.5 * 0.5)) < 1e-6  # fp32 table entries
    assert set(ref) - set(got) == {(0, 0, 0, 0)}
    for tok in got:
        assert abs(got[tok] - ref[tok]) < 1e-6, tok
    assert abs(got[(0, 0)] - math.log(0.6 * 0.2 * 0.5 + 0.6 * 0.8 * 0.5 * 0.5)) < 1e-6


def test_equal_last_label_and_length_alone_do_not_merge():
    """The collision case of a transcript hash: 'ab' and 'bb' share the last
    label and the length, and reach the same frame in the same iteration; only
    equal token sequences merge, so both survive with their own scores."""
    table = {(0, ()): _lp(0.3, 0.3, 0.4), (0, (0,)): _lp(0.0, 0.5, 0.5), (0, (1,)): _lp(0.0, 0.5, 0.5),
             (0, (0, 1)): _lp(0.0, 0.0, 1.0), (0, (1, 1)): _lp(0.0, 0.0, 1.0)}
    sc = B.TableScorer(table, 3, BLANK)
    _, finals = B.malsd_beam(1, sc, beam=8, blank=BLANK, max_symbols=3, score_norm=False)
    got = {tok: float(s) for f in finals if f is not None for tok, s in [f]}
    assert set(got) == {(), (0,), (1,), (0, 1), (1, 1)}
    assert abs(got[(0, 1)] - math.log(0.15)) < 1e-6 and abs(got[(1, 1)] - math.log(0.15)) < 1e-6


@pytest.mark.parametrize("chunks", [[16], [2] * 8, [1, 0, 3, 5, 0, 7], [0, 16]])
def test_streamed_beam_equals_the_whole_utterance(chunks):
    """Frames pushed in chunks (iterations wait while a running hypothesis
    needs a frame not yet pushed) give the same beam as all frames at once."""
    dc = TINY_DECODER
    W = synth.make_decoder_weights(dc, 0)
    for s in range(3):
        z = synth.make_joint_frames(16, 10 + s, dc.joint_dim)
        best, finals = B.malsd_beam(16, B.PredictorScorer(z, W, dc), beam=4, blank=dc.blank,
                                    max_symbols=dc.max_symbols)
        st = B.StreamingMalsd(B.PredictorScorer(z, W, dc), beam=4, blank=dc.blank, max_symbols=dc.max_symbols)
        for n in chunks:
            st.push(n)
        got_best, got_finals = st.flush()
        assert got_best == best
        assert [f and (f[0], float(f[1])) for f in got_finals] == [f and (f[0], float(f[1])) for f in finals]


def test_logsumexp_and_log_softmax_match_library_routines():
    """The fp32 log-sum-exp used by recombination against numpy's logaddexp
    (with -inf members and an all -inf set), and the scorer's log-softmax
    against torch.log_softmax of the same joint logits."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    for xs in (rng.normal(size=7) * 5, np.array([0.3, NEG, -2.0, NEG]), np.array([80.0, 79.5, -300.0])):
        ref = np.logaddexp.reduce(xs.astype(np.float32).astype(np.float64))
        assert abs(float(B.logsumexp32(xs)) - ref) < 1e-5 * max(1.0, abs(ref))
    assert B.logsumexp32([NEG, NEG]) == NEG
    dc = TINY_DECODER
    W = synth.make_decoder_weights(dc, 2)
    z = synth.make_joint_frames(3, 5, dc.joint_dim)
    sc = B.PredictorScorer(z, W, dc)
    st = sc.advance(sc.init_state(), 4)
    for t in range(3):
        lp = sc.log_probs(t, st)
        ref = torch.log_softmax(torch.from_numpy(D.joint_logits(z[t], st.p, W).astype(np.float64)), 0).numpy()
        np.testing.assert_allclose(lp, ref, rtol=0, atol=2e-5)
        assert abs(float(np.exp(lp.astype(np.float64)).sum()) - 1.0) < 1e-5
