"""GPU parity of the batched greedy RNN-T + EOU decoder (include/cac_decode.h)
against the fp32 oracle (oracle/decoder.py) on seeded projected-encoder frames.

Both sides decide every argmax in fp32 but sum in different orders, so where the
oracle's top-1 / top-2 logit margin is within fp32 rounding the GPU may take the
other class.  The comparison walks the oracle's decisions: emissions must match
exactly up to the first decision where they differ, and that decision must be
such a near tie (margin <= TIE); the stream is not compared after it.
Predictor states are compared (fp32 tolerance) for streams without one."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import TINY_DECODER, EOU_DECODER  # noqa: E402
from oracle import decoder as O  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIE = 1e-3       # logit margin below which fp32 evaluation order may flip a decision
STATE_TOL = 1e-4


def _native():
    from cache_aware_conformer_gb300 import native
    return native


def _make(dc, n_streams, seed=0, tweak=None):
    W = synth.make_decoder_weights(dc, seed)
    if tweak:
        tweak(W)
    dec = _native().Decoder(dc, synth.pack_decoder_weights(dc, W), n_streams)
    return W, dec


def _compare(em_gpu, z, state, W, dc):
    """Emissions of the GPU for frames z from `state` against the oracle's
    decisions; returns (oracle state after z or None if diverged at a tie,
    number of decisions)."""
    rec = O.decision_margins(z, state, W, dc)
    j = 0
    for t, k, margin in rec:
        if k != dc.blank:
            ok = j < len(em_gpu) and em_gpu[j] == (t, k)
            if ok:
                j += 1
                continue
        else:
            ok = not (j < len(em_gpu) and em_gpu[j][0] == t)
            if ok:
                continue
        assert margin <= TIE, f"decision at frame {t}: oracle {k} (margin {margin:.3g}), gpu {em_gpu[j:j + 2]}"
        return None, len(rec)
    assert j == len(em_gpu), (em_gpu[j:], "emitted beyond the oracle's decisions")
    _, st = O.decode_chunk(z, state, W, dc)
    return st, len(rec)


def _gpu_emissions(tokens, frames, counts):
    tok, fr, cn = tokens.cpu().numpy(), frames.cpu().numpy(), counts.cpu().numpy()
    return [[(int(fr[b, i]), int(tok[b, i])) for i in range(cn[b])] for b in range(len(cn))]


def _run(dc, n_streams, n_frames, T, seed=0, tweak=None, resets=None, sample=None, strided=False):
    """Decode n_streams x n_frames in steps of T frames; resets: {step: [ids]}.
    Compares every (sampled) stream against the oracle; returns stats."""
    W, dec = _make(dc, n_streams, seed, tweak)
    ids = list(range(n_streams))
    zs = np.stack([synth.make_joint_frames(n_frames, s, dc.joint_dim) for s in ids])
    sample = ids if sample is None else sample
    states = {s: O.DecoderState.fresh(W, dc) for s in sample}
    live = set(sample)
    total_em, decisions, ties = 0, 0, 0
    for step, t0 in enumerate(range(0, n_frames, T)):
        if resets and step in resets:
            dec.reset(resets[step])
            for s in resets[step]:
                if s in states:
                    states[s] = O.DecoderState.fresh(W, dc)
                    live.add(s)
        zc = zs[:, t0:t0 + T]
        if strided:  # slots T + 3 frames apart
            big = torch.zeros(n_streams, zc.shape[1] + 3, dc.joint_dim, device=DEV)
            big[:, :zc.shape[1]] = torch.from_numpy(zc).to(DEV)
            zt = big[:, :zc.shape[1]]
        else:
            zt = torch.from_numpy(np.ascontiguousarray(zc)).to(DEV)
        tokens, frames, counts = dec.step(ids, zt)
        dec.check()
        em = _gpu_emissions(tokens, frames, counts)
        cn = counts.cpu().numpy()
        assert (cn >= 0).all() and (cn <= zc.shape[1] * dc.max_symbols).all()
        for b in ids:
            f = [t for t, _ in em[b]]
            assert f == sorted(f) and all(0 <= t < zc.shape[1] for t in f)
            assert all(0 <= k < dc.classes and k != dc.blank for _, k in em[b])
            total_em += len(em[b])
        for s in sorted(live):
            st, nd = _compare(em[s], zc[s], states[s], W, dc)
            decisions += nd
            if st is None:
                ties += 1
                live.discard(s)
            else:
                states[s] = st
    for s in sorted(live):
        h, c, p, primed = dec.state(s)
        assert primed == 1
        np.testing.assert_allclose(h, states[s].h, rtol=0, atol=STATE_TOL)
        np.testing.assert_allclose(c, states[s].c, rtol=0, atol=STATE_TOL)
        np.testing.assert_allclose(p, states[s].p, rtol=0, atol=STATE_TOL)
    dec.close()
    print(f"[decode] {dc.vocab}-token x {n_streams} streams x {n_frames} frames: {total_em} emissions, "
          f"{decisions} compared decisions, {ties} near-tie divergences, {len(live)} states compared")
    return total_em, decisions, ties, len(live)


def test_tiny_decoder_matches_oracle():
    em, nd, ties, live = _run(TINY_DECODER, 8, 30, 2)
    assert em > 0 and ties <= 1 and live >= 7


def test_eou_decoder_matches_oracle_64_streams():
    em, nd, ties, live = _run(EOU_DECODER, 64, 20, 2)
    assert em > 100 and ties <= 2


def test_full_size_256_streams_sampled():
    """256 streams, two frames per step (one 160 ms push), six steps; 16
    sampled streams against the oracle, properties on all."""
    sample = [0, 255] + list(range(17, 255, 17))
    em, nd, ties, live = _run(EOU_DECODER, 256, 12, 2, sample=sample)
    assert ties <= 2 and live >= 14


def test_resets_and_strided_frames():
    em, nd, ties, live = _run(TINY_DECODER, 6, 24, 4, resets={2: [1, 4], 4: [4]}, strided=True)
    assert ties <= 1


def test_eou_emitted_and_advances_predictor():
    """EOU favoured: it is emitted often, and the predictor advances on it."""
    def tweak(W):
        W["out.b"][TINY_DECODER.eou] += 2.5
    em, nd, ties, live = _run(TINY_DECODER, 4, 16, 2, tweak=tweak)
    W, dec = _make(TINY_DECODER, 1, tweak=tweak)
    z = torch.from_numpy(synth.make_joint_frames(8, 0, TINY_DECODER.joint_dim)[None]).to(DEV)
    tokens, frames, counts = dec.step([0], z)
    toks = tokens[0, :counts[0]].cpu().numpy().tolist()
    assert TINY_DECODER.eou in toks
    dec.close()


def test_forced_blank_after_max_symbols():
    dc = replace(TINY_DECODER, blank_bias=-1e4)
    W, dec = _make(dc, 3)
    z = torch.from_numpy(np.stack([synth.make_joint_frames(5, s, dc.joint_dim) for s in range(3)])).to(DEV)
    tokens, frames, counts = dec.step([0, 1, 2], z)
    assert counts.cpu().numpy().tolist() == [5 * dc.max_symbols] * 3
    fr = frames.cpu().numpy()
    assert (fr == np.repeat(np.arange(5), dc.max_symbols)[None]).all()
    dec.close()


def test_all_blank_keeps_primed_state():
    dc = replace(EOU_DECODER, blank_bias=1e4)
    W, dec = _make(dc, 2)
    z = torch.from_numpy(np.stack([synth.make_joint_frames(6, s, dc.joint_dim) for s in range(2)])).to(DEV)
    tokens, frames, counts = dec.step([1, 0], z)
    assert counts.cpu().numpy().tolist() == [0, 0]
    fresh = O.DecoderState.fresh(W, dc)
    h, c, p, primed = dec.state(1)
    assert primed == 1
    np.testing.assert_allclose(h, fresh.h, rtol=0, atol=STATE_TOL)
    np.testing.assert_allclose(p, fresh.p, rtol=0, atol=STATE_TOL)
    dec.close()


def test_degenerate_calls():
    native = _native()
    W, dec = _make(TINY_DECODER, 4)
    z = torch.zeros(2, 0, TINY_DECODER.joint_dim, device=DEV)
    tokens, frames, counts = dec.step([0, 1], z)  # T = 0: nothing decoded, counts zero
    assert counts.cpu().numpy().tolist() == [0, 0]
    zz = torch.zeros(2, 2, TINY_DECODER.joint_dim, device=DEV)
    for bad in ([0, 0], [0, 4], [-1, 1]):
        with pytest.raises(native.CacError):
            dec.step(bad, zz)
    dec.check()
    dec.close()


def test_bounded_waits_give_up_and_context_survives():
    """Failure detection without a GPU fault: the library's mbarrier wait and
    the decoder's grid barrier, given nothing that satisfies them, give up
    after their limits and latch CAC_E_TIMEOUT; the context keeps working."""
    native = _native()
    assert native.wait_selftest(0) == -8   # CAC_E_TIMEOUT
    assert native.wait_selftest(1) == -8
    assert native.wait_selftest(2) == -1   # CAC_E_INVAL
    em, nd, ties, live = _run(TINY_DECODER, 2, 6, 2)
    assert live + ties == 2
