"""Chained steps (cac_pool_set_chains(p, 1), off by default): the projections
and LayerNorms between two attention launches run as one persistent kernel
whose 128-row blocks move phase by phase on completion counters ("True
streaming encode — implementation spec", §Per-chunk flow steps 2-4).

Both paths compute the same step in bf16 with fp32 accumulation, but split-K
sums run in different orders, and bf16 roundings downstream turn those fp32
differences into independent rounding patterns: two correct pools differ by
about as much as each differs from the fp64 oracle (~1e-2 at 3 layers, measured).
So each path is compared with the oracle on sampled streams (the bf16 bar), the
chained path must be no less accurate than the per-projection one, and the two
must agree in direction (cosine).  The chained step is deterministic (the last
split to finish adds the partials in split order): a graph replay equals the
eager launch bit for bit.  Cases: ragged batches (partial row blocks), one
stream, resets, a flush with an odd last chunk, d_model 1024.  (The other
streaming parity tests run the default per-projection path.)"""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import EOU_120M, C600M  # noqa: E402
from oracle import conformer as O  # noqa: E402

from _util import BF16_MAX_ABS, BF16_MIN_COS, cosine, max_abs  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _pair(cfg, S, nmax=2):
    from cache_aware_conformer_gb300 import native
    W = synth.make_weights(cfg, 0)
    model = native.Model(cfg, synth.pack_weights(cfg, W))
    a = native.Pool(model, S, nmax)
    a.set_chains(True)
    b = native.Pool(model, S, nmax)
    b.set_chains(False)
    ia = [a.create_stream() for _ in range(S)]
    ib = [b.create_stream() for _ in range(S)]
    return W, model, a, b, ia, ib


def _run(cfg, S, steps, resets, seed, sample):
    W, model, a, b, ia, ib = _pair(cfg, S)
    mel = np.stack([synth.make_mel(16 * steps + 8, seed + s) for s in range(S)])
    md = torch.from_numpy(mel).to(DEV)
    got = {k: [] for k in ("a", "b")}
    la0, lb0 = a.launch_count(), b.launch_count()
    for t in range(steps):
        if t in resets:
            a.reset([ia[i] for i in resets[t]])
            b.reset([ib[i] for i in resets[t]])
        chunk = md[:, 16 * t:16 * (t + 1)].contiguous()
        ea, _, _ = a.push(ia, chunk)
        eb, _, _ = b.push(ib, chunk)
        got["a"].append(ea.cpu().numpy())
        got["b"].append(eb.cpu().numpy())
    la, lb = a.launch_count() - la0, b.launch_count() - lb0
    tail = md[:, 16 * steps:16 * steps + 8].contiguous()
    ea, _, na = a.flush(ia, tail, [8] * S)
    eb, _, nb = b.flush(ib, tail, [8] * S)
    assert list(na) == list(nb) == [1] * S
    got["a"].append(ea[:, :1].cpu().numpy())
    got["b"].append(eb[:, :1].cpu().numpy())
    a.check()
    b.check()
    for s in sample:
        sa, sb = a.get_state(ia[s]), b.get_state(ib[s])
        assert (sa["subT"], sa["Lc"], sa["finished"]) == (sb["subT"], sb["Lc"], sb["finished"])
    ga, gb = np.concatenate(got["a"], 1), np.concatenate(got["b"], 1)
    for s in sample:
        enc = O.StreamingEncoder(W, cfg)
        outs = []
        for t in range(steps):
            if t in resets and s in resets[t]:
                enc.reset()
            outs.append(enc.push(mel[s, 16 * t:16 * (t + 1)])[0])
        outs.append(enc.flush(mel[s, 16 * steps:16 * steps + 8])[0])
        ref = np.concatenate(outs)
        da, db = max_abs(ga[s], ref), max_abs(gb[s], ref)
        ca = cosine(ga[s], ref)
        print(f"[chain] S={S} stream {s}: chained {da:.2e} (cos {ca:.7f}), per-projection {db:.2e}")
        assert np.isfinite(ga[s]).all()
        assert da <= BF16_MAX_ABS and ca >= BF16_MIN_COS
        assert da <= 1.5 * db + 2e-3, (s, da, db)
    assert cosine(ga, gb) >= 0.99999
    return la, lb


@pytest.mark.parametrize("S", [256, 37, 129, 1])
def test_chained_step_matches_oracle_like_per_projection_launches(S):
    cfg = replace(EOU_120M, n_layers=3)
    resets = {2: [1, S - 1]} if S > 3 else {}
    sample = sorted({0, S // 2, S - 1} | ({1} if S > 3 else set()))
    la, lb = _run(cfg, S, 4, resets, 100, sample)
    assert 2 * la < lb    # far fewer launches per step


def test_chained_step_600m_shapes():
    """d_model 1024: FF hidden activations as split operands, 1024-wide LayerNorm rows."""
    _run(replace(C600M, n_layers=2), 64, 3, {1: [5]}, 500, [0, 5, 63])


def test_chained_step_is_deterministic_under_graph_replay():
    from cache_aware_conformer_gb300 import native
    cfg = replace(EOU_120M, n_layers=2)
    S = 128
    model = native.Model(cfg, synth.pack_weights(cfg, synth.make_weights(cfg, 0)))
    pools = []
    for graphs in (True, False):
        p = native.Pool(model, S, 2)
        p.set_chains(True)
        p.set_graphs(graphs)
        pools.append((p, [p.create_stream() for _ in range(S)]))
    mel = torch.from_numpy(np.stack([synth.make_mel(96, 300 + s) for s in range(S)])).to(DEV)
    bufs = [(torch.empty(S, 2, cfg.d_model, device=DEV), torch.empty(S, 2, cfg.joint_dim, device=DEV),
             torch.empty(S, 16, 128, device=DEV)) for _ in pools]
    for t in range(6):   # step 0 eager, step 1 captured, then replays
        outs = []
        for (p, ids), (enc, joint, buf) in zip(pools, bufs):
            buf.copy_(mel[:, 16 * t:16 * (t + 1)])
            p.push_into(ids, buf, enc, joint)
            outs.append((enc.cpu().numpy(), joint.cpu().numpy()))
        assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1]), t
    for p, _ in pools:
        p.check()
