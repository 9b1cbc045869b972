"""Full-size GPU parity: the 17-layer d_model-512 encoder in bf16 against the
fp64 oracle, (a) one 30 s stream pushed at 160 ms plus the ragged flush, and
(b) the benchmark's own 256-stream launch configuration (random even start
offsets reached by pre-roll, 1 % resets per step, CUDA graphs on), checked on
sampled streams that the oracle replays one by one."""
import multiprocessing as mp
import os
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import EOU_120M, WORKLOADS  # noqa: E402

from _util import assert_close, max_abs, cosine  # noqa: E402

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


def _oracle_stream_30s(args):
    cfg, blob_path = args
    from oracle import conformer as O
    W = synth.unpack_weights(cfg, np.load(blob_path, mmap_mode="r"))
    mel = synth.make_mel(3000, 0)
    enc = O.StreamingEncoder(W, cfg)
    outs = [enc.push(mel[i:i + 16]) for i in range(0, 2992, 16)]
    outs.append(enc.flush(mel[2992:]))
    return np.concatenate([o[0] for o in outs]), np.concatenate([o[1] for o in outs])


def _oracle_schedule(args):
    """Replay one stream of the 256-stream schedule: pre-roll, then steps with resets."""
    cfg, blob_path, sid, pre, chunks, resets = args
    from oracle import conformer as O
    W = synth.unpack_weights(cfg, np.load(blob_path, mmap_mode="r"))
    mel = synth.make_mel(375 * 16, sid)
    enc = O.StreamingEncoder(W, cfg)
    for r in range(pre):
        enc.push(mel[16 * r: 16 * (r + 1)])
    out = []
    for c, rs in zip(chunks, resets):
        if rs:
            enc.reset()
        e, j = enc.push(mel[16 * c: 16 * (c + 1)])
        out.append((e, j, enc.subT, enc.Lc))
    return out


@pytest.fixture(scope="module", autouse=True)
def single_threaded_blas_children():
    """Spawned oracle workers inherit these before they import numpy (one BLAS
    thread each, so parallel workers do not oversubscribe the host cores)."""
    keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    old = {k: os.environ.get(k) for k in keys}
    for k in keys:
        os.environ[k] = "1"
    yield
    for k, v in old.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = v


@pytest.fixture(scope="module")
def eou_blob(tmp_path_factory):
    cfg = EOU_120M
    W = synth.make_weights_parallel(cfg, seed=0, workers=8)
    blob = synth.pack_weights(cfg, W)
    path = str(tmp_path_factory.mktemp("w") / "eou.npy")
    np.save(path, blob)
    return cfg, blob, path


def test_config2_one_stream_30s(eou_blob):
    from cache_aware_conformer_gb300 import native
    cfg, blob, path = eou_blob
    with mp.get_context("spawn").Pool(1) as pool:
        fut = pool.map_async(_oracle_stream_30s, [(cfg, path)])
        model = native.Model(cfg, blob)
        p = native.Pool(model, 1, 2)
        sid = p.create_stream()
        p.set_graphs(True)
        mel = synth.make_mel(3000, 0)
        md = torch.from_numpy(mel).to(DEV)
        buf = torch.empty(1, 16, 128, device=DEV)
        enc = torch.empty(1, 2, cfg.d_model, device=DEV)
        joint = torch.empty(1, 2, cfg.joint_dim, device=DEV)
        es, js = [], []
        for i in range(0, 2992, 16):
            buf.copy_(md[i:i + 16][None])
            p.push_into([sid], buf, enc, joint)
            es.append(enc[0].cpu().numpy().copy())
            js.append(joint[0].cpu().numpy().copy())
        e, j, n = p.flush([sid], md[None, 2992:].contiguous(), [8])
        es.append(e[0, :n[0]].cpu().numpy())
        js.append(j[0, :n[0]].cpu().numpy())
        p.check()
        er, jr = fut.get()[0]
    ge, gj = np.concatenate(es), np.concatenate(js)
    assert ge.shape == er.shape == (375, cfg.d_model)
    assert_close(ge, er, cfg, "enc 30 s")
    assert cosine(gj, jr) >= 0.999 and max_abs(gj, jr) <= 6e-2


def test_config3_256_streams_sampled(eou_blob):
    """The benchmark's 256-stream schedule (pre-roll to even start offsets, 1 %
    resets per step, an utterance that ends restarts) for long enough that the
    sampled stream closest to its end wraps around: streams 0, S-1, that stream
    and 13 seeded others, every step compared with the oracle's replay."""
    import bench
    cfg, blob, path = eou_blob
    wl = WORKLOADS["eou120m_256streams_60s"]
    S = wl.streams
    n = wl.push_mel // 8
    chunks = int(round(wl.seconds * 100)) // wl.push_mel
    pre = synth.start_offsets(S, wl.max_start_offset, seed=7) // n
    wrap = int(np.argmax(pre))                                  # nearest to its utterance's end
    steps = max(100, chunks - int(pre[wrap]) + 4)
    rng = np.random.default_rng(3)
    others = rng.choice([s for s in range(1, S - 1) if s != wrap], 13, replace=False).tolist()
    sample = sorted({0, S - 1, wrap, *others})
    w = bench.StreamWorkload(wl, 0, torch.device(DEV), steps, workers=8)
    assert (w.pre == pre).all()
    # the schedule exercises what it should: mid-run resets and an utterance wrap
    reset_streams = {s for t in range(1, steps) for s in w.resets[t].tolist() if s in sample}
    assert len(reset_streams) >= 2, reset_streams
    assert any(int(w.cidx[t][wrap]) == 0 for t in range(1, steps))
    jobs = []
    for s in sample:
        jobs.append((cfg, path, s, int(w.pre[s]), [int(w.cidx[t][s]) for t in range(steps)],
                     [bool(s in set(w.resets[t].tolist())) for t in range(steps)]))
    with mp.get_context("spawn").Pool(min(len(sample), os.cpu_count() or 1)) as pool:
        fut = pool.map_async(_oracle_schedule, jobs)
        w.pool.set_graphs(True)
        got = []
        for t in range(steps):
            w.step()
            got.append((w.enc[sample].cpu().numpy(), w.joint[sample].cpu().numpy()))
        w.pool.check()
        states = {s: w.pool.get_state(s) for s in sample}
        ref = fut.get()
    for k, s in enumerate(sample):
        ge = np.concatenate([g[0][k] for g in got])
        re = np.concatenate([r[0] for r in ref[k]])
        assert_close(ge, re, cfg, f"stream {s} ({steps} steps)")
        # bookkeeping: subT and Lc after the last step are exact
        assert states[s]["subT"] == ref[k][-1][2] and states[s]["Lc"] == ref[k][-1][3]


# ---------------------------------------------------------------------------
# the 600M encoder (24 layers, d_model 1024) and the provisional-tail variant,
# each in the launch configuration the benchmark times, on sampled outputs
# ---------------------------------------------------------------------------
def _oracle_offline_window(args):
    cfg, blob_path, wid, T, silence = args
    from oracle import conformer as O
    W = synth.unpack_weights(cfg, np.load(blob_path, mmap_mode="r"))
    enc, joint = O.encode_offline(synth.make_mel(T, wid, silence_frac=silence), W, cfg)
    return enc, joint


def _oracle_schedule_any(args):
    """Replay one stream of a benchmark schedule (pre-roll, then steps with
    resets); chunked or provisional-tail encoder by the config."""
    cfg, blob_path, sid, pre, chunks, resets, push_mel, n_chunks, silence = args
    from oracle import conformer as O
    W = synth.unpack_weights(cfg, np.load(blob_path, mmap_mode="r"))
    mel = synth.make_mel(n_chunks * push_mel, sid, silence_frac=silence)
    enc = O.ProvisionalTailEncoder(W, cfg) if cfg.provisional else O.StreamingEncoder(W, cfg)
    for r in range(pre):
        enc.push(mel[push_mel * r: push_mel * (r + 1)])
    out = []
    for c, rs in zip(chunks, resets):
        if rs:
            enc.reset()
        e, _ = enc.push(mel[push_mel * c: push_mel * (c + 1)])
        out.append(e)
    return out


@pytest.fixture(scope="module")
def c600m_blob(tmp_path_factory):
    from cache_aware_conformer_gb300.config import C600M
    W = synth.make_weights_parallel(C600M, seed=0, workers=8)
    blob = synth.pack_weights(C600M, W)
    del W
    path = str(tmp_path_factory.mktemp("w600") / "c600m.npy")
    np.save(path, blob)
    return C600M, path


def test_config4a_offline_600m_sampled(c600m_blob):
    """32 windows of 1501 mel through the offline encode the benchmark times;
    windows 0 and 31 against the oracle's offline encode."""
    import bench
    cfg, path = c600m_blob
    wl = WORKLOADS["c600m_offline_32x15s"]
    sample = [0, wl.offline_batch - 1]
    jobs = [(cfg, path, w, wl.offline_mel, wl.silence_frac) for w in sample]
    with mp.get_context("spawn").Pool(len(sample)) as pool:
        fut = pool.map_async(_oracle_offline_window, jobs)
        w = bench.OfflineWorkload(wl, 0, torch.device(DEV), workers=8)
        w.step()
        torch.cuda.synchronize()
        got = [(w.enc[k].cpu().numpy(), w.joint[k].cpu().numpy()) for k in sample]
        w.model.check()
        ref = fut.get()
    for (ge, gj), (re, rj), k in zip(got, ref, sample):
        assert ge.shape == re.shape == (188, cfg.d_model)
        assert_close(ge, re, cfg, f"offline window {k}")


def _stream_schedule_test(wl, cfg, path, steps, sample):
    import bench
    w = bench.StreamWorkload(wl, 0, torch.device(DEV), steps, workers=8)
    jobs = [(cfg, path, s, int(w.pre[s]), [int(w.cidx[t][s]) for t in range(steps)],
             [bool(s in set(w.resets[t].tolist())) for t in range(steps)], w.push_mel, w.chunks, wl.silence_frac)
            for s in sample]
    with mp.get_context("spawn").Pool(len(sample)) as pool:
        fut = pool.map_async(_oracle_schedule_any, jobs)
        w.pool.set_graphs(True)
        got = {s: [] for s in sample}
        for t in range(steps):
            r = w.resets[t]
            if len(r):
                w.pool.reset([w.ids[i] for i in r])
            w.staging.copy_(w.step_mel[t])
            n_out = w.pool.push_into(w.ids, w.staging, w.enc, w.joint)
            for s in sample:
                got[s].append(w.enc[s, :n_out[s]].cpu().numpy())
            w.t += 1
        w.pool.check()
        ref = fut.get()
    for k, s in enumerate(sample):
        assert [g.shape[0] for g in got[s]] == [e.shape[0] for e in ref[k]], f"stream {s}: emitted frame counts"
        ge, re = np.concatenate(got[s]), np.concatenate(ref[k])
        assert_close(ge, re, cfg, f"stream {s}")


def test_config4b_600m_64_streams_sampled(c600m_blob):
    """Config 4b's 64-stream launch configuration, with resets added (5 % per
    stream and step) so that sampled streams restart mid-run."""
    cfg, path = c600m_blob
    wl = replace(WORKLOADS["c600m_64streams_30s"], reset_prob=0.05)
    sample = [0, 31, wl.streams - 1]
    assert any(synth.reset_mask(wl.streams, t, wl.reset_prob, seed=11)[s] for t in range(1, 16) for s in sample)
    _stream_schedule_test(wl, cfg, path, 16, sample)


def test_config5_provisional_128_streams_sampled(eou_blob):
    from cache_aware_conformer_gb300.config import EOU_RC3
    wl = WORKLOADS["eou120m_rc3_128streams_30s"]
    cfg = wl.model
    W = synth.make_weights_parallel(cfg, seed=0, workers=8)
    path = eou_blob[2].replace("eou.npy", "rc3.npy")
    np.save(path, synth.pack_weights(cfg, W))
    del W
    _stream_schedule_test(wl, cfg, path, 16, [0, 64, wl.streams - 1])


def test_config5_provisional_resets_with_pending_lookahead(eou_blob):
    """Provisional-tail pool reset between passes while subsampled frames wait
    in the x0 ring (16 lookahead frames are always pending mid-stream): the
    reset stream must restart like the oracle's ProvisionalTailEncoder.reset()."""
    wl = replace(WORKLOADS["eou120m_rc3_128streams_30s"], reset_prob=0.05)
    cfg = wl.model
    sample = [0, 64, wl.streams - 1]
    assert sum(synth.reset_mask(wl.streams, t, wl.reset_prob, seed=11)[s] for t in range(1, 16) for s in sample) >= 2
    W = synth.make_weights_parallel(cfg, seed=0, workers=8)
    path = eou_blob[2].replace("eou.npy", "rc3r.npy")
    np.save(path, synth.pack_weights(cfg, W))
    del W
    _stream_schedule_test(wl, cfg, path, 16, sample)
