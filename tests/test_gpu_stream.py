"""GPU parity of the streaming chunk step against the fp64 oracle, through the C-ABI.

Every test here runs the CUDA library (tcgen05 GEMMs in bf16 mode, SIMT GEMMs in
fp32 mode) on seeded synthetic inputs and compares element by element with the
oracle's streaming encoder on the same inputs."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import TINY, EOU_120M  # noqa: E402
from oracle import conformer as O  # noqa: E402

from _util import assert_close, make_model, max_abs, cosine  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"

EOU2 = replace(EOU_120M, n_layers=2)


def _push(pool, ids, mels):
    enc, joint, n_out = pool.push(ids, torch.from_numpy(np.stack(mels)).to(DEV))
    return enc.cpu().numpy(), joint.cpu().numpy(), n_out


# ---------------------------------------------------------------------------
# per-kernel taps: each kernel of the step against the oracle's intermediates
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [TINY, EOU2], ids=["fp32", "bf16"])
def test_kernel_taps_match_oracle(cfg):
    from cache_aware_conformer_gb300 import native
    W, model = make_model(cfg)
    pool = native.Pool(model, 4, 8)
    sid = pool.create_stream()
    ref = O.StreamingEncoder(W, cfg)
    mel = synth.make_mel(160, 1)
    pool.set_trace(True)
    names = ["ff1", "att", "x_att", "glu", "conv", "x_conv", "out"]
    # chunk 1 exercises the first-chunk padding, chunk 3 a filled cache
    for k in range(5):
        chunk = mel[32 * k: 32 * (k + 1)]
        tr = {}
        ref.push(chunk, trace=tr)
        _push(pool, [sid], [chunk])
        pool.check()
        # the whole-step bars, at every tap and every layer (no growth with
        # depth): the residual stream keeps a scale of about one, so a kernel
        # that adds error in a deeper layer fails here as it would in the first
        tol = 1e-4 if cfg.dtype == "fp32" else 3e-2
        assert max_abs(pool.read_trace(0, 7, 4), tr["sub"]) <= tol, ("sub", k)
        for l in range(cfg.n_layers):
            for t, name in enumerate(names):
                got = pool.read_trace(l, t, 4)
                d = max_abs(got, tr[name][l])
                assert d <= tol, (k, l, name, d)


# ---------------------------------------------------------------------------
# whole-step parity
# ---------------------------------------------------------------------------
def test_tiny_fp32_stream_320_frames_matches_oracle():
    """3.2 s pushed 16 mel frames (160 ms) at a time, fp32 mode, <= 1e-4."""
    from cache_aware_conformer_gb300 import native
    cfg = TINY
    W, model = make_model(cfg)
    pool = native.Pool(model, 2, 8)
    sid = pool.create_stream()
    ref = O.StreamingEncoder(W, cfg)
    mel = synth.make_mel(320, 0)
    for i in range(0, 320, 16):
        e, j, n_out = _push(pool, [sid], [mel[i:i + 16]])
        er, jr = ref.push(mel[i:i + 16])
        assert n_out == [2]
        assert_close(e[0], er, cfg, f"enc push {i // 16}")
        assert_close(j[0], jr, cfg, f"joint push {i // 16}")
    pool.check()


@pytest.mark.parametrize("gemm_simt", [False, True], ids=["tcgen05", "simt"])
def test_bf16_multistream_mixed_push_sizes(gemm_simt):
    """Several streams, pushes of 16/32/64 mel, ragged flush, bf16 tolerance."""
    from cache_aware_conformer_gb300 import native
    cfg = EOU2
    W, model = make_model(cfg, gemm_simt=gemm_simt)
    pool = native.Pool(model, 8, 8)
    ids = [pool.create_stream() for _ in range(3)]
    refs = [O.StreamingEncoder(W, cfg) for _ in ids]
    mels = [synth.make_mel(700, 10 + k) for k in range(3)]
    pos = 0
    got = [[] for _ in ids]
    want = [[] for _ in ids]
    for n in [16, 32, 64, 16, 48, 64, 64, 128, 64, 16, 32, 64, 64]:
        if pos + n > 690:
            break
        e, j, n_out = _push(pool, ids, [m[pos:pos + n] for m in mels])
        for b, r in enumerate(refs):
            er, jr = r.push(mels[b][pos:pos + n])
            got[b].append(e[b]); want[b].append(er)
        pos += n
    rem = [700 - pos - 3 * k for k in range(3)]
    mel_t = torch.from_numpy(np.stack([np.pad(m[pos:], ((0, 0), (0, 0))) for m in mels])).to(DEV)
    e, j, n_out = pool.flush(ids, mel_t, rem)
    for b, r in enumerate(refs):
        er, jr = r.flush(mels[b][pos:pos + rem[b]])
        assert n_out[b] == er.shape[0] == (rem[b] + 7) // 8
        got[b].append(e[b, :n_out[b]].cpu().numpy()); want[b].append(er)
    for b in range(3):
        assert_close(np.concatenate(got[b]), np.concatenate(want[b]), cfg, f"stream {b}")
    pool.check()


def test_tcgen05_and_simt_gemm_paths_agree():
    """The same bf16 step on the tcgen05 GEMM and on the SIMT twin: only the fp32
    accumulation order differs."""
    from cache_aware_conformer_gb300 import native
    cfg = EOU2
    mel = synth.make_mel(128, 3)
    outs = []
    for simt in (False, True):
        _, model = make_model(cfg, gemm_simt=simt)
        pool = native.Pool(model, 2, 8)
        sid = pool.create_stream()
        outs.append([_push(pool, [sid], [mel[i:i + 32]])[:2] for i in range(0, 128, 32)])
        pool.check()
    for (e0, j0), (e1, j1) in zip(*outs):
        assert max_abs(e0, e1) < 2e-2 and cosine(e0, e1) > 0.9999


def test_graph_replay_matches_eager():
    from cache_aware_conformer_gb300 import native
    cfg = EOU2
    _, model = make_model(cfg)
    res = []
    for graphs in (False, True):
        pool = native.Pool(model, 4, 8)
        ids = [pool.create_stream() for _ in range(4)]
        pool.set_graphs(graphs)
        mel_all = np.stack([synth.make_mel(160, 20 + k) for k in range(4)])
        mel_dev = torch.from_numpy(mel_all).to(DEV)
        enc = torch.zeros(4, 2, cfg.d_model, device=DEV)
        joint = torch.zeros(4, 2, cfg.joint_dim, device=DEV)
        outs = []
        buf = torch.empty(4, 16, 128, device=DEV)   # one staging buffer: the graph key repeats
        for i in range(0, 160, 16):
            buf.copy_(mel_dev[:, i:i + 16])
            pool.push_into(ids, buf, enc, joint)
            outs.append(enc.cpu().numpy().copy())
        res.append(np.concatenate(outs, 1))
        if graphs:
            # 10 pushes: 1 eager, 1 capture + replay, 8 replays of the same graph
            assert pool.launch_count() > 0
        pool.check()
        pool.close()
    assert np.array_equal(res[0], res[1])


def test_state_bookkeeping_is_exact():
    """subT, Lc, the K/V ring contents in absolute-position order and the conv tail
    match the oracle's caches after pushes, resets and more pushes."""
    from cache_aware_conformer_gb300 import native
    cfg = replace(TINY, att_left=10)
    W, model = make_model(cfg)
    pool = native.Pool(model, 4, 8)
    sid = pool.create_stream()
    ref = O.StreamingEncoder(W, cfg)
    mel = synth.make_mel(480, 5)
    for k, n in enumerate([16, 32, 16, 64, 16, 16, 48]):
        off = sum([16, 32, 16, 64, 16, 16, 48][:k])
        _push(pool, [sid], [mel[off:off + n]])
        ref.push(mel[off:off + n])
        st = pool.get_state(sid)
        assert st["subT"] == ref.subT and st["Lc"] == ref.Lc == min(ref.subT, 10)
        for l in range(cfg.n_layers):
            assert max_abs(st["k"][l, :ref.Lc], ref.k[l]) <= 1e-4
            assert max_abs(st["v"][l, :ref.Lc], ref.v[l]) <= 1e-4
            assert max_abs(st["conv"][l], ref.conv[l]) <= 1e-4
        assert max_abs(st["mel_tail"], ref.mel_tail) <= 1e-6
    pool.reset([sid])
    ref.reset()
    st = pool.get_state(sid)
    assert st["subT"] == 0 and st["Lc"] == 0
    e, _, _ = _push(pool, [sid], [mel[:16]])
    er, _ = ref.push(mel[:16])
    assert_close(e[0], er, cfg, "after reset")


def test_state_export_import_migrates_a_stream():
    from cache_aware_conformer_gb300 import native
    cfg = TINY
    W, model = make_model(cfg)
    pool = native.Pool(model, 4, 8)
    a, b = pool.create_stream(), pool.create_stream()
    mel = synth.make_mel(400, 6)
    for i in range(0, 320, 32):
        _push(pool, [a], [mel[i:i + 32]])
    pool.set_state(b, pool.get_state(a))
    ea, _, _ = _push(pool, [a], [mel[320:352]])
    eb, _, _ = _push(pool, [b], [mel[320:352]])
    assert max_abs(ea, eb) == 0.0


def test_errors_are_reported():
    from cache_aware_conformer_gb300 import native
    cfg = TINY
    _, model = make_model(cfg)
    pool = native.Pool(model, 2, 8)
    sid = pool.create_stream()
    with pytest.raises(native.CacError) as e:
        pool.push([sid], torch.zeros(1, 24, 128, device=DEV))
    assert e.value.code == -2  # not a multiple of 16 mel frames
    with pytest.raises(native.CacError) as e:
        pool.push([sid, sid], torch.zeros(2, 16, 128, device=DEV))
    assert e.value.code == -1  # duplicate id
    bad = torch.zeros(1, 16, 128, device=DEV)
    bad[0, 3, 7] = float("nan")
    pool.push([sid], bad)
    with pytest.raises(native.CacError) as e:
        pool.check()
    assert e.value.code == -7
    pool.flush([sid], None, [0])
    with pytest.raises(native.CacError) as e:
        pool.push([sid], torch.zeros(1, 16, 128, device=DEV))
    assert e.value.code == -3  # push after flush without reset
    pool.reset([sid])
    pool.push([sid], torch.zeros(1, 16, 128, device=DEV))
    pool.check()


def test_pool_exhaustion_and_a_refused_allocation_leave_the_library_usable():
    """Faults injected on the host: a pool hands out at most max_streams ids
    (CAC_E_NOMEM after that, a destroyed id is handed out again), and a pool
    larger than the device's memory is refused with CAC_E_NOMEM; afterwards
    pushes on the existing pool run and report no error (the refused
    allocation leaves no error behind for the next launch check)."""
    from cache_aware_conformer_gb300 import native
    cfg = EOU2
    W, model = make_model(cfg)
    pool = native.Pool(model, 2, 8)
    a, b = pool.create_stream(), pool.create_stream()
    with pytest.raises(native.CacError) as e:
        pool.create_stream()
    assert e.value.code == -4
    pool.destroy_stream(b)
    assert pool.create_stream() == b
    # 2,000,000 streams of this model: 328 GB for each of the K and V rings
    with pytest.raises(native.CacError) as e:
        native.Pool(model, 2_000_000, 8)
    assert e.value.code == -4
    mel = synth.make_mel(32, 4)
    enc, _, n_out = _push(pool, [a, b], [mel, mel])
    pool.check()
    model.check()
    ref = O.StreamingEncoder(W, cfg)
    e_ref, _ = ref.push(mel)
    assert n_out == [4, 4] and np.array_equal(enc[0], enc[1])
    assert_close(enc[0], e_ref, cfg, "after a refused pool")


def test_push_host_matches_device_push():
    from cache_aware_conformer_gb300 import native
    cfg = EOU2
    _, model = make_model(cfg)
    pools = [native.Pool(model, 2, 8) for _ in range(2)]
    ids = [p.create_stream() for p in pools]
    mel = synth.make_mel(64, 9)
    e0, j0, _ = _push(pools[0], [ids[0]], [mel])
    e1, j1, n1 = pools[1].push_host([ids[1]], mel[None])
    assert n1 == [8] and np.array_equal(e0, e1) and np.array_equal(j0, j1)
    # page-locked buffers take the direct-copy path: same results
    pools.append(native.Pool(model, 2, 8))
    ids.append(pools[2].create_stream())
    mel_p = torch.from_numpy(mel[None]).pin_memory()
    out = (torch.empty(1, 8, cfg.d_model).pin_memory(), torch.empty(1, 8, cfg.joint_dim).pin_memory())
    e2, j2, n2 = pools[2].push_host([ids[2]], mel_p, out=out)
    assert n2 == [8] and np.array_equal(e0, e2.numpy()) and np.array_equal(j0, j2.numpy())


def test_push_host_sub_batches_match_device_push():
    """A host-buffer push over 256 streams runs as concurrent 64-stream
    sub-batches that copy their own mel slices in and frames out: equal to the
    device push of the same mel bit for bit, over several 160 ms steps (graph
    replay on both pools), with page-locked and with pageable buffers."""
    from cache_aware_conformer_gb300 import native
    cfg = EOU2
    _, model = make_model(cfg)
    S = 256
    pools = [native.Pool(model, S, 2) for _ in range(3)]
    for p in pools:
        p.set_graphs(True)
    ids = [[p.create_stream() for _ in range(S)] for p in pools]
    out = (torch.empty(S, 2, cfg.d_model).pin_memory(), torch.empty(S, 2, cfg.joint_dim).pin_memory())
    for step in range(4):
        mel = np.stack([synth.make_mel(16, 100 * step + s) for s in range(S)])
        e0, j0, _ = _push(pools[0], ids[0], list(mel))
        e1, j1, n1 = pools[1].push_host(ids[1], torch.from_numpy(mel).pin_memory(), out=out)
        e2, j2, n2 = pools[2].push_host(ids[2], mel)
        assert n1 == [2] * S and n2 == [2] * S
        assert np.array_equal(e0, e1.numpy()) and np.array_equal(j0, j1.numpy()), step
        assert np.array_equal(e0, e2) and np.array_equal(j0, j2), step
    for p in pools:
        p.check()


@pytest.mark.parametrize("S", [256, 16], ids=["sub_batches", "one_batch"])
def test_push_host_async_pipelined_matches_device_push(S):
    """Queued host-buffer pushes (cac_stream_push_host_async), each queued
    before the host reads the previous one's frames from a second pair of
    page-locked buffers, with resets queued between them: equal bit for bit
    to device pushes of the same mel (graph replay on both pools), for a push
    that runs as concurrent sub-batches (256 streams) and one that runs as one
    batch (16).  Pageable buffers are refused before anything is queued."""
    from cache_aware_conformer_gb300 import native
    cfg = EOU2
    _, model = make_model(cfg)
    pools = [native.Pool(model, S, 2) for _ in range(2)]
    for p in pools:
        p.set_graphs(True)
    ids = [[p.create_stream() for _ in range(S)] for p in pools]
    steps = 6
    mels = [np.stack([synth.make_mel(16, 7000 + 100 * step + s) for s in range(S)]) for step in range(steps)]
    resets = {2: [0, S // 2, S - 1], 4: [1, 5]}
    want = []
    for step in range(steps):
        pools[0].reset([ids[0][i] for i in resets.get(step, [])])
        e0, j0, _ = _push(pools[0], ids[0], list(mels[step]))
        want.append((e0, j0))
    host_mel = [torch.from_numpy(m).pin_memory() for m in mels]
    outs = [(torch.empty(S, 2, cfg.d_model).pin_memory(), torch.empty(S, 2, cfg.joint_dim).pin_memory())
            for _ in range(2)]
    evs = [torch.cuda.Event() for _ in range(2)]
    for step in range(steps):
        pools[1].reset([ids[1][i] for i in resets.get(step, [])])
        n_out = pools[1].push_host_async(ids[1], host_mel[step], outs[step % 2])
        assert n_out == [2] * S
        evs[step % 2].record()
        if step > 0:  # the previous push's frames, read while this one runs
            evs[(step - 1) % 2].synchronize()
            e, j = outs[(step - 1) % 2]
            assert np.array_equal(e.numpy(), want[step - 1][0]), step - 1
            assert np.array_equal(j.numpy(), want[step - 1][1]), step - 1
    evs[(steps - 1) % 2].synchronize()
    e, j = outs[(steps - 1) % 2]
    assert np.array_equal(e.numpy(), want[-1][0]) and np.array_equal(j.numpy(), want[-1][1])
    for bad in ((torch.from_numpy(mels[0]), outs[0]),
                (host_mel[0], (torch.empty(S, 2, cfg.d_model), outs[0][1]))):
        with pytest.raises(native.CacError) as err:
            pools[1].push_host_async(ids[1], *bad)
        assert err.value.code == -1
    for p in pools:
        p.check()


def test_c600m_shape_multistream():
    """The 600M encoder's layer shapes (d_model 1024, 16 heads, ff 4096), two
    layers, three streams with 160 / 320 / 640 ms pushes and a ragged flush."""
    from dataclasses import replace
    from cache_aware_conformer_gb300 import native
    from cache_aware_conformer_gb300.config import C600M
    cfg = replace(C600M, n_layers=2)
    W, model = make_model(cfg)
    pool = native.Pool(model, 4, 8)
    ids = [pool.create_stream() for _ in range(3)]
    refs = [O.StreamingEncoder(W, cfg) for _ in ids]
    mels = [synth.make_mel(300, 40 + k) for k in range(3)]
    pos = 0
    got = [[] for _ in ids]
    want = [[] for _ in ids]
    for n in [16, 32, 16, 64, 16, 32, 64]:
        e, j, n_out = _push(pool, ids, [m[pos:pos + n] for m in mels])
        for b, r in enumerate(refs):
            er, jr = r.push(mels[b][pos:pos + n])
            got[b].append(e[b]); want[b].append(er)
        pos += n
    rem = [300 - pos - 5 * k for k in range(3)]
    mel_t = torch.from_numpy(np.stack([m[pos:] for m in mels])).to(DEV)
    e, j, n_out = pool.flush(ids, mel_t, rem)
    for b, r in enumerate(refs):
        er, jr = r.flush(mels[b][pos:pos + rem[b]])
        got[b].append(e[b, :n_out[b]].cpu().numpy()); want[b].append(er)
        assert_close(np.concatenate(got[b]), np.concatenate(want[b]), cfg, f"c600m stream {b}")
    pool.check()
