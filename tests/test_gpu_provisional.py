"""GPU parity of the right-context provisional-tail variant against the
oracle's same algorithm ("True streaming encode", §Status, Nemotron variant):
window mask [p - 70, p + 3], passes of emit + lookahead frames emitting
`emit`, K/V and conv tail committed for emitted frames only, and the flush
that drains the held-back frames with truncated lookahead."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import TINY, EOU_RC3  # noqa: E402
from oracle import conformer as O  # noqa: E402

from _util import assert_close, make_model  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [replace(TINY, right_context=3, emit_frames=4, lookahead_frames=16),
                                 replace(EOU_RC3, n_layers=2)], ids=["fp32", "bf16"])
def test_provisional_tail_matches_oracle(cfg):
    from cache_aware_conformer_gb300 import native
    W, model = make_model(cfg)
    pool = native.Pool(model, 4, 8)
    ids = [pool.create_stream() for _ in range(3)]
    lens = [960, 1100, 700]                      # different lengths: streams drain at different times
    mels = [synth.make_mel(n, 70 + k) for k, n in enumerate(lens)]
    refs = [O.ProvisionalTailEncoder(W, cfg) for _ in ids]
    got = [[] for _ in ids]
    want = [[] for _ in ids]
    pos = 0
    while pos + 32 <= min(lens):
        e, j, n_out = pool.push(ids, torch.from_numpy(np.stack([m[pos:pos + 32] for m in mels])).cuda())
        for b, r in enumerate(refs):
            er, jr = r.push(mels[b][pos:pos + 32])
            assert n_out[b] == er.shape[0], (pos, b, n_out[b], er.shape)
            got[b].append(e[b, :n_out[b]].cpu().numpy())
            want[b].append(er)
        pos += 32
    # the rest of every stream goes through flush (ragged tails, held-back frames)
    rest = [m[pos:] for m in mels]
    stride = max(len(x) for x in rest)
    mel_t = np.zeros((3, stride, 128), np.float32)
    for b, x in enumerate(rest):
        mel_t[b, :len(x)] = x
    e, j, n_out = pool.flush(ids, torch.from_numpy(mel_t).cuda(), [len(x) for x in rest])
    pool.check()
    for b, r in enumerate(refs):
        er, jr = r.flush(rest[b])
        assert n_out[b] == er.shape[0]
        got[b].append(e[b, :n_out[b]].cpu().numpy())
        want[b].append(er)
        g, w_ = np.concatenate(got[b]), np.concatenate(want[b])
        assert g.shape == w_.shape == (O.subsampled_len(lens[b]), cfg.d_model)
        assert_close(g, w_, cfg, f"stream {b}")


def test_provisional_push_emits_nothing_until_lookahead_is_full():
    from cache_aware_conformer_gb300 import native
    cfg = replace(TINY, right_context=3, emit_frames=4, lookahead_frames=16)
    _, model = make_model(cfg)
    pool = native.Pool(model, 2, 8)
    sid = pool.create_stream()
    mel = synth.make_mel(320, 9)
    outs = [pool.push([sid], torch.from_numpy(mel[None, i:i + 32]).cuda())[2][0] for i in range(0, 320, 32)]
    # 4 frames per push; the first pass needs 20 frames waiting (5 pushes)
    assert outs == [0, 0, 0, 0, 4, 4, 4, 4, 4, 4]
    st = pool.get_state(sid)
    assert st["subT"] == 24 and st["finished"] == 0
