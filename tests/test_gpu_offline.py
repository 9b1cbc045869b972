"""GPU parity of the offline chunked-causal encode against the fp64 oracle, and
of streaming against offline on the GPU (the pages' gate, at bf16 tolerance)."""
from dataclasses import replace

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import TINY, EOU_120M, C600M  # noqa: E402
from oracle import conformer as O  # noqa: E402

from _util import assert_close, make_model  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("cfg,lens", [
    (TINY, [320, 203, 57]),
    (replace(EOU_120M, n_layers=2), [1501, 800, 9]),
    (replace(C600M, n_layers=2), [1501, 1337]),
    (replace(EOU_120M, n_layers=2, att_chunk=4, att_left=20), [1501, 1100, 37]),
    (replace(EOU_120M, n_layers=2, att_chunk=1, att_left=33), [1400, 1501]),
    (replace(EOU_120M, n_layers=1), [1203]),
], ids=["fp32-tiny", "bf16-eou", "bf16-600m", "bf16-chunk4-left20", "bf16-chunk1-left33", "bf16-one-short"])
def test_offline_encode_matches_oracle(cfg, lens):
    W, model = make_model(cfg)
    t = max(lens)
    mels = [synth.make_mel(n, 40 + k) for k, n in enumerate(lens)]
    batch = np.zeros((len(lens), t, 128), np.float32)
    for k, m in enumerate(mels):
        batch[k, :len(m)] = m
    enc, joint, out_len = model.encode_offline(torch.from_numpy(batch).to(DEV), lens)
    model.check()
    for k, m in enumerate(mels):
        er, jr = O.encode_offline(m, W, cfg)
        assert out_len[k] == er.shape[0] == O.subsampled_len(len(m))
        assert_close(enc[k, :out_len[k]].cpu().numpy(), er, cfg, f"enc window {k}")
        assert_close(joint[k, :out_len[k]].cpu().numpy(), jr, cfg, f"joint window {k}")


def test_gpu_streaming_equals_gpu_offline():
    """The gate of the pages on the GPU itself: chunk-by-chunk with caches vs the
    offline masked encode of the same audio (bf16; both round the same way up to
    accumulation order, so the bf16 tolerance applies)."""
    from cache_aware_conformer_gb300 import native
    cfg = replace(EOU_120M, n_layers=3)
    _, model = make_model(cfg)
    mel = synth.make_mel(1203, 77)
    enc_off, _, out_len = model.encode_offline(torch.from_numpy(mel[None]).to(DEV), [1203])
    pool = native.Pool(model, 2, 8)
    sid = pool.create_stream()
    outs = []
    for i in range(0, 1200, 16):
        e, _, _ = pool.push([sid], torch.from_numpy(mel[None, i:i + 16]).to(DEV))
        outs.append(e[0].cpu().numpy())
    e, _, n = pool.flush([sid], torch.from_numpy(mel[None, 1200:]).to(DEV), [3])
    outs.append(e[0, :n[0]].cpu().numpy())
    st = np.concatenate(outs)
    assert st.shape[0] == out_len[0] == 151
    assert_close(st, enc_off[0, :151].cpu().numpy(), cfg, "stream vs offline")


def test_offline_many_tiles_persistent_gemm():
    """Enough windows that every projection of the 600M layer shapes has more
    than two 128 x 128 output tiles per SM (the persistent GEMM path), with
    ragged lengths so the last row tile is partial; sampled windows against the
    oracle."""
    cfg = replace(C600M, n_layers=2)
    W, model = make_model(cfg)
    lens = [1501] * 40
    lens[17], lens[39] = 777, 1203
    batch = np.zeros((len(lens), 1501, 128), np.float32)
    sample = [0, 17, 39]
    mels = {}
    for k, n in enumerate(lens):
        m = synth.make_mel(n, 300 + k)
        batch[k, :n] = m
        if k in sample:
            mels[k] = m
    enc, joint, out_len = model.encode_offline(torch.from_numpy(batch).to(DEV), lens)
    model.check()
    for k in sample:
        er, jr = O.encode_offline(mels[k], W, cfg)
        assert out_len[k] == er.shape[0]
        assert_close(enc[k, :out_len[k]].cpu().numpy(), er, cfg, f"enc window {k}")
        assert_close(joint[k, :out_len[k]].cpu().numpy(), jr, cfg, f"joint window {k}")
