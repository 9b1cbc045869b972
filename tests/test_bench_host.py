"""Host logic of the benchmark's oracle legs, on CPU: the reference arm's JSON
line (the oracle timed on the host cores in place of a reference program) and
the bounded oracle sample behind `cpu_baseline`, for the streaming, the
provisional-tail and the offline forms of a workload."""
import json
import os
import subprocess
import sys
from dataclasses import replace

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from cache_aware_conformer_gb300 import synth  # noqa: E402
from cache_aware_conformer_gb300.config import TINY, WORKLOADS  # noqa: E402


def _tiny_blob(cfg):
    return synth.pack_weights(cfg, synth.make_weights(cfg, 0))


def test_reference_arm_line_on_the_tiny_workload():
    """`bench.py --impl reference` prints one JSON line with the contract's keys;
    the oracle sample never holds more streams than the workload has."""
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32",
                          "--steps", "2", "--warmup", "3", "--ref-steps", "2"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["unit"] == "audio-s/s" and d["value"] > 0
    assert d["steps"] == 2 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "tiny_fp32" and d["config"]["streams_sampled"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "audio-s/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # audio counted: one stream x 2 pushes of 160 ms in the timed steps
    assert d["value"] == pytest.approx(1 * 2 * 0.16 / (d["ms_per_step"] * 2 / 1e3), rel=1e-6)


def test_oracle_sample_is_clamped_to_the_workload_and_memory():
    blob = np.zeros(1000, dtype=np.float32)
    assert bench.oracle_workers(blob, 1) == 1
    assert 1 <= bench.oracle_workers(blob, 10 ** 6) <= bench.cpu_cores()
    huge = np.zeros(1, dtype=np.float32)
    huge = np.lib.stride_tricks.as_strided(huge, shape=(1 << 46,), strides=(0,))  # 2^46 floats, no memory
    assert bench.oracle_workers(huge, 64) == 1


def test_workload_mel_is_the_gpu_legs_stream():
    wl = WORKLOADS["tiny_fp32"]
    m = bench.workload_mel(wl, 0)
    assert m.shape == (320, 128)
    assert np.array_equal(m, synth.make_mels_parallel(320, [0], wl.silence_frac, workers=1)[0])


@pytest.mark.parametrize("kind", ["streaming", "provisional", "offline"])
def test_cpu_baseline_forms(kind):
    """cpu_baseline times the oracle form the workload runs: chunked streaming
    pushes, provisional-tail pushes (the right-context encoder, 320 ms), or
    offline encodes of whole windows; one worker per stream or window of the
    sample, audio counted per push or window."""
    base = WORKLOADS["tiny_fp32"]
    if kind == "streaming":
        wl = replace(base, streams=3)
    elif kind == "provisional":
        wl = replace(base, model=replace(TINY, right_context=3, emit_frames=4, lookahead_frames=8),
                     streams=2, push_mel=32)
    else:
        wl = replace(base, offline_batch=2, offline_mel=96)
    cb = bench.cpu_baseline(wl, _tiny_blob(wl.model), 2)
    units = wl.offline_batch or wl.streams
    assert cb["kind"] == "oracle" and cb["unit"] == "audio-s/s" and cb["value"] > 0
    assert 1 <= cb["cores"] <= units
    assert cb["single_core"]["cores"] == 1 and cb["single_core"]["value"] > 0
    assert ("windows" in cb["sample"]) == (kind == "offline")
    if kind == "provisional":
        assert "320 ms" in cb["sample"]
