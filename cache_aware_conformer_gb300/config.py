"""Model and workload configurations of the cache-aware Conformer encoder step.

Plain data only.  The five workloads are the streaming Parakeet-EOU shapes
(17 layers, hidden 512, attention context 70: "Parakeet-EOU-120M — Streaming ASR
Model", §Config table), the chunked-causal mask with chunk 2 and left context 70
and the 14-mel-frame subsampling tail ("True streaming encode — implementation
spec", §Why this is provably correct and §State), the 600M-class offline window
of 1501 mel frames -> 188 encoder frames with a 640-wide joint projection
("Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon", §1.3), and the
right-context-3 provisional-tail variant ("True streaming encode", §Status,
Nemotron variant).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

DTYPE_F32 = "fp32"
DTYPE_BF16 = "bf16"

MEL_BINS = 128
SUB_FACTOR = 8            # three stride-2 convolutions
MEL_TAIL = 14             # 2 + 2*2 + 4*2 mel frames of causal left context
MEL_PER_FRAME = 8         # mel frames per subsampled frame
FRAME_SEC = 0.08          # 8 mel frames at a 10 ms hop


@dataclass(frozen=True)
class ModelConfig:
    n_layers: int
    d_model: int
    n_heads: int
    ff_dim: int
    dw_kernel: int = 9
    att_left: int = 70
    att_chunk: int = 2
    mel_bins: int = MEL_BINS
    joint_dim: int = 640
    dtype: str = DTYPE_BF16
    # provisional-tail variant: window mask [p - att_left, p + right_context];
    # each pass computes emit_frames + lookahead_frames frames and emits emit_frames.
    right_context: int = 0
    emit_frames: int = 0
    lookahead_frames: int = 0

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_heads

    @property
    def provisional(self) -> bool:
        return self.right_context > 0


@dataclass(frozen=True)
class Workload:
    name: str
    model: ModelConfig
    streams: int = 1
    seconds: float = 30.0
    push_mel: int = 16            # mel frames per push (160 ms)
    offline_batch: int = 0        # >0: offline chunked-causal encode of this many windows
    offline_mel: int = 0          # mel frames per offline window
    reset_prob: float = 0.0
    max_start_offset: int = 0     # start offsets drawn on 0..max_start_offset-1, rounded down to even
    silence_frac: float = 0.2
    extra: dict = field(default_factory=dict)


TINY = ModelConfig(n_layers=2, d_model=64, n_heads=4, ff_dim=256, dtype=DTYPE_F32)
EOU_120M = ModelConfig(n_layers=17, d_model=512, n_heads=8, ff_dim=2048)
C600M = ModelConfig(n_layers=24, d_model=1024, n_heads=16, ff_dim=4096)
EOU_RC3 = replace(EOU_120M, right_context=3, emit_frames=4, lookahead_frames=16)

WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", TINY, streams=1, seconds=3.2, push_mel=16),
    "eou120m_1stream_30s": Workload("eou120m_1stream_30s", EOU_120M, streams=1, seconds=30.0),
    "eou120m_256streams_60s": Workload(
        "eou120m_256streams_60s", EOU_120M, streams=256, seconds=60.0,
        reset_prob=0.01, max_start_offset=500),
    "c600m_offline_32x15s": Workload(
        "c600m_offline_32x15s", C600M, offline_batch=32, offline_mel=1501),
    "c600m_64streams_30s": Workload("c600m_64streams_30s", C600M, streams=64, seconds=30.0),
    "eou120m_rc3_128streams_30s": Workload(
        "eou120m_rc3_128streams_30s", EOU_RC3, streams=128, seconds=30.0, push_mel=32),
}


@dataclass(frozen=True)
class DecoderConfig:
    """Greedy RNN-T decoder with an end-of-utterance class: an LSTM predictor
    over the last emitted token, a joint ReLU(enc_proj + pred_proj) -> logits
    over vocab + blank + EOU, argmax per decision.  Ids: tokens 0 .. vocab-1,
    blank = vocab, eou = vocab + 1."""
    vocab: int = 1024
    pred_dim: int = 640           # LSTM hidden / embedding width
    joint_dim: int = 640          # width of both projections into the joint
    max_symbols: int = 10         # emissions per encoder frame before forcing a blank
    blank_bias: float = 3.4       # synthetic init: offset on the blank bias (about 0.3 emissions per frame)

    @property
    def blank(self) -> int:
        return self.vocab

    @property
    def eou(self) -> int:
        return self.vocab + 1

    @property
    def classes(self) -> int:
        return self.vocab + 2


EOU_DECODER = DecoderConfig()
TINY_DECODER = DecoderConfig(vocab=30, pred_dim=64, joint_dim=64, max_symbols=3)


def subsampled_len(t_mel: int) -> int:
    """Encoder frames produced from t_mel mel frames: ceil(.) three times."""
    t = t_mel
    for _ in range(3):
        t = (t + 1) // 2
    return t
