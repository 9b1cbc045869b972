"""Host-side 6-bit palettisation of an encoder's weight matrices, the input of
cac_model_create_palette ("Fast Accuracy-Preserving RNNT Beam Search on Apple
Silicon", §1.3: the encoder keeps every weight matrix as a 64-entry lookup
table plus 6-bit indices; vectors and the depthwise taps stay dense).

A quick table per matrix: the 64 quantiles (i + 1/2) / 64 of the matrix's
entries (of an evenly strided sample of at most 65,536 of them), rounded to
bf16; every entry then takes the nearest table value, ties to the lower
index.  This is a compression tool for users of the library, not an optimal
quantiser: a table from any other method goes through the same entry point.
"""
from __future__ import annotations

import numpy as np

from .config import ModelConfig

N_LEVELS = 64
SAMPLE = 1 << 16


def matrix_names(n_layers: int) -> list[str]:
    """The palettised matrices in the order cac_model_create_palette takes their tables."""
    names = ["sub.w1", "sub.w2", "sub.w3", "sub.wo", "joint.w"]
    for l in range(n_layers):
        p = f"l{l}."
        names += [p + "ff1.w1", p + "ff1.w2", p + "att.wq", p + "att.wk", p + "att.wv", p + "att.wo",
                  p + "att.wpos", p + "conv.w_pw1", p + "conv.w_pw2", p + "ff2.w1", p + "ff2.w2"]
    return names


def to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bf16 (ties to even), as float32."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def palettize(w: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(table [64] float32 of bf16 values, sorted; decoded weights of w's shape)."""
    flat = np.asarray(w, dtype=np.float32).reshape(-1)
    step = max(1, flat.size // SAMPLE)
    q = np.quantile(flat[::step].astype(np.float64), (np.arange(N_LEVELS) + 0.5) / N_LEVELS)
    table = np.sort(to_bf16(q.astype(np.float32)))
    mid = (table[:-1].astype(np.float64) + table[1:]) / 2.0
    idx = np.searchsorted(mid, flat.astype(np.float64), side="left")  # a tie goes to the lower entry
    return table, table[idx].reshape(np.shape(w))


def palettize_model(cfg: ModelConfig, W: dict) -> tuple[dict, np.ndarray]:
    """The weight dict with every palettised matrix replaced by its decoded
    values, and the tables [5 + 11 L][64] in the library's order."""
    out = dict(W)
    tables = []
    for name in matrix_names(cfg.n_layers):
        table, dec = palettize(W[name])
        out[name] = dec
        tables.append(table)
    return out, np.stack(tables).astype(np.float32)
