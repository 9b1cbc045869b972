"""Oracle: compressed encoder weights — 6-bit palettisation and per-channel int8.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module.  It shares no code with the CUDA library.

Sources:
  * "Fast Accuracy-Preserving RNNT Beam Search on Apple Silicon", §1.3 (table
    and the reverse-engineered facts): the encoders store their weights as
    mixed FP16 and 6-bit palettes — 64-entry lookup tables — while the small
    recurrent decoder and the joint stay dense; the encoder-side joint
    projection is the last operation of the encoder program.
  * "True streaming encode — implementation spec", §Status (the Nemotron
    variant): an int8 encoder.

Readings where the pages are silent (each is listed in the design notes):
  * one 64-entry table per weight matrix: every subsampling conv, the
    subsampling output linear, per layer the FF, Q/K/V/out/position and both
    pointwise-conv matrices, and the encoder-side joint projection.  Vectors
    (biases, LayerNorm and batch-norm affines, positional biases) and the
    depthwise taps stay dense ("mixed");
  * the table is Lloyd's k-means in one dimension over the matrix's entries.
    Initial centres: the quantiles (i + 1/2)/64 of a density proportional to
    the cube root of the entries' histogram (n/64 equal bins for n entries,
    at least 64 and at most 2048), the point
    density of the optimal high-resolution quantiser (Panter and Dite, 1951;
    Bennett's integral) — plain quantiles of the entries converge far more
    slowly on bell-shaped weights.  Then alternate "assign every entry to its
    nearest centre" and "move every centre to the mean of its entries" until
    no assignment changes (at most 300 rounds); a centre that loses all its
    entries stays where it is.  A matrix with at most 64 distinct values
    takes those values as its table (the zero-error optimum, which Lloyd's
    iteration need not find), padded with copies of the largest;
  * table entries are rounded to the stored type (fp16 as on the pages, or
    bf16 for a path whose operands are bf16), and each entry's index is then
    taken against the rounded table: the nearest entry, ties to the lower
    index;
  * packed storage: a row's indices form a little-endian bit stream, index i
    in bits [6 i, 6 i + 6); a row is padded to whole bytes;
  * int8: symmetric per output row, scale = max |w| / 127 (1 for a row of
    zeros), q = w / scale rounded half to even, in [-127, 127]; the weight the
    GEMM sees is q * scale (weights only; activations keep their type).

Parity pins: tests/test_oracle_compress_pins.py (a packed-byte fixture and
round trip; exact reproduction of a matrix with at most 64 distinct values;
nearest-entry assignment by brute force; the k-means objective never
increasing; the uniform distribution's optimal 64-level quantiser (centres
(i + 1/2)/64, error 1/(12 * 64^2)); scikit-learn's KMeans objective on
bell-shaped data; int8 bounds, extremes and half-even ties; which tensors change).
Readings that no page fixes (every function is still pinned above): table
granularity, the k-means initialisation, the packing order and the int8
scheme; only the 64-entry tables are the pages'.
"""
from __future__ import annotations

import numpy as np

N_LEVELS = 64
BITS = 6


def _round_to(v, dtype: str):
    v = np.asarray(v, dtype=np.float64)
    if dtype == "fp16":
        return v.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        # round to nearest even on the upper 16 bits of the fp32 pattern
        b = v.astype(np.float32).view(np.uint32).astype(np.uint64)
        b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
        return b.astype(np.uint32).view(np.float32).astype(np.float64)
    if dtype == "fp64":
        return v
    raise ValueError(dtype)


def nearest_index(values, table):
    """Index of the nearest table entry for every value; ties to the lower index."""
    v = np.asarray(values, dtype=np.float64).reshape(-1, 1)
    d = np.abs(v - np.asarray(table, dtype=np.float64).reshape(1, -1))
    return np.argmin(d, axis=1)  # argmin returns the first minimum


def companded_centres(x, k: int = N_LEVELS):
    """k initial centres at the quantiles (i + 1/2)/k of the cube root of the
    histogram of x (n/64 bins, clipped to 64 .. 2048; linear within a bin)."""
    x = np.asarray(x, dtype=np.float64).reshape(-1)
    bins = int(min(max(x.size // 64, 64), 2048))
    h, edges = np.histogram(x, bins=bins)
    d = np.cbrt(h.astype(np.float64))
    cdf = np.concatenate([[0.0], np.cumsum(d)])
    cdf /= cdf[-1]
    return np.interp((np.arange(k) + 0.5) / k, cdf, edges)


def lloyd_1d(values, k: int = N_LEVELS, max_rounds: int = 300):
    """Lloyd's k-means on scalars from companded initial centres.
    Returns (centres fp64 [k], objective after every round)."""
    x = np.asarray(values, dtype=np.float64).reshape(-1)
    c = companded_centres(x, k)
    assign = nearest_index(x, c)
    history = [float(np.mean((x - c[assign]) ** 2))]
    for _ in range(max_rounds):
        for j in range(k):
            members = x[assign == j]
            if members.size:
                c[j] = members.mean()
        new = nearest_index(x, c)
        history.append(float(np.mean((x - c[new]) ** 2)))
        if np.array_equal(new, assign):
            break
        assign = new
    return c, history


def palettize(w, table_dtype: str = "fp16"):
    """(table [64] fp64 holding values of table_dtype, indices uint8 of w's shape)."""
    w = np.asarray(w, dtype=np.float64)
    distinct = np.unique(w)
    if distinct.size <= N_LEVELS:
        c = np.concatenate([distinct, np.full(N_LEVELS - distinct.size, distinct[-1])])
    else:
        c, _ = lloyd_1d(w.reshape(-1))
    table = _round_to(c, table_dtype)
    idx = nearest_index(w.reshape(-1), table).astype(np.uint8).reshape(w.shape)
    return table, idx


def depalettize(table, idx):
    return np.asarray(table, dtype=np.float64)[np.asarray(idx, dtype=np.int64)]


def pack6(idx):
    """[rows][K] indices < 64 -> [rows][ceil(6 K / 8)] bytes (little-endian bit stream per row)."""
    idx = np.asarray(idx, dtype=np.int64)
    rows, K = idx.shape
    nbytes = (BITS * K + 7) // 8
    out = np.zeros((rows, nbytes), dtype=np.uint8)
    for r in range(rows):
        acc = 0
        for i in range(K):
            acc |= int(idx[r, i]) << (BITS * i)
        out[r] = np.frombuffer(acc.to_bytes(nbytes, "little"), dtype=np.uint8)
    return out


def unpack6(packed, K: int):
    packed = np.asarray(packed, dtype=np.uint8)
    rows = packed.shape[0]
    out = np.zeros((rows, K), dtype=np.uint8)
    for r in range(rows):
        acc = int.from_bytes(packed[r].tobytes(), "little")
        for i in range(K):
            out[r, i] = (acc >> (BITS * i)) & (N_LEVELS - 1)
    return out


def int8_quantize(w):
    """Per output row (axis 0): (q int8 [rows][...], scale fp64 [rows])."""
    w = np.asarray(w, dtype=np.float64)
    flat = w.reshape(w.shape[0], -1)
    m = np.max(np.abs(flat), axis=1)
    scale = np.where(m > 0, m / 127.0, 1.0)
    q = np.clip(np.rint(flat / scale[:, None]), -127, 127).astype(np.int8)  # rint: half to even
    return q.reshape(w.shape), scale


def int8_dequantize(q, scale):
    q = np.asarray(q, dtype=np.float64)
    return (q.reshape(q.shape[0], -1) * np.asarray(scale, dtype=np.float64)[:, None]).reshape(q.shape)


def compressed_names(n_layers: int):
    """The matrices the compressed encoder stores in compressed form."""
    names = ["sub.w1", "sub.w2", "sub.w3", "sub.wo", "joint.w"]
    for l in range(n_layers):
        p = f"l{l}."
        names += [p + "ff1.w1", p + "ff1.w2", p + "att.wq", p + "att.wk", p + "att.wv", p + "att.wo",
                  p + "att.wpos", p + "conv.w_pw1", p + "conv.w_pw2", p + "ff2.w1", p + "ff2.w2"]
    return names


def compress_weights(W: dict, n_layers: int, scheme: str = "palette6", table_dtype: str = "fp16"):
    """A copy of the weight dict with every compressed matrix replaced by what
    its compressed form decodes to (fp64); everything else unchanged.  The
    encoder oracle run on the result is the compressed encoder."""
    out = dict(W)
    for name in compressed_names(n_layers):
        w = np.asarray(W[name], dtype=np.float64)
        if scheme == "palette6":
            table, idx = palettize(w, table_dtype)
            out[name] = depalettize(table, idx)
        elif scheme == "int8":
            q, s = int8_quantize(w)
            out[name] = int8_dequantize(q, s)
        else:
            raise ValueError(scheme)
    return out
