"""Shared helpers for the GPU parity tests: model construction and metrics."""
import numpy as np

from cache_aware_conformer_gb300 import synth

BF16_MAX_ABS = 3e-2     # bf16 mode: max |delta| on encoder frames
BF16_MIN_COS = 0.999    # bf16 mode: cosine similarity on encoder frames
F32_MAX_ABS = 1e-4      # fp32 mode


def max_abs(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.abs(a - b).max()) if a.size else 0.0


def cosine(a, b):
    a, b = np.asarray(a, np.float64).ravel(), np.asarray(b, np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))


def assert_close(gpu, ref, cfg, what=""):
    """The tolerance the workload states: fp32 1e-4; bf16 3e-2 and cosine 0.999."""
    d = max_abs(gpu, ref)
    print(f"[parity] {what}: max|d| {d:.3e} cos {cosine(gpu, ref):.7f} ({cfg.dtype})")
    if cfg.dtype == "fp32":
        assert d <= F32_MAX_ABS, f"{what}: max|d| {d:.3e} > {F32_MAX_ABS}"
    else:
        c = cosine(gpu, ref)
        assert d <= BF16_MAX_ABS and c >= BF16_MIN_COS, f"{what}: max|d| {d:.3e}, cos {c:.6f}"
    return d


def make_model(cfg, seed=0, gemm_simt=False):
    from cache_aware_conformer_gb300 import native
    W = synth.make_weights(cfg, seed)
    return W, native.Model(cfg, synth.pack_weights(cfg, W), gemm_simt=gemm_simt)
