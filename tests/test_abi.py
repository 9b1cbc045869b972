"""Host-side checks of the C-ABI library: it builds, loads without a GPU, and
exports every function include/cac.h declares; host-only calls agree with the
weight-layout generator."""
import os
import re
import subprocess

import pytest

from cache_aware_conformer_gb300 import synth
from cache_aware_conformer_gb300.config import TINY, EOU_120M, C600M, EOU_RC3

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    from cache_aware_conformer_gb300 import native as nat
    if not os.path.exists(nat.LIB_PATH):
        from cache_aware_conformer_gb300 import build
        build.build()
    return nat


def declared_functions():
    text = "".join(open(os.path.join(ROOT, "include", h)).read() for h in ("cac.h", "cac_ops.h", "cac_decode.h", "cac_frontend.h", "cac_beam.h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cac_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("cac_model_create", "cac_pool_create", "cac_stream_push", "cac_stream_flush",
                 "cac_stream_reset", "cac_encode_offline", "cac_stream_get_state"):
        assert must in names


def test_library_exports_every_declared_symbol(native):
    out = subprocess.run(["nm", "-D", "--defined-only", native.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (cac_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    assert set(native.SYMBOLS) == set(declared_functions())
    lib = native.lib()
    for n in declared_functions():
        assert getattr(lib, n) is not None


@pytest.mark.parametrize("cfg", [TINY, EOU_120M, C600M, EOU_RC3])
def test_weights_size_matches_layout(native, cfg):
    assert native.weights_size(cfg) == synth.weights_size(cfg)


def test_invalid_config_has_no_size(native):
    from dataclasses import replace
    assert native.weights_size(replace(TINY, n_heads=3)) == 0       # d_model % n_heads != 0
    assert native.lib().cac_strerror(-2).decode().startswith("push not aligned")


def test_decoder_blob_layout_matches_the_header():
    """include/cac_decode.h: emb [C][P], w_ih, w_hh [4P][P], b_ih, b_hh [4P],
    pred.w [J][P], pred.b [J], out.w [C][J], out.b [C]; C = vocab + 2."""
    from cache_aware_conformer_gb300.config import EOU_DECODER, TINY_DECODER
    for dc in (TINY_DECODER, EOU_DECODER):
        C, P, J = dc.vocab + 2, dc.pred_dim, dc.joint_dim
        names = [n for n, _, _ in synth.decoder_layout(dc)]
        assert names == ["emb", "lstm.w_ih", "lstm.w_hh", "lstm.b_ih", "lstm.b_hh", "pred.w", "pred.b",
                         "out.w", "out.b"]
        blob = synth.pack_decoder_weights(dc, synth.make_decoder_weights(dc, 0))
        assert blob.size == C * P + 2 * 4 * P * P + 2 * 4 * P + J * P + J + C * J + C
        assert (dc.blank, dc.eou, dc.classes) == (dc.vocab, dc.vocab + 1, C)
        assert P % 64 == 0 and J % 64 == 0  # the kernel's tiling rule (CAC_E_UNSUPPORTED otherwise)
