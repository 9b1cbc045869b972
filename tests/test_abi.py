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
    text = "".join(open(os.path.join(ROOT, "include", h)).read() for h in ("cac.h", "cac_ops.h", "cac_decode.h"))
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
