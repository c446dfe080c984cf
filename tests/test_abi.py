"""The C ABI without a GPU: the library loads, exports every symbol include/tfl.h
declares, and its host-only logic (qualification, sizes, RoPE table) is right."""
import ctypes
import os
import re

import numpy as np
import pytest

from gqa_decoder_forward_gb300 import build, synth, tfl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return tfl.lib()


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(tfl_[a-z_0-9]+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(L):
    declared = _declared_functions()
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(L, name), name
    assert declared == set(tfl.SIGNATURES), "the binding must cover exactly the declared entry points"


def _cfg(shape, **kw):
    return tfl.config(shape, **kw)


def test_qualification_accepts_the_served_geometries(L):
    for shape in (synth.NANBEIGE_33B, synth.NANBEIGE_33B.with_layers(1), synth.TINY, synth.TINY.with_layers(1)):
        code, msg = tfl.tfl_qualify(_cfg(shape))
        assert code == tfl.TFL_OK, msg


@pytest.mark.parametrize("change", [
    dict(hidden=8192), dict(ffn=28672), dict(n_q=64), dict(n_kv=4), dict(vocab=128256),
    dict(rope_theta=5e5), dict(layers=53), dict(head_dim=64), dict(layers=0)])
def test_qualification_refuses_geometry_changes_by_name(L, change):
    c = _cfg(synth.NANBEIGE_33B)
    for k, v in change.items():
        setattr(c, k, v)
    code, msg = tfl.tfl_qualify(c)
    assert code == tfl.TFL_E_GEOMETRY
    assert "refused" in msg


def test_llama31_8b_shape_is_refused(L):
    s = synth.ModelShape(4096, 32, 32, 8, 128, 14336, 128256, 5e5)
    code, msg = tfl.tfl_qualify(_cfg(s))
    assert code == tfl.TFL_E_GEOMETRY and "not a qualified geometry" in msg
    assert tfl.tfl_workspace_bytes(_cfg(s)) == 0


@pytest.mark.parametrize("field,val", [("max_rows", 0), ("max_rows", 2049), ("max_decode_rows", 65),
                                       ("max_context", 0), ("rms_eps", 0.0)])
def test_qualification_refuses_bad_limits(L, field, val):
    c = _cfg(synth.TINY)
    setattr(c, field, val)
    code, _ = tfl.tfl_qualify(c)
    assert code == tfl.TFL_E_ARG


def test_kv_bytes_match_the_pages_208_kib_per_token(L):
    c = _cfg(synth.NANBEIGE_33B)
    per_pos = 52 * 2 * 8 * 128 * 2
    assert per_pos == 212992
    for P in (128, 8192, 131072):
        table = ((P // 128) * 4 + 255) // 256 * 256
        assert tfl.tfl_kv_bytes(c, P) == table + P * per_pos
    # ragged capacity rounds up to whole pages
    assert tfl.tfl_kv_bytes(c, 129) == 256 + 256 * per_pos


def test_workspace_grows_with_limits(L):
    a = tfl.tfl_workspace_bytes(_cfg(synth.TINY, max_context=4096))
    b = tfl.tfl_workspace_bytes(_cfg(synth.TINY, max_context=8192))
    assert 0 < a < b


def test_rope_table_equals_the_oracles_bit_for_bit(L, orc):
    n = 262144   # positions 0 .. 262143, as in the pages' FP64 RoPE test
    c, s = tfl.tfl_rope_table(1.2e8, n)
    oc, os_ = orc.rope_table(1.2e8, 128, n)
    assert np.array_equal(c, oc)
    assert np.array_equal(s, os_)


def test_init_without_a_gpu_fails_cleanly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    c = _cfg(synth.TINY)
    w = tfl.tfl_weights()
    h = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(64)
    code = L.tfl_init(ctypes.byref(c), ctypes.byref(w), ctypes.cast(buf, ctypes.c_void_p), 64, ctypes.byref(h))
    assert code in (tfl.TFL_E_ARG, tfl.TFL_E_CUDA, tfl.TFL_E_WORKSPACE)
    assert L.tfl_last_error()
