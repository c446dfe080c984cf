"""Oracle model-level pins: composition of the pinned primitives, the invariants the
pages require of any implementation (one-row steps == windows, resumed == fresh),
and the geometry figures the pages print (CPU only)."""
import os

import numpy as np
import pytest

from gqa_decoder_forward_gb300 import synth
from tests import _ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# A small model of the same family (GQA 4 q / 2 KV heads, head 128) for fast CPU tests.
SMALL = synth.ModelShape(hidden=256, layers=2, n_q=4, n_kv=2, head_dim=128, ffn=384, vocab=512)


def _np_weights(shape, seed, **kw):
    w = synth.model_weights(shape, seed, "cpu", **kw)
    out = {k: synth.bits(w[k]) for k in ("embed", "final_norm", "lm_head")}
    for k in synth.LAYER_KEYS:
        out[k] = [synth.bits(t) for t in w[k]]
    return out


def _model(orc, shape, seed, max_pos, **kw):
    c = orc.Config(shape.hidden, shape.layers, shape.n_q, shape.n_kv, shape.head_dim, shape.ffn,
                   shape.vocab, shape.rope_theta, shape.rms_eps)
    return orc.Model(c, _np_weights(shape, seed, **kw), max_pos)


@pytest.fixture(scope="module")
def small_weights():
    return _np_weights(SMALL, 3)


def _mk(orc, weights, max_pos=64):
    s = SMALL
    c = orc.Config(s.hidden, s.layers, s.n_q, s.n_kv, s.head_dim, s.ffn, s.vocab, s.rope_theta, s.rms_eps)
    return orc.Model(c, weights, max_pos)


def test_layer_composition_matches_pinned_primitives(orc, small_weights):
    """orc_layer == rmsnorm -> q,k,v -> rope -> cache -> attention -> o -> add -> norm ->
    gate/up -> swiglu -> down -> add, composed here from the separately pinned parts."""
    m = _mk(orc, small_weights)
    s = SMALL
    w = small_weights
    ids = synth.uniform_ids(4, 6, s.vocab).numpy()
    pos = np.arange(6, dtype=np.int32)
    _, trace = m.forward(ids, pos, want_logits=False, want_trace=True)
    h = w["embed"][ids]
    assert np.array_equal(trace[0], h)
    c, sn = orc.rope_table(s.rope_theta, s.head_dim, 6)
    K = np.zeros((6, s.n_kv, s.head_dim), np.uint16)
    V = np.zeros_like(K)
    for l in range(s.layers):
        xn = orc.rmsnorm(h, w["attn_norm"][l], s.rms_eps)
        q = orc.linear(w["wq"][l], xn).reshape(6, s.n_q, s.head_dim)
        k = orc.linear(w["wk"][l], xn).reshape(6, s.n_kv, s.head_dim)
        v = orc.linear(w["wv"][l], xn).reshape(6, s.n_kv, s.head_dim)
        q = orc.rope_apply(q, pos, c, sn)
        K[:] = orc.rope_apply(k, pos, c, sn)
        V[:] = v
        assert np.array_equal(m.K[l, :6], K) and np.array_equal(m.V[l, :6], V)
        o = orc.attention(q, pos, K, V)
        h = orc.residual_add(h, orc.linear(w["wo"][l], o))
        xn = orc.rmsnorm(h, w["ffn_norm"][l], s.rms_eps)
        a = orc.swiglu(orc.linear(w["wg"][l], xn), orc.linear(w["wu"][l], xn))
        h = orc.residual_add(h, orc.linear(w["wd"][l], a))
        assert np.array_equal(trace[l + 1], h), l
    logits = m.head(h)
    assert np.array_equal(logits, orc.linear(w["lm_head"], orc.rmsnorm(h, w["final_norm"], s.rms_eps)))


def test_zero_output_projections_make_layers_identity(orc, small_weights):
    w = dict(small_weights)
    w["wo"] = [np.zeros_like(a) for a in w["wo"]]
    w["wd"] = [np.zeros_like(a) for a in w["wd"]]
    m = _mk(orc, w)
    ids = np.array([5, 9, 11], np.int32)
    _, trace = m.forward(ids, np.arange(3, dtype=np.int32), want_logits=False, want_trace=True)
    for l in range(SMALL.layers + 1):
        assert np.array_equal(trace[l] & 0x7FFF, w["embed"][ids] & 0x7FFF)


def test_one_row_steps_equal_windows(orc, small_weights):
    ids = synth.uniform_ids(5, 24, SMALL.vocab).numpy()
    # prompt of 8, then a 16-row window vs 16 one-row steps
    a = _mk(orc, small_weights)
    a.forward(ids[:8], np.arange(8, dtype=np.int32))
    la, _ = a.forward(ids[8:], np.arange(8, 24, dtype=np.int32))
    b = _mk(orc, small_weights)
    b.forward(ids[:8], np.arange(8, dtype=np.int32))
    lb = np.concatenate([b.forward(ids[i:i + 1], np.array([i], np.int32))[0] for i in range(8, 24)])
    assert np.array_equal(la, lb)
    assert np.array_equal(a.K, b.K) and np.array_equal(a.V, b.V)


def test_resumed_equals_fresh(orc, small_weights):
    ids = synth.uniform_ids(6, 30, SMALL.vocab).numpy()
    fresh = _mk(orc, small_weights)
    lf, _ = fresh.forward(ids, np.arange(30, dtype=np.int32))
    res = _mk(orc, small_weights)
    res.forward(ids[:13], np.arange(13, dtype=np.int32))
    # a kept prefix of 9 positions; the rest is recomputed from position 9
    res.K[:, 9:] = 0x7FC0
    res.V[:, 9:] = 0x7FC0
    lr, _ = res.forward(ids[9:], np.arange(9, 30, dtype=np.int32))
    assert np.array_equal(lr, lf[9:])


def test_window_rows_do_not_see_later_rows(orc, small_weights):
    ids = synth.uniform_ids(7, 10, SMALL.vocab).numpy()
    a = _mk(orc, small_weights)
    la, _ = a.forward(ids, np.arange(10, dtype=np.int32))
    ids2 = ids.copy()
    ids2[6:] = (ids2[6:] + 1) % SMALL.vocab
    b = _mk(orc, small_weights)
    lb, _ = b.forward(ids2, np.arange(10, dtype=np.int32))
    assert np.array_equal(la[:6], lb[:6])
    assert not np.array_equal(la[6], lb[6])


def test_tiny_model_greedy_is_deterministic_and_finite(orc):
    m = _model(orc, synth.TINY, 1, 96)
    ids = synth.uniform_ids(2, 64, synth.TINY.vocab).numpy()
    logits, _ = m.forward(ids, np.arange(64, dtype=np.int32))
    g, st = orc.argmax(logits)
    assert st == 0 and np.all((g >= 0) & (g < synth.TINY.vocab))
    v = _ref.bf16_to_float(logits)
    assert np.all(np.isfinite(v)) and v.std() > 0


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = float(v)
    return out


def test_33b_geometry_matches_the_pages():
    g = _golden("geometry_33b.txt")
    m = synth.NANBEIGE_33B
    for k in ("hidden", "layers", "n_q", "n_kv", "head_dim", "ffn", "vocab"):
        assert getattr(m, k) == g[k], k
    assert m.rope_theta == g["rope_theta"]
    per_layer = sum(int(np.prod(s)) for s in synth.layer_tensor_shapes(m).values())
    params = m.layers * per_layer + 2 * m.vocab * m.hidden + m.hidden
    assert params == g["params"]
    assert round(params * 2 / 2 ** 30, 1) == g["release_gib"]
    kv = m.layers * 2 * m.n_kv * m.head_dim * 2
    assert kv == g["kv_bytes_per_token"]
    assert kv * 16384 / 2 ** 30 == g["kv_gib_16k"]
    assert kv * 32768 / 2 ** 30 == g["kv_gib_32k"]
    assert kv * 65536 / 2 ** 30 == g["kv_gib_64k"]
