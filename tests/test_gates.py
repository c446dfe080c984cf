"""The comparison gates of the GPU tests, checked on the CPU with the oracle: a
1-ulp change at any internal rounding point of a fused op stays inside the
rounding-point bound, and a larger planted change is caught."""
import numpy as np
import pytest

from gqa_decoder_forward_gb300 import synth
from tests import gpu_util as gu

S = synth.ModelShape(hidden=512, layers=1, n_q=4, n_kv=2, head_dim=128, ffn=768, vocab=256)


def _bump(bits, frac, seed, k=1):
    r = np.random.default_rng(seed)
    b = bits.copy().ravel()
    idx = r.choice(b.size, max(1, int(frac * b.size)), replace=False)
    b[idx] = (b[idx].astype(np.int32) + k * r.choice([-1, 1], idx.size)).astype(np.uint16)
    return b.reshape(bits.shape)


@pytest.fixture(scope="module")
def chain(orc):
    hw = {k: [synth.bits(synth.layer_weight(S, 5, 0, k))] for k in synth.LAYER_KEYS}
    K, V = synth.kv_contents(S, 6, 0, 40)
    h = synth.bits(synth.hidden_rows(S, 7, 3, std=1.0))
    pos = np.arange(40, 43, dtype=np.int32)
    return hw, gu.oracle_chain(orc, S, hw, 0, h, pos, synth.bits(K), synth.bits(V))


def test_swiglu_bound_covers_one_ulp_at_g_and_u(orc, chain):
    _, ch = chain
    b = gu.bound_swiglu(ch["g"], ch["u"], ch["sg"], ch["a"])
    for seed in range(4):
        a2 = orc.swiglu(_bump(ch["g"], 0.2, seed), _bump(ch["u"], 0.2, seed + 10))
        gu.assert_bound_gate(a2, ch["a"], b, "swiglu")
    with pytest.raises(AssertionError):
        gu.assert_bound_gate(orc.swiglu(_bump(ch["g"], 0.3, 1, k=8), ch["u"]), ch["a"], b)


def test_rope_bound_covers_one_ulp_at_the_projection(orc, chain):
    _, ch = chain
    c, s = orc.rope_table(S.rope_theta, 128, 43)
    pos = np.arange(40, 43, dtype=np.int32)
    b = gu.bound_rope(ch["qp"], ch["cos"], ch["sin"], ch["q"])
    for seed in range(4):
        q2 = orc.rope_apply(_bump(ch["qp"], 0.3, seed), pos, c, s)
        gu.assert_bound_gate(q2, ch["q"], b, "rope")
    with pytest.raises(AssertionError):
        gu.assert_bound_gate(orc.rope_apply(_bump(ch["qp"], 0.3, 2, k=16), pos, c, s), ch["q"], b)


def test_residual_and_norm_bounds(orc, chain):
    hw, ch = chain
    b = gu.bound_residual(ch["yo"], ch["h1"])
    gu.assert_bound_gate(orc.residual_add(ch["h_in"], _bump(ch["yo"], 0.3, 3)), ch["h1"], b, "residual")
    with pytest.raises(AssertionError):
        gu.assert_bound_gate(orc.residual_add(ch["h_in"], _bump(ch["yo"], 0.3, 3, k=8)), ch["h1"], b)
    bn = gu.bound_norm(ch["y2"], hw["ffn_norm"][0], ch["xn2"])
    y2 = _bump(ch["y2"], 0.3, 4)
    xn2 = orc.bf16_round(gu.bf16_to_f64(hw["ffn_norm"][0]) * gu.bf16_to_f64(y2))
    gu.assert_bound_gate(xn2, ch["xn2"], bn, "norm")


def test_plain_gate_catches_two_ulp_drift():
    x = synth.bits(synth.normal_bf16(1, 1, (5000,), 1.0))
    gu.assert_hidden_gate(_bump(x, 0.5, 1), x)
    with pytest.raises(AssertionError):
        gu.assert_hidden_gate(_bump(x, 0.01, 1, k=2), x)
    with pytest.raises(AssertionError):
        y = x.copy()
        y[7] = (int(y[7]) + 5) & 0xFFFF
        gu.assert_hidden_gate(y, x)
