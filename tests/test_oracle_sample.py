"""Pins of the oracle's seeded sampler against closed forms (no GPU).

Reading pinned (the pages name a GPU draw beside argmax and the release's
recommended temperature / top-p / top-k settings, but fix no algorithm):
candidates = ids whose logit is at least the k-th largest (ties included);
weights exp((z - z_max) / T); nucleus = values from the largest down until the
running mass reaches p of the candidates' mass (ties at the cut included);
draw = smallest id whose running weight, in id order over the nucleus, exceeds
u times the nucleus mass.
"""
import math

import numpy as np
import pytest


def _bits(x: float) -> int:
    """bf16 bit pattern of x rounded to nearest even (through fp32, exact for these inputs)."""
    b = int(np.array([x], np.float32).view(np.uint32)[0])
    if (b & 0x7F800000) == 0x7F800000:
        return b >> 16 | (0x40 if b & 0x7FFFFF else 0)
    return (b + 0x7FFF + ((b >> 16) & 1)) >> 16


def _val(bits: int) -> float:
    return float(np.array([bits << 16], np.uint32).view(np.float32)[0])


def _row(values):
    """bf16 bit patterns of a row (values rounded to bf16)."""
    return np.array([_bits(x) for x in values], np.uint16)[None, :]


def bf16_bits(x):
    return _bits(x)


def test_uniform_logits_give_floor_u_times_v(orc):
    V = 1000
    z = np.full((1, V), bf16_bits(0.5), np.uint16)
    for u in (0.0, 0.0004, 0.1234, 0.5, 0.77777, 0.9995):
        ids, st = orc.sample(z, 0.6, 0, 1.0, [u])
        assert st == 0 and ids[0] == math.floor(u * V), u


def test_top_k_one_and_tiny_p_are_argmax_or_split_a_tie(orc):
    rng = np.random.default_rng(1)
    z = (rng.standard_normal((4, 300)) * 2).astype(np.float64)
    z[2, 17] = z[2, 200] = z[2].max() + 1.0          # a tie for the maximum
    rows = np.concatenate([_row(r) for r in z])
    ref, _ = orc.argmax(rows)
    assert ref[2] == 17
    for u in (0.0, 0.3, 0.999):
        for k, p in ((1, 1.0), (0, 1e-9), (5, 1e-9)):
            ids, st = orc.sample(rows, 0.8, k, p, [u] * 4)
            want = ref.copy()
            want[2] = 17 if u < 0.5 else 200   # ties at the cut are kept: the two maxima share it
            assert st == 0 and np.array_equal(ids, want), (u, k, p)


def test_two_candidates_follow_the_logistic_probability(orc):
    # ids 3 and 11 hold the only non-negligible logits
    for a, b, T in ((1.0, 0.0, 1.0), (0.5, 1.25, 0.6), (-2.0, -2.0, 0.3)):
        vals = [-1e4] * 16
        vals[3], vals[11] = a, b
        z = _row(vals)
        av, bv = _val(_bits(a)), _val(_bits(b))
        p3 = 1.0 / (1.0 + math.exp((bv - av) / T))
        for u, want in ((p3 - 1e-6, 3), (p3 + 1e-6, 11), (0.0, 3), (0.999999, 11)):
            ids, _ = orc.sample(z, T, 0, 1.0, [u])
            assert ids[0] == want, (a, b, T, u)


def test_nucleus_cut_and_renormalised_draw(orc):
    # probabilities at T = 1: softmax of (ln 5, ln 3, ln 2) = (0.5, 0.3, 0.2), placed
    # at ids 7 (0.3), 2 (0.2) and 9 (0.5) so that id order differs from value order
    lg = {7: math.log(3.0), 2: math.log(2.0), 9: math.log(5.0)}
    vals = [-1e4] * 12
    for i, v in lg.items():
        vals[i] = v
    z = _row(vals)
    w = {i: math.exp(_val(_bits(v))) for i, v in lg.items()}         # the bf16 values
    # p = 0.6: nucleus {9, 7} (0.5 < 0.6, 0.5 + 0.3 >= 0.6); id order 7, 9
    mass = w[9] + w[7]
    cut = w[7] / mass
    for u, want in ((cut - 1e-6, 7), (cut + 1e-6, 9)):
        ids, _ = orc.sample(z, 1.0, 0, 0.6, [u])
        assert ids[0] == want, u
    # p = 0.45 keeps only id 9; p = 1 keeps all three, id order 2, 7, 9
    assert orc.sample(z, 1.0, 0, 0.45, [0.0])[0][0] == 9
    assert orc.sample(z, 1.0, 0, 0.45, [0.99])[0][0] == 9
    tot = w[2] + w[7] + w[9]
    for u, want in ((w[2] / tot - 1e-6, 2), (w[2] / tot + 1e-6, 7), ((w[2] + w[7]) / tot + 1e-6, 9)):
        assert orc.sample(z, 1.0, 0, 1.0, [u])[0][0] == want, u


def test_top_k_includes_ties_at_the_kth_value(orc):
    vals = [0.0] * 8
    vals[5], vals[1], vals[6] = 3.0, 2.0, 2.0   # k = 2: the 2nd largest value 2.0 is held twice
    z = _row(vals)
    seen = {int(orc.sample(z, 1.0, 2, 1.0, [u])[0][0]) for u in np.linspace(0, 0.999, 200)}
    assert seen == {1, 5, 6}
    seen3 = {int(orc.sample(z, 1.0, 3, 1.0, [u])[0][0]) for u in np.linspace(0, 0.999, 200)}
    assert seen3 == {1, 5, 6}                    # k = 3 gives the same three
    seen1 = {int(orc.sample(z, 1.0, 1, 1.0, [u])[0][0]) for u in np.linspace(0, 0.999, 50)}
    assert seen1 == {5}


def test_u_grid_reproduces_the_probabilities(orc):
    """A deterministic grid of u values (midpoints of N cells) lands on each id a
    number of times within one of N times its probability (inverse CDF)."""
    rng = np.random.default_rng(3)
    V, N, T, p = 40, 20000, 0.7, 0.9
    z = _row(list(rng.standard_normal(V) * 1.5))
    zz = np.array([_val(int(b)) for b in z[0]])
    w = np.exp((zz - zz.max()) / T)
    order = np.argsort(-zz, kind="stable")
    run = np.cumsum(w[order])
    m = int(np.searchsorted(run, p * w.sum()))      # first index with run >= p * total
    keep = zz >= zz[order[m]]
    pk = np.where(keep, w, 0.0)
    pk /= pk.sum()
    us = (np.arange(N) + 0.5) / N
    ids, st = orc.sample(np.repeat(z, N, 0), T, 0, p, us)
    counts = np.bincount(ids, minlength=V)
    assert st == 0 and counts.sum() == N
    assert np.all(np.abs(counts - N * pk) <= 1.0 + 1e-9), np.max(np.abs(counts - N * pk))
    assert np.all(counts[~keep] == 0)


def test_nonfinite_rows_are_refused(orc):
    z = np.concatenate([_row([0.0, 1.0, 2.0]), _row([0.0, float("nan"), 2.0]), _row([float("inf"), 0.0, 0.0])])
    ids, st = orc.sample(z, 0.6, 0, 0.95, [0.5, 0.5, 0.5])
    assert st == -1 and ids[1] == -1 and ids[2] == -1 and 0 <= ids[0] <= 2


@pytest.mark.parametrize("T", [0.05, 100.0])
def test_temperature_limits(orc, T):
    vals = [0.0, 0.5, 1.0, 0.25]
    z = _row(vals)
    got = [int(orc.sample(z, T, 0, 1.0, [u])[0][0]) for u in (0.1, 0.35, 0.6, 0.85)]
    if T < 1:
        assert got == [2, 2, 2, 2]                  # cold: the maximum
    else:
        assert got == [0, 1, 2, 3]                  # hot: close to uniform, inverse CDF in id order
