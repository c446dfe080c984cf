"""GPU seeded sampling (tfl_sample) against the oracle's sampler on the same
bf16 logits and the same uniforms: ids equal row by row."""
import numpy as np
import pytest
import torch

from gqa_decoder_forward_gb300 import synth, tfl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

TINY = synth.TINY
L1 = synth.NANBEIGE_33B.with_layers(1)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gqa_decoder_forward_gb300 import build
    build.build()
    tfl.lib()


@pytest.fixture(scope="module")
def tiny_model():
    return tfl.Model(TINY, gu.gpu_weights(TINY, 1), max_context=256, max_rows=64, max_decode_rows=64)


@pytest.fixture(scope="module")
def big_model():
    # sampling reads no weight: a one-layer 33B-shaped model gives the 166,912-id vocabulary
    return tfl.Model(L1, gu.layer_weights(L1, 11), max_context=256, max_rows=16, max_decode_rows=16)


def _uniforms(seed, n):
    # seeded uniforms in [0, 1), exactly representable as float32
    return ((synth.uniform_ids(seed, n, 1 << 24, "cpu").to(torch.float64)) / float(1 << 24)).to(torch.float32)


def _run(m, logits, T, k, p, u):
    ids = torch.empty(logits.shape[0], dtype=torch.int32, device="cuda")
    m.sample(logits, T, k, p, u.cuda(), ids)
    st = m.status()
    return ids.cpu().numpy(), st


SETTINGS = [(0.6, 20, 0.95), (1.0, 0, 0.95), (0.6, 0, 1.0), (1.5, 50, 0.5), (0.3, 1, 1.0), (0.8, 3000, 0.9),
           (2.0, 0, 0.3)]


@pytest.mark.parametrize("T,k,p", SETTINGS)
def test_sample_matches_oracle_tiny_vocab(orc, tiny_model, T, k, p):
    rows = 48
    logits = synth.normal_bf16(70, 1, (rows, TINY.vocab), 2.0, "cuda")
    u = _uniforms(71, rows)
    got, st = _run(tiny_model, logits, T, k, p, u)
    ref, rst = orc.sample(synth.bits(logits), T, k, p, u.double().numpy())
    assert st == tfl.TFL_OK and rst == 0
    assert np.array_equal(got, ref), np.nonzero(got != ref)


@pytest.mark.parametrize("T,k,p", SETTINGS[:4])
def test_sample_matches_oracle_33b_vocab(orc, big_model, T, k, p):
    rows = 16
    logits = synth.normal_bf16(72, 1, (rows, L1.vocab), 1.5, "cuda")
    u = _uniforms(73, rows)
    got, st = _run(big_model, logits, T, k, p, u)
    ref, _ = orc.sample(synth.bits(logits), T, k, p, u.double().numpy())
    assert st == tfl.TFL_OK
    assert np.array_equal(got, ref), np.nonzero(got != ref)


def test_sample_ties_and_u_edges(orc, tiny_model):
    V = TINY.vocab
    base = torch.zeros((8, V), dtype=torch.bfloat16)
    base[:, ::7] = 1.0          # a large tie group
    base[:, 5] = 3.0
    base[:, 4000] = 3.0         # a tie for the maximum
    base[3] = -0.0              # all equal, with signed zeros mixed in
    base[3, ::2] = 0.0
    logits = base.cuda()
    # (u = 0.5 would put the target exactly on a cumulative boundary of this
    # symmetric row, where either side may round either way)
    for u_val in (0.0, 0.3721, 0.9999999):
        u = torch.full((8,), u_val, dtype=torch.float32)
        for T, k, p in ((1.0, 2, 1.0), (1.0, 10, 1.0), (0.5, 0, 0.5), (1.0, 0, 1.0)):
            got, st = _run(tiny_model, logits, T, k, p, u)
            ref, _ = orc.sample(synth.bits(logits), T, k, p, u.double().numpy())
            assert st == tfl.TFL_OK and np.array_equal(got, ref), (u_val, T, k, p, got, ref)


def test_sample_nonfinite_and_determinism(orc, tiny_model):
    logits = synth.normal_bf16(74, 1, (4, TINY.vocab), 2.0, "cuda")
    logits[1, 33] = float("nan")
    logits[2, 0] = float("-inf")
    u = _uniforms(75, 4)
    got, st = _run(tiny_model, logits, 0.7, 20, 0.95, u)
    assert st == tfl.TFL_E_NONFINITE
    assert got[1] == -1 and got[2] == -1 and got[0] >= 0 and got[3] >= 0
    assert tiny_model.status() == tfl.TFL_OK
    ok = logits[[0, 3]].contiguous()
    u03 = u[[0, 3]].contiguous()
    a, _ = _run(tiny_model, ok, 0.7, 20, 0.95, u03)
    b, _ = _run(tiny_model, ok, 0.7, 20, 0.95, u03)
    assert np.array_equal(a, b) and np.array_equal(a, got[[0, 3]])


def test_sample_arguments_are_checked(tiny_model):
    logits = torch.zeros((2, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    u = torch.zeros(2, dtype=torch.float32, device="cuda")
    ids = torch.empty(2, dtype=torch.int32, device="cuda")
    for T, k, p in ((0.0, 0, 1.0), (-1.0, 0, 1.0), (float("inf"), 0, 1.0), (1.0, -1, 1.0), (1.0, 0, 0.0)):
        with pytest.raises(tfl.TflError) as e:
            tiny_model.sample(logits, T, k, p, u, ids)
        assert e.value.code == tfl.TFL_E_ARG


def test_sample_scratch_cycle(orc, big_model):
    """The draw keeps per-value counts in the model's scratch and leaves them zero
    after every call: calls of different row counts and contents in sequence,
    with non-finite rows between them, each equal the oracle."""
    seq = [(16, 80, 1.5, (0.6, 20, 0.95)), (3, 81, 3.0, (1.0, 0, 0.9)), (5, 82, 0.5, (0.7, 50, 1.0)),
           (16, 83, 2.0, (0.9, 0, 0.5))]
    for i, (rows, seed, std, (T, k, p)) in enumerate(seq):
        logits = synth.normal_bf16(seed, 1, (rows, L1.vocab), std, "cuda")
        if i == 2:
            logits[1, 1000] = float("inf")
            logits[4, 7] = float("nan")
        u = _uniforms(seed + 1, rows)
        got, st = _run(big_model, logits, T, k, p, u)
        ref, _ = orc.sample(synth.bits(logits), T, k, p, u.double().numpy())
        if i == 2:
            assert st == tfl.TFL_E_NONFINITE and got[1] == -1 and got[4] == -1
            keep = [0, 2, 3]
            assert np.array_equal(got[keep], ref[keep]), (i, got, ref)
        else:
            assert st == tfl.TFL_OK
            assert np.array_equal(got, ref), (i, np.nonzero(got != ref))
