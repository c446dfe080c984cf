"""The persistent decode-step launch (one or two rows) against the launch-per-
operation path: logits and appended keys/values bit-identical."""
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


def _run(m, shape, prompts, feed, steps, persistent, seeded=None):
    m.set_persistent(persistent)
    kvs = []
    for s, p in enumerate(prompts):
        kv = m.kv(m_cap(m))
        if seeded is not None:
            K, V = seeded
            kv.write(0, 0, K, V)
            kv.reset(K.shape[0])
        else:
            m.prefill_chunk(kv, p)
        kvs.append(kv)
    outs = []
    for t in range(steps):
        ids = torch.stack([feed[s][t] for s in range(len(prompts))]).contiguous()
        lg = torch.empty((len(prompts), shape.vocab), dtype=torch.bfloat16, device="cuda")
        m.decode_step(kvs, ids, [1] * len(prompts), lg)
        outs.append(lg)
    assert m.status() == tfl.TFL_OK
    cache = [kv.read(l, 0, kv.length) for kv in kvs for l in range(shape.layers)]
    m.set_persistent(True)
    return outs, cache


def m_cap(m):
    return m._cap


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("streams", [1, 2])
def test_persistent_equals_per_op_tiny(streams):
    w = gu.gpu_weights(TINY, 1)
    m = tfl.Model(TINY, w, max_context=512, max_rows=256)
    m._cap = 512
    prompts = [synth.uniform_ids(60 + s, 130 + 77 * s, TINY.vocab, "cuda") for s in range(streams)]
    feed = [synth.uniform_ids(70 + s, 5, TINY.vocab, "cuda") for s in range(streams)]
    a_out, a_kv = _run(m, TINY, prompts, feed, 5, True)
    b_out, b_kv = _run(m, TINY, prompts, feed, 5, False)
    for x, y in zip(a_out, b_out):
        assert _same(x, y)
    for (ka, va), (kb, vb) in zip(a_kv, b_kv):
        assert _same(ka, kb) and _same(va, vb)


@pytest.fixture(scope="module")
def model33():
    # a whole one-layer model: a decode step gathers embedding rows and runs the
    # head, so the embedding table and lm_head must be full size here
    return gu.gpu_weights(L1, 11)


@pytest.mark.parametrize("streams", [1, 2])
def test_persistent_equals_per_op_33b_layer(model33, streams):
    w = model33
    K, V = synth.kv_contents(L1, 12, 0, 4095, "cuda")
    m = tfl.Model(L1, w, max_decode_rows=16, max_rows=16, max_context=4224)
    m._cap = 4224
    prompts = [None] * streams
    feed = [synth.uniform_ids(80 + s, 3, L1.vocab, "cuda") for s in range(streams)]
    a_out, a_kv = _run(m, L1, prompts, feed, 3, True, seeded=(K, V))
    b_out, b_kv = _run(m, L1, prompts, feed, 3, False, seeded=(K, V))
    for x, y in zip(a_out, b_out):
        assert _same(x, y)
        assert bool(torch.isfinite(x.float()).all())
    for (ka, va), (kb, vb) in zip(a_kv, b_kv):
        assert _same(ka, kb) and _same(va, vb)


def test_persistent_bad_token_raises_status():
    w = gu.gpu_weights(TINY, 1)
    m = tfl.Model(TINY, w, max_context=256, max_rows=64)
    kv = m.kv(64)
    m.prefill_chunk(kv, synth.uniform_ids(3, 10, TINY.vocab, "cuda"))
    lg = torch.empty((1, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.decode_step([kv], torch.tensor([TINY.vocab + 5], dtype=torch.int32, device="cuda"), [1], lg)
    assert m.status() == tfl.TFL_E_ARG
    assert kv.length == 11


def test_step_phases_are_reported_for_a_profiled_step():
    w = gu.gpu_weights(TINY, 1)
    m = tfl.Model(TINY, w, max_context=256, max_rows=64)
    kv = m.kv(128)
    m.prefill_chunk(kv, synth.uniform_ids(4, 40, TINY.vocab, "cuda"))
    lg = torch.empty((1, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    tfl.tfl_profile(m, True)
    m.decode_step([kv], synth.uniform_ids(5, 1, TINY.vocab, "cuda"), [1], lg)
    ph = tfl.tfl_step_phases(m)
    tfl.tfl_profile(m, False)
    assert set(ph) == set(tfl.STEP_PHASES)
    assert all(v >= 0 for v in ph.values())
    per_layer = sum(ph[k] for k in ("qkv", "attention", "merge", "o", "gate_up", "down"))
    assert 0 < per_layer * TINY.layers + ph["head"] <= ph["total"] * 1.001
    with pytest.raises(tfl.TflError):   # read once per profiled step
        tfl.tfl_step_phases(m)
