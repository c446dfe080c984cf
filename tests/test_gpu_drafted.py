"""Drafted greedy decode (tfl_decode_drafted) on the GPU: the ids equal plain
greedy one-row steps whatever the proposer guesses (copy drafts, a smaller
random-init drafter, a drafter that always guesses right), and the served
model's cache ends bit-identical to the plain run's."""
import numpy as np
import pytest
import torch

from gqa_decoder_forward_gb300 import synth, tfl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

TINY = synth.TINY
TINY1 = TINY.with_layers(1)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gqa_decoder_forward_gb300 import build
    build.build()
    tfl.lib()


@pytest.fixture(scope="module")
def weights():
    return gu.gpu_weights(TINY, 1), gu.gpu_weights(TINY1, 5)


def _model(shape, w):
    return tfl.Model(shape, w, max_rows=256, max_decode_rows=64, max_context=512)


def _prefilled(m, prompt, keep):
    kv = m.kv(m.cfg.max_context)
    m.prefill_chunk(kv, torch.tensor(prompt[:keep], dtype=torch.int32, device="cuda"))
    return kv


def plain_greedy(m, kv, pending, n):
    V = m.shape.vocab
    ids = torch.tensor([pending], dtype=torch.int32, device="cuda")
    logits = torch.empty((1, V), dtype=torch.bfloat16, device="cuda")
    out = torch.empty(n, dtype=torch.int32, device="cuda")
    for t in range(n):
        m.decode_step([kv], ids if t == 0 else out[t - 1:t], [1], logits)
        m.argmax(logits, out[t:t + 1])
    return out.cpu().numpy()


def _same_cache(a, b, n, layers):
    for l in range(layers):
        ka, va = a.read(l, 0, n)
        kb, vb = b.read(l, 0, n)
        assert torch.equal(ka.view(torch.int16), kb.view(torch.int16)), l
        assert torch.equal(va.view(torch.int16), vb.view(torch.int16)), l


PROMPT = [int(x) for x in synth.uniform_ids(61, 80, TINY.vocab, "cpu")]


@pytest.fixture(scope="module")
def plain(weights):
    w, _ = weights
    m = _model(TINY, w)
    kv = _prefilled(m, PROMPT, len(PROMPT) - 1)
    ids = plain_greedy(m, kv, PROMPT[-1], 52)
    assert m.status() == tfl.TFL_OK
    kv.reset(len(PROMPT) - 1 + 48)
    return m, kv, ids


@pytest.mark.parametrize("proposer", ["copy", "drafter", "self", "lagging"])
@pytest.mark.parametrize("k", [1, 3, 7, 15])
def test_drafted_equals_plain_tiny(weights, plain, proposer, k):
    w, wd = weights
    pm, pkv, ref = plain
    m = _model(TINY, w)
    kv = _prefilled(m, PROMPT, len(PROMPT) - 1)
    drafter = dkv = None
    if proposer in ("drafter", "lagging"):
        drafter = _model(TINY1, wd)
        dkv = _prefilled(drafter, PROMPT, len(PROMPT) - (1 if proposer == "drafter" else 9))
    elif proposer == "self":            # the same weights: every guess is right
        drafter = _model(TINY, w)
        dkv = _prefilled(drafter, PROMPT, len(PROMPT) - 1)
    ids, st = m.decode_drafted(kv, PROMPT, 48, k, drafter, dkv)
    assert np.array_equal(ids, ref[:48]), (proposer, k, ids, ref[:48])
    assert kv.length == len(PROMPT) - 1 + 48
    _same_cache(kv, pkv, kv.length, TINY.layers)
    assert st["target_rows"] == st["rounds"] + st["drafted"]
    assert st["rounds"] + st["accepted"] == 48 and 0 <= st["accepted"] <= st["drafted"]
    if proposer == "self":
        assert st["accepted"] == st["drafted"] and st["rounds"] == -(-48 // (k + 1))
    if drafter is not None:
        assert dkv.length <= kv.length
        assert drafter.status() == tfl.TFL_OK
    assert m.status() == tfl.TFL_OK


def test_drafted_resumes_where_it_stopped(weights, plain):
    """Drafted calls of 20 and 28 tokens with a drafter, then 4 with copy drafts,
    equal one plain run of 52."""
    w, wd = weights
    _, _, ref = plain
    m = _model(TINY, w)
    kv = _prefilled(m, PROMPT, len(PROMPT) - 1)
    d = _model(TINY1, wd)
    dkv = _prefilled(d, PROMPT, len(PROMPT) - 1)
    a, _ = m.decode_drafted(kv, PROMPT, 20, 5, d, dkv)
    b, _ = m.decode_drafted(kv, PROMPT + list(a), 28, 5, d, dkv)
    assert np.array_equal(np.concatenate([a, b]), ref[:48])
    c, _ = m.decode_drafted(kv, PROMPT + list(a) + list(b), 4, 3)
    assert np.array_equal(c, ref[48:])


def test_drafted_nonfinite_logits_stop_with_the_ids_so_far(weights):
    w, _ = weights
    bad = dict(w)
    bad["final_norm"] = torch.full_like(w["final_norm"], float("nan"))
    m = _model(TINY, bad)
    kv = _prefilled(m, PROMPT, len(PROMPT) - 1)
    with pytest.raises(tfl.TflError) as e:
        m.decode_drafted(kv, PROMPT, 8, 3)
    assert e.value.code == tfl.TFL_E_NONFINITE
    assert np.all(e.value.ids == -1) and e.value.stats["rounds"] == 1
    assert kv.length == len(PROMPT)
    assert m.status() == tfl.TFL_E_NONFINITE


def test_drafted_arguments_are_checked(weights):
    w, wd = weights
    m = _model(TINY, w)
    kv = _prefilled(m, PROMPT, len(PROMPT) - 1)
    d = _model(TINY1, wd)
    dkv = _prefilled(d, PROMPT, len(PROMPT) - 1)
    cases = [
        dict(context=PROMPT[:-1], n=4, k=3),                    # length(kv) != n_context - 1
        dict(context=PROMPT, n=4, k=0),                         # draft_len < 1
        dict(context=PROMPT, n=4, k=16),                        # draft_len > 15
        dict(context=PROMPT, n=0, k=3),                         # n_tokens < 1
        dict(context=PROMPT[:-1] + [TINY.vocab], n=4, k=3),     # an id outside the vocabulary
    ]
    for c in cases:
        with pytest.raises(tfl.TflError) as e:
            m.decode_drafted(kv, c["context"], c["n"], c["k"])
        assert e.value.code == tfl.TFL_E_ARG, c
    with pytest.raises(tfl.TflError) as e:
        m.decode_drafted(kv, PROMPT, 512, 3)                    # the cache cannot hold the reply
    assert e.value.code == tfl.TFL_E_CAPACITY
    far = _prefilled(d, PROMPT, len(PROMPT) - 20)               # the drafter lags 20 > 16 tokens
    with pytest.raises(tfl.TflError) as e:
        m.decode_drafted(kv, PROMPT, 4, 3, d, far)
    assert e.value.code == tfl.TFL_E_ARG
    with pytest.raises(tfl.TflError) as e:
        m.decode_drafted(kv, PROMPT, 4, 3, m, kv)               # drafting for itself
    assert e.value.code == tfl.TFL_E_ARG
    with pytest.raises(tfl.TflError) as e:
        m.decode_drafted(kv, PROMPT, 4, 3, d, kv)               # a cache of another model
    assert e.value.code == tfl.TFL_E_ARG
    assert kv.length == len(PROMPT) - 1 and dkv.length == len(PROMPT) - 1   # nothing ran


L2 = synth.NANBEIGE_33B.with_layers(2)
L1 = synth.NANBEIGE_33B.with_layers(1)


def test_drafted_equals_plain_33b_vocab():
    """A two-layer model of the 33B shape (166,912 ids) with a one-layer drafter
    and with copy drafts: ids and cache equal the plain run."""
    w, wd = gu.gpu_weights(L2, 11), gu.gpu_weights(L1, 12)
    prompt = [int(x) for x in synth.uniform_ids(62, 100, L2.vocab, "cpu")]
    mk = lambda s, ww: tfl.Model(s, ww, max_rows=128, max_decode_rows=16, max_context=256)
    m = mk(L2, w)
    pkv = _prefilled(m, prompt, len(prompt) - 1)
    ref = plain_greedy(m, pkv, prompt[-1], 24)
    d = mk(L1, wd)
    for drafter in (None, d):
        kv = _prefilled(m, prompt, len(prompt) - 1)
        dkv = _prefilled(d, prompt, len(prompt) - 1) if drafter else None
        ids, st = m.decode_drafted(kv, prompt, 24, 7, drafter, dkv)
        assert np.array_equal(ids, ref), (drafter, ids, ref)
        _same_cache(kv, pkv, kv.length, L2.layers)
        assert st["rounds"] + st["accepted"] == 24
    assert m.status() == tfl.TFL_OK and d.status() == tfl.TFL_OK
