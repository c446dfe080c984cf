"""The give-up path of the kernels' bounded device waits, made to run out on
purpose with no fault: each wait polls something that never happens (a
grid-barrier counter target no CTA reaches, an mbarrier phase with no arrival)
with a short poll limit.  The wait must give up, leave TFL_E_DEVICE in the
status word and return, and the model must then run a normal decode step that
gives the same bits as before."""
import pytest
import torch

from gqa_decoder_forward_gb300 import synth, tfl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

TINY = synth.TINY


@pytest.fixture(scope="module")
def model():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gqa_decoder_forward_gb300 import build
    build.build()
    w = gu.gpu_weights(TINY, 1)
    return tfl.Model(TINY, w, max_rows=64, max_decode_rows=16, max_context=256)


def _step(m, kv, ids, rows):
    kv.reset(40)
    lg = torch.empty((rows, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.decode_step([kv], ids[40:40 + rows].contiguous(), [rows], lg)
    return lg


@pytest.mark.parametrize("which", [0, 1])
def test_wait_that_runs_out_reports_device_status_and_model_recovers(model, which):
    m = model
    ids = synth.uniform_ids(3, 64, TINY.vocab, "cuda")
    kv = m.kv(128)
    m.prefill_chunk(kv, ids[:40].contiguous())
    before = {r: _step(m, kv, ids, r) for r in (1, 3)}   # persistent (1 row) and per-launch (3 rows)
    assert m.status() == tfl.TFL_OK
    tfl.tfl_wait_probe(m, which, 10000)
    assert m.status() == tfl.TFL_E_DEVICE
    assert m.status() == tfl.TFL_OK            # read and cleared
    for r, lg in before.items():
        again = _step(m, kv, ids, r)
        assert m.status() == tfl.TFL_OK
        assert torch.equal(again.view(torch.int16), lg.view(torch.int16)), r


def test_wait_probe_arguments_are_checked(model):
    for which, limit in ((2, 100), (-1, 100), (0, 0), (1, (1 << 20) + 1)):
        with pytest.raises(tfl.TflError) as e:
            tfl.tfl_wait_probe(model, which, limit)
        assert e.value.code == tfl.TFL_E_ARG
