"""Full-size parity: the 52-layer 33B-shaped model (random-init bf16, 61.7 GiB),
in the launch configuration the benchmark times (one stream, decode rows), against
the oracle's own 52-layer forward over a seeded cache, plus bit-exact invariants."""
import numpy as np
import pytest
import torch

from gqa_decoder_forward_gb300 import synth, tfl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

FULL = synth.NANBEIGE_33B
CTX = 4096
CAP = CTX + 64


@pytest.fixture(scope="module")
def full(orc):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gqa_decoder_forward_gb300 import build
    build.build()
    w = gu.gpu_weights(FULL, 21)
    m = tfl.Model(FULL, w, max_rows=64, max_decode_rows=32, max_context=CAP)
    kvK, kvV = [], []
    for l in range(FULL.layers):
        K, V = synth.kv_contents(FULL, 22, l, CTX, "cuda")
        kvK.append(K)
        kvV.append(V)
    return w, m, kvK, kvV


def _seeded(m, kvK, kvV):
    kv = m.kv(CAP)
    for l in range(FULL.layers):
        kv.write(l, 0, kvK[l], kvV[l])
    kv.reset(CTX)
    return kv


def _bump(bits, frac, seed):
    r = np.random.default_rng(seed)
    b = bits.copy().ravel()
    idx = r.choice(b.size, max(1, int(frac * b.size)), replace=False)
    b[idx] = (b[idx].astype(np.int32) + r.choice([-1, 1], idx.size)).astype(np.uint16)
    return b.reshape(bits.shape)


def test_full_model_decode_logits_at_the_oracles_noise_floor(orc, full):
    """One decode row of the 52-layer model against the oracle's 52-layer forward.
    Random N(0, 0.02) weights make the stack amplify rounding-level differences,
    so the yardstick is the oracle's own divergence when one rounding point (the
    residual stream after layer 0) moves by 1 ulp in 1% of its elements: the GPU
    path must stay within 3x of that floor, which a real defect exceeds by orders
    of magnitude."""
    w, m, kvK, kvV = full
    hw = gu.host_weights(w)
    om = gu.oracle_model(orc, FULL, hw, CAP)
    for l in range(FULL.layers):
        om.K[l, :CTX] = synth.bits(kvK[l])
        om.V[l, :CTX] = synth.bits(kvV[l])
    pos = np.array([CTX], np.int32)
    ids = synth.uniform_ids(23, 2, FULL.vocab, "cuda")
    for i in range(2):
        kv = _seeded(m, kvK, kvV)
        logits = torch.empty((1, FULL.vocab), dtype=torch.bfloat16, device="cuda")
        m.decode_step([kv], ids[i:i + 1].contiguous(), [1], logits)
        nxt = torch.empty(1, dtype=torch.int32, device="cuda")
        m.argmax(logits, nxt)
        assert m.status() == tfl.TFL_OK
        got = synth.bits(logits)

        def run(perturb_seed=None):
            h = hw["embed"][ids[i:i + 1].cpu().numpy()]
            for l in range(FULL.layers):
                h = om.layer(l, h, pos)
                if l == 0 and perturb_seed is not None:
                    h = _bump(h, 0.01, perturb_seed)
            return om.head(h)

        ref = run()
        floors = [run(seed) for seed in (1, 2)]
        kl_floor = max(gu.kl_mean(ref, f) for f in floors)
        err_floor = max(float(np.abs(gu.bf16_to_f64(f) - gu.bf16_to_f64(ref)).max()) for f in floors)
        kl = gu.kl_mean(ref, got)
        err = float(np.abs(gu.bf16_to_f64(got) - gu.bf16_to_f64(ref)).max())
        print(f"row {i}: GPU KL {kl:.3e} max|dlogit| {err:.4f}; oracle 1-ulp floor KL {kl_floor:.3e} "
              f"max|dlogit| {err_floor:.4f}")
        assert kl <= max(1e-4, 3 * kl_floor), (kl, kl_floor)
        assert err <= max(0.05, 3 * err_floor), (err, err_floor)
        rt = int(gu.bf16_to_f64(ref[0]).argmax())
        gt = int(nxt.item())
        assert rt == gt or (gu.near_tie(ref[0], rt, gt) and gu.near_tie(got[0], rt, gt)) or kl_floor > 1e-4


@pytest.mark.parametrize("layer", [0, 25, 51])
def test_full_model_sampled_layers_every_op(orc, full, layer):
    w, m, kvK, kvV = full
    hw = {k: [synth.bits(w[k][layer]) if i == layer else None for i in range(FULL.layers)]
          for k in synth.LAYER_KEYS}
    kv = _seeded(m, kvK, kvV)
    R = 4
    h_in = synth.bits(synth.hidden_rows(FULL, 31 + layer, R, "cuda", std=1.0))
    pos = np.arange(CTX, CTX + R, dtype=np.int32)
    ch = gu.oracle_chain(orc, FULL, hw, layer, h_in, pos, synth.bits(kvK[layer]), synth.bits(kvV[layer]))
    gu.check_ops(tfl, m, kv, layer, ch, CTX)


def test_full_model_steps_equal_windows(full):
    w, m, kvK, kvV = full
    ids = synth.uniform_ids(24, 16, FULL.vocab, "cuda")
    a = _seeded(m, kvK, kvV)
    win = torch.empty((16, FULL.vocab), dtype=torch.bfloat16, device="cuda")
    m.decode_step([a], ids, [16], win)
    b = _seeded(m, kvK, kvV)
    steps = torch.empty_like(win)
    for i in range(16):
        m.decode_step([b], ids[i:i + 1].contiguous(), [1], steps[i:i + 1])
    assert torch.equal(win.view(torch.int16), steps.view(torch.int16))
    for l in (0, 51):
        ka, va = a.read(l, CTX, 16)
        kb, vb = b.read(l, CTX, 16)
        assert torch.equal(ka.view(torch.int16), kb.view(torch.int16))
        assert torch.equal(va.view(torch.int16), vb.view(torch.int16))


def test_full_model_concurrent_equals_solo(full):
    w, m, kvK, kvV = full
    ids = synth.uniform_ids(25, 3, FULL.vocab, "cuda")
    kvs = [_seeded(m, kvK, kvV) for _ in range(2)]
    kvs[1].reset(CTX - 77)       # a second stream at another position
    both = torch.empty((3, FULL.vocab), dtype=torch.bfloat16, device="cuda")
    m.decode_step(kvs, ids, [1, 2], both)
    solo0, solo1 = _seeded(m, kvK, kvV), _seeded(m, kvK, kvV)
    solo1.reset(CTX - 77)
    s0 = torch.empty((1, FULL.vocab), dtype=torch.bfloat16, device="cuda")
    s1 = torch.empty((2, FULL.vocab), dtype=torch.bfloat16, device="cuda")
    m.decode_step([solo0], ids[:1].contiguous(), [1], s0)
    m.decode_step([solo1], ids[1:].contiguous(), [2], s1)
    assert torch.equal(both[:1].view(torch.int16), s0.view(torch.int16))
    assert torch.equal(both[1:].view(torch.int16), s1.view(torch.int16))
