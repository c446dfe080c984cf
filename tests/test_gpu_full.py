"""Full-size parity: the 52-layer 33B-shaped model (random-init bf16, 61.7 GiB),
in the launch configuration the benchmark times (one stream, decode rows), against
the oracle's 52-layer forward over a seeded cache (teacher-forced, at every depth
of a sweep), plus the bit-exact invariants: one-row steps == windows and
concurrent == solo, at 16 streams x 8,192 and 2 streams x 131,072 positions."""
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


DEPTHS = (1, 2, 4, 8, 16, 52)
TF_POSITIONS = 64


def _fidelity(ref, got):
    """KL(ref || got) mean over positions, max |delta logit|, and top-1 agreement
    under the pages' near-tie rule (a differing winner counts as agreeing when
    both sides' two contenders are within one bf16 step)."""
    fr, fg = gu.bf16_to_f64(ref), gu.bf16_to_f64(got)
    tr, tg = fr.argmax(-1), fg.argmax(-1)
    agree = [bool(tr[i] == tg[i] or (gu.near_tie(ref[i], tr[i], tg[i]) and gu.near_tie(got[i], tr[i], tg[i])))
             for i in range(len(tr))]
    return {"kl": gu.kl_mean(ref, got), "max": float(np.abs(fr - fg).max()), "top1": float(np.mean(agree)),
            "misses": int(len(agree) - sum(agree))}


def test_full_model_teacher_forced_depth_sweep(orc, full):
    """Teacher-forced fidelity of the 52-layer model and of its 1/2/4/8/16-layer
    truncations (the same weights) against the oracle: 64 consecutive positions
    of one seeded id sequence after a seeded 4,096-position cache, decoded by the
    GPU as one-row persistent steps (the benchmark's launch configuration) and by
    the oracle as one causal window.  Random N(0, 0.02) weights make the stack
    amplify rounding-level differences, so each depth is judged against the
    floor of the method itself: the oracle with its projection sums taken in
    fp32 in increasing k order (the literal "fp32 sums rounded once", a second
    faithful implementation) against the same oracle in double.  The GPU must
    stay within 1.5x of that floor's KL and max |delta logit| at every depth and
    lose at most two more top-1 positions (near-tie rule) than it; where the
    floor is at the pages' own figures (depths 1 and 2) the GPU must reach top-1
    >= 99% and, at depth 1, mean KL <= 1e-4.  The residual stream after the
    last layer of each depth is judged the same way: relative rms difference
    within 1.5x of the floor's, and the share of elements within 1 bf16 ulp at
    least 0.8x the floor's."""
    w, _, kvK, kvV = full
    V = FULL.vocab
    cap = CTX + TF_POSITIONS + 8
    ids = synth.uniform_ids(26, TF_POSITIONS, V, "cuda")
    gpu, gpu_h = {}, {}
    emb = w["embed"][ids.long()].contiguous()        # the rows' embeddings (the residual stream's start)
    for d in DEPTHS:
        wd = {k: w[k] for k in ("embed", "final_norm", "lm_head")}
        for k in synth.LAYER_KEYS:
            wd[k] = w[k][:d]
        m = tfl.Model(FULL.with_layers(d), wd, max_rows=64, max_decode_rows=16, max_context=cap)
        kv = m.kv(cap)
        for l in range(d):
            kv.write(l, 0, kvK[l], kvV[l])
        kv.reset(CTX)
        lg = torch.empty((TF_POSITIONS, V), dtype=torch.bfloat16, device="cuda")
        for t in range(TF_POSITIONS):
            m.decode_step([kv], ids[t:t + 1].contiguous(), [1], lg[t:t + 1])
        assert m.status() == tfl.TFL_OK
        gpu[d] = synth.bits(lg)
        kv = m.kv(cap)
        for l in range(d):
            kv.write(l, 0, kvK[l], kvV[l])
        kv.reset(CTX)
        hid = torch.empty_like(emb)
        for t in range(TF_POSITIONS):
            tfl.tfl_decode_hidden(m, [kv], [1], emb[t:t + 1], hid[t:t + 1])
        gpu_h[d] = synth.bits(hid)
        del m, kv, lg, hid
    hw = gu.host_weights(w)
    om = gu.oracle_model(orc, FULL, hw, cap)
    for l in range(FULL.layers):
        om.K[l, :CTX] = synth.bits(kvK[l])
        om.V[l, :CTX] = synth.bits(kvV[l])
    pos = np.arange(CTX, CTX + TF_POSITIONS, dtype=np.int32)
    idn = ids.cpu().numpy()
    _, tr = om.forward(idn, pos, want_logits=False, want_trace=True)
    ref = {d: om.head(tr[d]) for d in DEPTHS}
    with orc.fp32_sums():
        _, tr32 = om.forward(idn, pos, want_logits=False, want_trace=True)
        floor = {d: om.head(tr32[d]) for d in DEPTHS}
    for d in DEPTHS:
        g, f = _fidelity(ref[d], gpu[d]), _fidelity(ref[d], floor[d])
        print(f"depth {d:2d}: GPU KL {g['kl']:.3e} max {g['max']:.4f} top-1 {g['top1']:.4f} | fp32-sum oracle "
              f"KL {f['kl']:.3e} max {f['max']:.4f} top-1 {f['top1']:.4f}")
        assert g["kl"] <= 1.5 * f["kl"], (d, g, f)
        assert g["max"] <= 1.5 * f["max"], (d, g, f)
        assert g["misses"] <= f["misses"] + 2, (d, g, f)
        if d <= 2:
            assert g["top1"] >= 0.99, (d, g)
        if d == 1:
            assert g["kl"] <= 1e-4, g
        # the residual stream after d layers
        gr, fr = gu.rel_rms(gpu_h[d], tr[d]), gu.rel_rms(tr32[d], tr[d])
        gq = float(np.mean(gu.ulp_dist(gpu_h[d], tr[d]) <= 1))
        fq = float(np.mean(gu.ulp_dist(tr32[d], tr[d]) <= 1))
        print(f"          hidden: GPU rel rms {gr:.4f}, within 1 ulp {gq:.3f} | fp32-sum oracle {fr:.4f}, {fq:.3f}")
        assert gr <= 1.5 * fr, (d, gr, fr)
        assert gq >= 0.8 * fq, (d, gq, fq)


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


def _seeded_caches(model, n_pos, cap, lengths, seed=22):
    """Caches of the full model holding the seeded keys and values of n_pos
    positions in every layer, with the given lengths."""
    kvs = [model.kv(cap) for _ in lengths]
    for l in range(FULL.layers):
        K, V = synth.kv_contents(FULL, seed, l, n_pos, "cuda")
        for kv in kvs:
            kv.write(l, 0, K, V)
        del K, V
    for kv, n in zip(kvs, lengths):
        kv.reset(n)
    return kvs


def _greedy_concurrent_equals_solo(model, kvs, lengths, steps, first_ids):
    """steps greedy decode steps of all streams together (one row each), then of
    each stream alone from the same state: logits and ids equal bit for bit."""
    S = len(kvs)
    V = FULL.vocab
    ids = first_ids.clone()
    batched = []
    for _ in range(steps):
        lg = torch.empty((S, V), dtype=torch.bfloat16, device="cuda")
        model.decode_step(kvs, ids, [1] * S, lg)
        model.argmax(lg, ids)
        batched.append((lg, ids.clone()))
    assert model.status() == tfl.TFL_OK
    for s in range(S):
        kvs[s].reset(lengths[s])
        cur = first_ids[s:s + 1].clone()
        for t in range(steps):
            lg = torch.empty((1, V), dtype=torch.bfloat16, device="cuda")
            model.decode_step([kvs[s]], cur, [1], lg)
            model.argmax(lg, cur)
            assert torch.equal(lg.view(torch.int16), batched[t][0][s:s + 1].view(torch.int16)), (s, t)
            assert int(cur.item()) == int(batched[t][1][s].item()), (s, t)
    assert model.status() == tfl.TFL_OK


def test_full_model_16_streams_at_8k_equal_solo(full):
    """Sixteen streams of one row each at 8,192 - 97 s positions (6,737..8,192:
    14 to 17 units of 512 keys), three greedy steps together (the launch per
    operation with the TMA-fed attention over 16 one-row streams) against each
    stream alone (the persistent step): bit-equal logits and ids."""
    w, _, _, _ = full
    n_pos = 8192
    m = tfl.Model(FULL, w, max_rows=64, max_decode_rows=16, max_context=n_pos + 64)
    lengths = [n_pos - 97 * s for s in range(16)]
    kvs = _seeded_caches(m, n_pos, n_pos + 64, lengths)
    _greedy_concurrent_equals_solo(m, kvs, lengths, 3, synth.uniform_ids(41, 16, FULL.vocab, "cuda"))


def test_full_model_2_streams_at_131k_equal_solo(full):
    """Two streams at 131,072 and 130,995 positions (55.8 GB of keys and values),
    three greedy steps together (one persistent launch for both rows) against
    each alone: bit-equal logits and ids."""
    w, _, _, _ = full
    n_pos = 131072
    m = tfl.Model(FULL, w, max_rows=64, max_decode_rows=16, max_context=n_pos + 16)
    lengths = [n_pos, n_pos - 77]
    kvs = _seeded_caches(m, n_pos, n_pos + 16, lengths)
    _greedy_concurrent_equals_solo(m, kvs, lengths, 3, synth.uniform_ids(42, 2, FULL.vocab, "cuda"))
    del kvs
    torch.cuda.empty_cache()
