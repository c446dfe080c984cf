"""GPU parity: libtfl (through the C ABI) against the oracle on the same seeded
inputs, and the GPU path's own bit-exact invariants."""
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


# ---- inputs --------------------------------------------------------------------------

def test_generator_is_device_independent():
    for shape, std, mean in (((4099,), 0.02, 0.0), ((1000,), 0.1, 1.0), ((333, 7), 1.7, 0.0)):
        a = synth.normal_bf16(5, 17, shape, std, "cpu", mean=mean)
        b = synth.normal_bf16(5, 17, shape, std, "cuda", mean=mean).cpu()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(synth.uniform_ids(3, 5000, 166912, "cpu"), synth.uniform_ids(3, 5000, 166912, "cuda").cpu())


# ---- the tiny model, end to end --------------------------------------------------------

@pytest.fixture(scope="module")
def tiny(orc):
    w = gu.gpu_weights(TINY, 1)
    hw = gu.host_weights(w)
    return w, hw


def _tiny_model(w, **kw):
    kw.setdefault("max_context", 256)
    kw.setdefault("max_rows", 256)
    return tfl.Model(TINY, w, **kw)


def test_tiny_prefill_logits_match_oracle(orc, tiny):
    w, hw = tiny
    ids = synth.uniform_ids(2, 64, TINY.vocab, "cuda")
    m = _tiny_model(w)
    kv = m.kv(128)
    logits = torch.empty((64, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.prefill_chunk(kv, ids, logits, all_rows=True)
    assert m.status() == tfl.TFL_OK
    om = gu.oracle_model(orc, TINY, hw, 128)
    ref, _ = om.forward(ids.cpu().numpy(), np.arange(64, dtype=np.int32))
    got = synth.bits(logits)
    err = np.abs(gu.bf16_to_f64(got) - gu.bf16_to_f64(ref)).max()
    assert err <= 0.05, err
    assert gu.kl_mean(ref, got) <= 1e-4
    top_ref = gu.bf16_to_f64(ref).argmax(-1)
    top_got = gu.bf16_to_f64(got).argmax(-1)
    assert np.mean(top_ref == top_got) >= 0.99 or all(
        gu.near_tie(ref[i], top_ref[i], top_got[i]) for i in np.nonzero(top_ref != top_got)[0])
    # layer 0's keys and values come straight from the embedding rows: hidden-state gate
    k, v = kv.read(0, 0, 64)
    gu.assert_hidden_gate(synth.bits(k), om.K[0, :64], "K layer 0")
    gu.assert_hidden_gate(synth.bits(v), om.V[0, :64], "V layer 0")


@pytest.mark.parametrize("R", [1, 5, 16])
def test_tiny_every_op_every_layer(orc, tiny, R):
    """The hidden-state gate (<= 1 ulp for >= 99.9%, <= 4 ulp max) at every
    rounding point of every layer, each kernel fed the oracle's bf16 inputs."""
    w, hw = tiny
    m = _tiny_model(w, max_context=512)
    kv = m.kv(512)
    ids = synth.uniform_ids(2, 300 + R, TINY.vocab, "cuda")
    om = gu.oracle_model(orc, TINY, hw, 512)
    _, trace = om.forward(ids.cpu().numpy(), np.arange(300 + R, dtype=np.int32), want_logits=False,
                          want_trace=True)
    pos = np.arange(300, 300 + R, dtype=np.int32)
    for l in range(TINY.layers):
        kv.write(l, 0, gu.to_torch_bits(om.K[l, :300]), gu.to_torch_bits(om.V[l, :300]))
        ch = gu.oracle_chain(orc, TINY, hw, l, trace[l][300:], pos, om.K[l, :300], om.V[l, :300])
        assert np.array_equal(ch["h2"], trace[l + 1][300:])  # the chain is the oracle's layer
        gu.check_ops(tfl, m, kv, l, ch, 300, head=(orc, hw, TINY) if l == TINY.layers - 1 else None)


def test_tiny_layer_fed_oracle_input(orc, tiny):
    """A whole GPU layer fed the oracle's bf16 layer input: relative rms difference
    of the residual stream within two bf16 steps."""
    w, hw = tiny
    ids = synth.uniform_ids(2, 64, TINY.vocab, "cuda")
    om = gu.oracle_model(orc, TINY, hw, 128)
    _, trace = om.forward(ids.cpu().numpy(), np.arange(64, dtype=np.int32), want_logits=False, want_trace=True)
    for l in range(TINY.layers):
        wl = {k: w[k] for k in ("embed", "final_norm", "lm_head")}
        for k in synth.LAYER_KEYS:
            wl[k] = [w[k][l]]
        m = tfl.Model(TINY.with_layers(1), wl, max_context=256)
        kv = m.kv(128)
        h_in = gu.to_torch_bits(trace[l])
        h_out = torch.empty_like(h_in)
        tfl.tfl_prefill_hidden(m, kv, h_in, h_out)
        err = gu.rel_rms(synth.bits(h_out), trace[l + 1])
        assert err <= gu.LAYER_REL_RMS, (l, err)


def test_tiny_greedy_16_matches_oracle(orc, tiny):
    w, hw = tiny
    ids = synth.uniform_ids(2, 64, TINY.vocab, "cuda")
    m = _tiny_model(w)
    kv = m.kv(128)
    last = torch.empty((1, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.prefill_chunk(kv, ids, last)
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    m.argmax(last, nxt)
    gpu_ids, gpu_rows = [], []
    step_logits = torch.empty((1, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    for i in range(16):
        gpu_ids.append(int(nxt.item()))
        m.decode_step([kv], nxt, [1], step_logits)
        gpu_rows.append(synth.bits(step_logits)[0])
        m.argmax(step_logits, nxt)
    assert m.status() == tfl.TFL_OK

    om = gu.oracle_model(orc, TINY, hw, 128)
    ref_last, _ = om.forward(ids.cpu().numpy(), np.arange(64, dtype=np.int32))
    rid, _ = orc.argmax(ref_last[-1:])
    cur = int(rid[0])
    for i in range(16):
        if cur != gpu_ids[i]:
            # the pages' near-tie rule: both sides' two contenders within one bf16 step
            prev = ref_last[-1] if i == 0 else ref_row
            prev_gpu = synth.bits(last)[0] if i == 0 else gpu_rows[i - 1]
            assert gu.near_tie(prev, cur, gpu_ids[i]), f"greedy step {i}: {cur} vs {gpu_ids[i]} not a near tie"
            assert gu.near_tie(prev_gpu, cur, gpu_ids[i]), f"greedy step {i}: GPU side not a near tie"
            break
        ref_row, _ = om.forward(np.array([cur], np.int32), np.array([64 + i], np.int32))
        ref_row = ref_row[0]
        err = np.abs(gu.bf16_to_f64(gpu_rows[i]) - gu.bf16_to_f64(ref_row)).max()
        assert err <= 0.05, (i, err)
        cur = int(orc.argmax(ref_row[None])[0][0])


# ---- GPU self-invariants (bit-exact) ------------------------------------------------

def _prefix(m, kv, ids):
    m.prefill_chunk(kv, ids)


def test_one_row_steps_equal_windows_tiny(tiny):
    w, _ = tiny
    m = _tiny_model(w)
    ids = synth.uniform_ids(9, 300, TINY.vocab, "cuda")
    for R in (7, 16):
        a = m.kv(256)
        b = m.kv(256)
        _prefix(m, a, ids[:150])
        _prefix(m, b, ids[:150])
        win = torch.empty((R, TINY.vocab), dtype=torch.bfloat16, device="cuda")
        m.decode_step([a], ids[150:150 + R].contiguous(), [R], win)
        steps = torch.empty_like(win)
        for i in range(R):
            m.decode_step([b], ids[150 + i:151 + i].contiguous(), [1], steps[i:i + 1])
        assert torch.equal(win.view(torch.int16), steps.view(torch.int16)), R
        for l in range(TINY.layers):
            ka, va = a.read(l, 0, 150 + R)
            kb, vb = b.read(l, 0, 150 + R)
            assert torch.equal(ka.view(torch.int16), kb.view(torch.int16))
            assert torch.equal(va.view(torch.int16), vb.view(torch.int16))


def test_concurrent_equals_solo_tiny(tiny):
    w, _ = tiny
    m = _tiny_model(w)
    S = 5
    prompts = [synth.uniform_ids(41 + s, 20 + 37 * s, TINY.vocab, "cuda") for s in range(S)]
    rows = [1, 3, 1, 2, 1]
    steps = 4
    # batched
    kvs = [m.kv(256) for _ in range(S)]
    for s in range(S):
        _prefix(m, kvs[s], prompts[s])
    feed = [synth.uniform_ids(90 + s, steps * 3, TINY.vocab, "cuda") for s in range(S)]
    tot = sum(rows)
    batched = []
    for t in range(steps):
        ids = torch.cat([feed[s][t * 3:t * 3 + rows[s]] for s in range(S)]).contiguous()
        lg = torch.empty((tot, TINY.vocab), dtype=torch.bfloat16, device="cuda")
        m.decode_step(kvs, ids, rows, lg)
        batched.append(lg)
    # solo
    for s in range(S):
        kv = m.kv(256)
        _prefix(m, kv, prompts[s])
        off = sum(rows[:s])
        for t in range(steps):
            lg = torch.empty((rows[s], TINY.vocab), dtype=torch.bfloat16, device="cuda")
            m.decode_step([kv], feed[s][t * 3:t * 3 + rows[s]].contiguous(), [rows[s]], lg)
            assert torch.equal(lg.view(torch.int16), batched[t][off:off + rows[s]].view(torch.int16)), (s, t)


def test_resumed_equals_fresh_tiny(tiny):
    w, _ = tiny
    m = _tiny_model(w, max_rows=256)
    ids = synth.uniform_ids(77, 230, TINY.vocab, "cuda")
    fresh = m.kv(256)
    lf = torch.empty((230, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.prefill_chunk(fresh, ids, lf, all_rows=True)
    res = m.kv(256)
    m.prefill_chunk(res, ids[:150])
    res.reset(101)                      # keep a prefix of 101 positions
    lr = torch.empty((129, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.prefill_chunk(res, ids[101:].contiguous(), lr, all_rows=True)
    assert torch.equal(lr.view(torch.int16), lf[101:].view(torch.int16))


# ---- one 33B-shaped layer over a seeded 4,096-position cache ---------------------------

@pytest.fixture(scope="module")
def layer33(orc):
    w = gu.layer_weights(L1, 11)
    hw = gu.host_weights(w)
    K, V = synth.kv_contents(L1, 12, 0, 4096, "cuda")
    return w, hw, K, V


def _seeded(m, K, V, cap):
    kv = m.kv(cap)
    kv.write(0, 0, K, V)
    kv.reset(K.shape[0])
    return kv


@pytest.mark.parametrize("R", [1, 7, 16])
def test_33b_layer_every_op(orc, layer33, R):
    """Hidden-state gate at every rounding point of a 33B-shaped layer, each
    kernel fed the oracle's bf16 inputs, over a seeded 4,096-position cache."""
    w, hw, K, V = layer33
    m = tfl.Model(L1, w, max_decode_rows=16, max_rows=16, max_context=4224)
    kv = _seeded(m, K, V, 4224)
    h_in = synth.bits(synth.hidden_rows(L1, 13, R, "cuda"))
    pos = np.arange(4096, 4096 + R, dtype=np.int32)
    ch = gu.oracle_chain(orc, L1, hw, 0, h_in, pos, synth.bits(K), synth.bits(V))
    gu.check_ops(tfl, m, kv, 0, ch, 4096)


@pytest.mark.parametrize("R", [1, 16])
def test_33b_layer_fed_oracle_input(orc, layer33, R):
    w, hw, K, V = layer33
    m = tfl.Model(L1, w, max_decode_rows=16, max_rows=16, max_context=4224)
    kv = _seeded(m, K, V, 4224)
    h_in = synth.hidden_rows(L1, 13, R, "cuda")
    h_out = torch.empty_like(h_in)
    tfl.tfl_decode_hidden(m, [kv], [R], h_in, h_out)
    om = gu.oracle_model(orc, L1, hw, 4224)
    om.K[0, :4096] = synth.bits(K)
    om.V[0, :4096] = synth.bits(V)
    ref = om.layer(0, synth.bits(h_in), np.arange(4096, 4096 + R, dtype=np.int32))
    err = gu.rel_rms(synth.bits(h_out), ref)
    assert err <= gu.LAYER_REL_RMS, err


@pytest.mark.parametrize("R", [7, 16])
def test_33b_layer_steps_equal_windows(layer33, R):
    w, _, K, V = layer33
    m = tfl.Model(L1, w, max_decode_rows=16, max_rows=16, max_context=4224)
    h_in = synth.hidden_rows(L1, 14, R, "cuda")
    a = _seeded(m, K, V, 4224)
    b = _seeded(m, K, V, 4224)
    win = torch.empty_like(h_in)
    tfl.tfl_decode_hidden(m, [a], [R], h_in, win)
    steps = torch.empty_like(h_in)
    for i in range(R):
        tfl.tfl_decode_hidden(m, [b], [1], h_in[i:i + 1], steps[i:i + 1])
    assert torch.equal(win.view(torch.int16), steps.view(torch.int16))
    ka, va = a.read(0, 4096, R)
    kb, vb = b.read(0, 4096, R)
    assert torch.equal(ka.view(torch.int16), kb.view(torch.int16))
    assert torch.equal(va.view(torch.int16), vb.view(torch.int16))


@pytest.mark.parametrize("rows", [[16, 8], [16, 16], [16, 16, 16]], ids=["24", "32", "48"])
def test_33b_layer_wide_steps_equal_one_row_steps_and_match_oracle(orc, layer33, rows):
    """Steps of 17-64 rows in all (several streams of up to 16 rows, each a causal
    window) run the projections with 32- and 64-row activation boxes (paired
    weight stages up to 32 rows): every stream's rows equal the same rows run as
    one-row steps bit for bit, and every op matches the oracle at that many rows."""
    w, hw, K, V = layer33
    R = sum(rows)
    m = tfl.Model(L1, w, max_decode_rows=64, max_rows=64, max_context=4224)
    h_in = synth.hidden_rows(L1, 17, R, "cuda")
    kvs = [_seeded(m, K, V, 4224) for _ in rows]
    wide = torch.empty_like(h_in)
    tfl.tfl_decode_hidden(m, kvs, rows, h_in, wide)
    r0 = 0
    for n in rows:
        kv = _seeded(m, K, V, 4224)
        for i in range(n):
            one = torch.empty_like(h_in[:1])
            tfl.tfl_decode_hidden(m, [kv], [1], h_in[r0 + i:r0 + i + 1].contiguous(), one)
            assert torch.equal(one.view(torch.int16), wide[r0 + i:r0 + i + 1].view(torch.int16)), (r0, i)
        r0 += n
    kv = _seeded(m, K, V, 4224)
    pos = np.arange(4096, 4096 + R, dtype=np.int32)
    ch = gu.oracle_chain(orc, L1, hw, 0, synth.bits(h_in), pos, synth.bits(K), synth.bits(V))
    gu.check_ops(tfl, m, kv, 0, ch, 4096)


# ---- the prompt-chunk path (tensor-core GEMM projections) -------------------------------

@pytest.mark.parametrize("R", [1, 200])
def test_tiny_prompt_ops_every_layer(orc, tiny, R):
    """Each prompt-chunk op (projections on the tensor-core GEMM over 128-row
    tiles with a ragged tail) fed the oracle's bf16 inputs, gated like the
    decode ops."""
    w, hw = tiny
    m = _tiny_model(w, max_context=512)
    kv = m.kv(512)
    P = 40
    ids = synth.uniform_ids(3, P + R, TINY.vocab, "cuda")
    om = gu.oracle_model(orc, TINY, hw, 512)
    _, trace = om.forward(ids.cpu().numpy(), np.arange(P + R, dtype=np.int32), want_logits=False,
                          want_trace=True)
    pos = np.arange(P, P + R, dtype=np.int32)
    for l in range(TINY.layers):
        kv.write(l, 0, gu.to_torch_bits(om.K[l, :P]), gu.to_torch_bits(om.V[l, :P]))
        ch = gu.oracle_chain(orc, TINY, hw, l, trace[l][P:], pos, om.K[l, :P], om.V[l, :P])
        gu.check_ops(tfl, m, kv, l, ch, P, prompt=True)


def test_33b_prompt_ops(orc, layer33):
    """The prompt ops of a 33B-shaped layer over 130 rows (two 128-row tiles, the
    second ragged) after a seeded 4,096-position cache."""
    w, hw, K, V = layer33
    R = 130
    m = tfl.Model(L1, w, max_decode_rows=16, max_rows=R, max_context=4352)
    kv = _seeded(m, K, V, 4352)
    h_in = synth.bits(synth.hidden_rows(L1, 15, R, "cuda"))
    pos = np.arange(4096, 4096 + R, dtype=np.int32)
    ch = gu.oracle_chain(orc, L1, hw, 0, h_in, pos, synth.bits(K), synth.bits(V))
    gu.check_ops(tfl, m, kv, 0, ch, 4096, prompt=True)


SAMPLED = np.array([0, 1, 127, 128, 1023, 1500, 2047])


def test_33b_full_chunk_projections_sampled(orc, layer33):
    """A full 2,048-row chunk through each prompt GEMM (the launch configuration
    the benchmark times); sampled rows against the oracle, gated as the ops."""
    w, hw, K, V = layer33
    N, H, QD, F, D = 2048, L1.hidden, L1.n_q * 128, L1.ffn, 128
    m = tfl.Model(L1, w, max_decode_rows=64, max_rows=N, max_context=4096 + N)
    kv = _seeded(m, K, V, 4096 + N)
    S = SAMPLED
    pos = 4096 + S.astype(np.int32)
    c, s = orc.rope_table(L1.rope_theta, D, 4096 + N)
    A = gu.abs_bits

    def gate(name, got, ref, bound):
        gu.assert_bound_gate(synth.bits(got)[S].reshape(ref.shape), ref, bound, name)

    # QKV + RoPE, keys/values into the cache
    xn = synth.normal_bf16(21, 0, (N, H), 1.0, "cuda")
    q = torch.empty((N, QD), dtype=torch.bfloat16, device="cuda")
    tfl.tfl_layer_op(m, "qkv_rope", 0, xn, q, kv, 4096, prompt=True)
    x = synth.bits(xn)[S]
    for name, wk, nh in (("q", "wq", L1.n_q), ("k", "wk", L1.n_kv)):
        pre = orc.linear(hw[wk][0], x).reshape(len(S), nh, D)
        pre_abs = orc.linear(A(hw[wk][0]), A(x)).reshape(len(S), nh, D)
        ref = orc.rope_apply(pre, pos, c, s)
        bound = gu.bound_rope(pre, c[pos], s[pos], ref, gu.acc_allowance(pre_abs, H))
        if name == "q":
            gate("q", q, ref, bound)
        else:
            k_got = torch.stack([kv.read(0, int(p), 1)[0][0] for p in pos])
            gu.assert_bound_gate(synth.bits(k_got).reshape(ref.shape), ref, bound, "k")
    v_ref = orc.linear(hw["wv"][0], x).reshape(len(S), L1.n_kv, D)
    v_abs = orc.linear(A(hw["wv"][0]), A(x)).reshape(len(S), L1.n_kv, D)
    v_got = torch.stack([kv.read(0, int(p), 1)[1][0] for p in pos])
    gu.assert_bound_gate(synth.bits(v_got).reshape(v_ref.shape), v_ref,
                         gu.bound_sum(v_ref, gu.acc_allowance(v_abs, H)), "v")

    # o projection + residual, in place
    o = synth.normal_bf16(22, 0, (N, QD), 0.5, "cuda")
    h = synth.hidden_rows(L1, 23, N, "cuda", std=0.5)
    h0 = synth.bits(h)[S]
    tfl.tfl_layer_op(m, "o_residual", 0, o, h, prompt=True)
    yo = orc.linear(hw["wo"][0], synth.bits(o)[S])
    yo_abs = orc.linear(A(hw["wo"][0]), A(synth.bits(o)[S]))
    ref = orc.residual_add(h0, yo)
    gate("o_residual", h, ref, gu.bound_residual(yo, ref, gu.acc_allowance(yo_abs, QD)))

    # gate/up + SwiGLU
    act = torch.empty((N, F), dtype=torch.bfloat16, device="cuda")
    tfl.tfl_layer_op(m, "gate_up", 0, xn, act, prompt=True)
    g = orc.linear(hw["wg"][0], x)
    u = orc.linear(hw["wu"][0], x)
    ref = orc.swiglu(g, u)
    sg = orc.swiglu(g, np.full_like(g, 0x3F80))
    gate("gate_up", act, ref, gu.bound_swiglu(g, u, sg, ref, gu.acc_allowance(orc.linear(A(hw["wg"][0]), A(x)), H),
                                             gu.acc_allowance(orc.linear(A(hw["wu"][0]), A(x)), H)))

    # down projection + residual
    a_in = synth.normal_bf16(24, 0, (N, F), 0.1, "cuda")
    h = synth.hidden_rows(L1, 25, N, "cuda", std=0.5)
    h0 = synth.bits(h)[S]
    tfl.tfl_layer_op(m, "down_residual", 0, a_in, h, prompt=True)
    yd = orc.linear(hw["wd"][0], synth.bits(a_in)[S])
    yd_abs = orc.linear(A(hw["wd"][0]), A(synth.bits(a_in)[S]))
    ref = orc.residual_add(h0, yd)
    gate("down_residual", h, ref, gu.bound_residual(yd, ref, gu.acc_allowance(yd_abs, F)))
    torch.cuda.synchronize()


def test_33b_prompt_chunking_is_bit_exact(layer33):
    """A 2,048-row prompt chunk equals the same rows split into chunks of 700, 1
    and 1,347 rows (row results independent of chunk boundaries and tiles)."""
    w, _, K, V = layer33
    N = 2048
    m = tfl.Model(L1, w, max_decode_rows=64, max_rows=N, max_context=4096 + N)
    h_in = synth.hidden_rows(L1, 16, N, "cuda")
    a = _seeded(m, K, V, 4096 + N)
    whole = torch.empty_like(h_in)
    tfl.tfl_prefill_hidden(m, a, h_in, whole)
    b = _seeded(m, K, V, 4096 + N)
    parts = torch.empty_like(h_in)
    r0 = 0
    for n in (700, 1, 1347):
        tfl.tfl_prefill_hidden(m, b, h_in[r0:r0 + n].contiguous(), parts[r0:r0 + n])
        r0 += n
    assert a.length == b.length == 4096 + N
    assert torch.equal(whole.view(torch.int16), parts.view(torch.int16))
    ka, va = a.read(0, 4096, N)
    kb, vb = b.read(0, 4096, N)
    assert torch.equal(ka.view(torch.int16), kb.view(torch.int16))
    assert torch.equal(va.view(torch.int16), vb.view(torch.int16))
    assert bool(torch.isfinite(whole.float()).all())


def test_prompt_op_arguments_are_checked(tiny):
    w, _ = tiny
    m = _tiny_model(w, max_rows=256)
    x = torch.zeros((257, TINY.hidden), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(tfl.TflError) as e:
        tfl.tfl_layer_op(m, "ffn_norm", 0, x, y, prompt=True)
    assert e.value.code == tfl.TFL_E_ARG
    lg = torch.empty((4, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tfl.TflError) as e:
        tfl.tfl_layer_op(m, "lm_head", 0, x[:4], lg, prompt=True)
    assert e.value.code == tfl.TFL_E_ARG


# ---- argmax, status, capacity ---------------------------------------------------------

def test_argmax_ties_and_nonfinite(orc, tiny):
    w, _ = tiny
    m = _tiny_model(w)
    L = synth.normal_bf16(3, 0, (6, TINY.vocab), 2.0, "cuda")
    L[0, 100] = L[0, 4000] = 64.0
    L[1, 7] = L[1, 6] = 64.0
    ids = torch.empty(6, dtype=torch.int32, device="cuda")
    m.argmax(L, ids)
    assert m.status() == tfl.TFL_OK
    ref, st = orc.argmax(synth.bits(L))
    assert st == 0 and np.array_equal(ids.cpu().numpy(), ref)
    assert ids[0].item() == 100 and ids[1].item() == 6
    for bad in (float("nan"), float("inf"), float("-inf")):
        L2 = L.clone()
        L2[2, 4095] = bad
        m.argmax(L2, ids)
        assert m.status() == tfl.TFL_E_NONFINITE
        assert ids[2].item() == -1 and ids[0].item() == 100
        assert m.status() == tfl.TFL_OK   # the status word was cleared


def test_capacity_is_refused_before_anything_runs(tiny):
    w, _ = tiny
    m = _tiny_model(w)
    kv = m.kv(70)
    ids = synth.uniform_ids(5, 70, TINY.vocab, "cuda")
    m.prefill_chunk(kv, ids[:64].contiguous())
    lg = torch.empty((6, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.decode_step([kv], ids[64:70].contiguous(), [6], lg)
    assert kv.length == 70
    with pytest.raises(tfl.TflError) as e:
        m.decode_step([kv], ids[:1].contiguous(), [1], lg[:1])
    assert e.value.code == tfl.TFL_E_CAPACITY and kv.length == 70
    with pytest.raises(tfl.TflError) as e:
        m.prefill_chunk(kv, ids[:1].contiguous())
    assert e.value.code == tfl.TFL_E_CAPACITY


def test_bad_token_id_raises_status(tiny):
    w, _ = tiny
    m = _tiny_model(w)
    kv = m.kv(16)
    ids = torch.tensor([5, TINY.vocab + 3], dtype=torch.int32, device="cuda")
    m.prefill_chunk(kv, ids)
    assert m.status() == tfl.TFL_E_ARG


def test_long_ragged_context_tiny(orc, tiny):
    """Keys over several 128-position blocks with a ragged last block."""
    w, hw = tiny
    m = _tiny_model(w, max_context=1100)
    kv = m.kv(1100)
    ids = synth.uniform_ids(55, 1003, TINY.vocab, "cuda")
    lg = torch.empty((1, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    for c in range(0, 1000, 64):
        m.prefill_chunk(kv, ids[c:min(1000, c + 64)].contiguous())
    lg3 = torch.empty((3, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.decode_step([kv], ids[1000:1003].contiguous(), [3], lg3)
    om = gu.oracle_model(orc, TINY, hw, 1100)
    ref, _ = om.forward(ids.cpu().numpy(), np.arange(1003, dtype=np.int32))
    got = synth.bits(lg3)
    assert np.abs(gu.bf16_to_f64(got) - gu.bf16_to_f64(ref[1000:])).max() <= 0.05
    assert gu.kl_mean(ref[1000:], got) <= 1e-4


@pytest.mark.parametrize("R", [1, 3, 8, 16])
def test_fused_norm_ops_equal_norm_then_projection(tiny, R):
    """The decode path applies the RMSNorm inside the projection that follows it
    (up to 8 rows); that must give exactly the norm op followed by the projection op."""
    w, _ = tiny
    m = _tiny_model(w, max_context=512)
    H, F, V = TINY.hidden, TINY.ffn, TINY.vocab
    h = synth.normal_bf16(81, 0, (R, H), 0.7, "cuda")
    for layer in range(TINY.layers):
        kv_a, kv_b = m.kv(512), m.kv(512)
        xn = torch.empty_like(h)
        tfl.tfl_layer_op(m, "attn_norm", layer, h, xn)
        q_ref = torch.empty((R, TINY.n_q * 128), dtype=torch.bfloat16, device="cuda")
        tfl.tfl_layer_op(m, "qkv_rope", layer, xn, q_ref, kv_a, 100)
        q = torch.empty_like(q_ref)
        tfl.tfl_layer_op(m, "norm_qkv_rope", layer, h, q, kv_b, 100)
        assert torch.equal(q.view(torch.int16), q_ref.view(torch.int16))
        ka, va = kv_a.read(layer, 100, R)
        kb, vb = kv_b.read(layer, 100, R)
        assert torch.equal(ka.view(torch.int16), kb.view(torch.int16))
        assert torch.equal(va.view(torch.int16), vb.view(torch.int16))

        tfl.tfl_layer_op(m, "ffn_norm", layer, h, xn)
        a_ref = torch.empty((R, F), dtype=torch.bfloat16, device="cuda")
        tfl.tfl_layer_op(m, "gate_up", layer, xn, a_ref)
        a = torch.empty_like(a_ref)
        tfl.tfl_layer_op(m, "norm_gate_up", layer, h, a)
        assert torch.equal(a.view(torch.int16), a_ref.view(torch.int16))
    tfl.tfl_layer_op(m, "final_norm", 0, h, xn)
    l_ref = torch.empty((R, V), dtype=torch.bfloat16, device="cuda")
    tfl.tfl_layer_op(m, "lm_head", 0, xn, l_ref)
    lg = torch.empty_like(l_ref)
    tfl.tfl_layer_op(m, "norm_lm_head", 0, h, lg)
    assert torch.equal(lg.view(torch.int16), l_ref.view(torch.int16))


# ---- prompt cache ---------------------------------------------------------------------

def test_resume_from_prefix_store_equals_fresh(tiny):
    """A prompt whose first 250 tokens sit in a stored cache: copy the prefix,
    prefill the rest, then decode; every logit equals the prompt prefilled fresh."""
    w, _ = tiny
    m = _tiny_model(w, max_rows=512, max_context=512)
    first = synth.uniform_ids(91, 300, TINY.vocab, "cuda")
    second = torch.cat([first[:250], synth.uniform_ids(92, 60, TINY.vocab, "cuda")]).contiguous()
    stored = m.kv(320)
    m.prefill_chunk(stored, first)
    store = tfl.PrefixStore(4)
    store.put(first.cpu().numpy(), stored)
    src, n = store.match(second.cpu().numpy())
    assert src is stored and n == 250
    resumed = m.kv(320)
    tfl.tfl_kv_copy_prefix(m, src, resumed, n)
    assert resumed.length == 250
    lr = torch.empty((60, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.prefill_chunk(resumed, second[250:].contiguous(), lr, all_rows=True)
    fresh = m.kv(320)
    lf = torch.empty((310, TINY.vocab), dtype=torch.bfloat16, device="cuda")
    m.prefill_chunk(fresh, second, lf, all_rows=True)
    assert torch.equal(lr.view(torch.int16), lf[250:].view(torch.int16))
    feed = synth.uniform_ids(93, 4, TINY.vocab, "cuda")
    for t in range(4):
        a = torch.empty((1, TINY.vocab), dtype=torch.bfloat16, device="cuda")
        b = torch.empty_like(a)
        m.decode_step([resumed], feed[t:t + 1].contiguous(), [1], a)
        m.decode_step([fresh], feed[t:t + 1].contiguous(), [1], b)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), t
    with pytest.raises(tfl.TflError):
        tfl.tfl_kv_copy_prefix(m, stored, resumed, 301)   # beyond length(src)


# ---- prompt attention: odd chunk shapes ----------------------------------------------

PATTN_CASES = [(0, 1), (0, 2), (0, 128), (0, 129), (0, 255), (0, 256), (0, 257), (5, 127), (127, 1), (127, 130),
               (300, 200), (383, 384), (640, 300)]


@pytest.fixture(scope="module")
def pattn_tiny(tiny):
    w, _ = tiny
    m = _tiny_model(w, max_rows=512, max_context=1024)
    kv = m.kv(1024)
    K = synth.normal_bf16(81, 0, (1024, TINY.n_kv, 128), 1.0, "cuda")
    V = synth.normal_bf16(82, 0, (1024, TINY.n_kv, 128), 1.0, "cuda")
    kv.write(0, 0, K, V)
    return m, kv, synth.bits(K), synth.bits(V)


@pytest.mark.parametrize("pos0,rows", PATTN_CASES)
def test_prompt_attention_chunk_shapes_tiny(orc, pattn_tiny, pos0, rows):
    """The prompt attention (two 128-row tiles per CTA; tile B empty, partial or
    one key block ahead of tile A) on chunks of odd sizes at odd positions, against
    the oracle's attention over the same cached keys and values."""
    m, kv, Kb, Vb = pattn_tiny
    q = synth.normal_bf16(83, pos0 * 1000 + rows, (rows, TINY.n_q * 128), 1.0, "cuda")
    out = torch.empty_like(q)
    tfl.tfl_layer_op(m, "attention", 0, q, out, kv=kv, pos0=pos0, prompt=True)
    n = pos0 + rows
    qb = synth.bits(q).reshape(rows, TINY.n_q, 128)
    ref = orc.attention(qb, np.arange(pos0, n, dtype=np.int32), Kb[:n], Vb[:n])
    # gate: 1 ulp of the output plus, times sum_t p_t |v_t| (computed in double),
    # the fp32 accumulation allowance sqrt(keys) 2^-24 and the representation
    # error of the weights as bf16 hi + lo, |p - hi - lo| <= 2^-16 p (|p - hi| <= 2^-8 p,
    # then lo = bf16(p - hi) within 2^-8 of p - hi: two roundings to 8 significant bits)
    qf, Kf, Vf = gu.bf16_to_f64(qb), gu.bf16_to_f64(Kb[:n, 0]), gu.bf16_to_f64(Vb[:n, 0])
    absum = np.empty((rows, TINY.n_q, 128))
    for r in range(rows):
        k = pos0 + r + 1
        s = qf[r] @ Kf[:k].T / np.sqrt(128.0)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        absum[r] = (p / p.sum(axis=1, keepdims=True)) @ np.abs(Vf[:k])
    keys = np.arange(pos0 + 1, n + 1, dtype=np.float64)[:, None, None]
    bound = gu.ulp_of(ref).reshape(rows, TINY.n_q, 128) + (np.sqrt(keys) * 2.0 ** -24 + 2.0 ** -16) * absum
    gu.assert_bound_gate(synth.bits(out).reshape(rows, TINY.n_q, 128), ref.reshape(rows, TINY.n_q, 128), bound,
                         f"prompt attention pos0 {pos0} rows {rows}")


def test_prompt_attention_rows_independent_of_chunking(pattn_tiny):
    """Rows 0..383 in one call equal the same rows in calls of 100, 1 and 283."""
    m, kv, _, _ = pattn_tiny
    q = synth.normal_bf16(84, 0, (384, TINY.n_q * 128), 1.0, "cuda")
    whole = torch.empty_like(q)
    tfl.tfl_layer_op(m, "attention", 0, q, whole, kv=kv, pos0=0, prompt=True)
    parts = torch.empty_like(q)
    r0 = 0
    for n in (100, 1, 283):
        o = torch.empty((n, q.shape[1]), dtype=torch.bfloat16, device="cuda")
        tfl.tfl_layer_op(m, "attention", 0, q[r0:r0 + n].contiguous(), o, kv=kv, pos0=r0, prompt=True)
        parts[r0:r0 + n] = o
        r0 += n
    assert torch.equal(whole.view(torch.int16), parts.view(torch.int16))
