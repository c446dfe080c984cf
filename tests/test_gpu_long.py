"""GPU parity at the sizes the kernels really run: decode attention over 131,000
positions and 16-row windows past 16,384 positions (more than 32 units of 512
keys, where the merge leaves its staged path), the prompt attention on full
2,048-row chunks of the 33B shape (G = 7) at the start of the cache and at
129,024 positions, and score patterns whose block maxima keep rising so that
the prompt kernel's lazy rescale of a non-zero output really runs.  Served
contexts reach 131,072 positions (pull request #1415, "Measured"), and the
pages validate "segmented attention over 262144 keys" (NInfer model card,
"Validation")."""
import numpy as np
import pytest
import torch

from gqa_decoder_forward_gb300 import synth, tfl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

L1 = synth.NANBEIGE_33B.with_layers(1)
TINY = synth.TINY
QD = L1.n_q * 128
LONG = 131072


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from gqa_decoder_forward_gb300 import build
    build.build()
    tfl.lib()


def _layer_model(shape, max_context, max_rows=16, max_decode_rows=16):
    """A one-layer model for the attention ops (the ops read only the cache and
    their inputs; the projections are random-init like the other tests)."""
    w = gu.layer_weights(shape, 11)
    return tfl.Model(shape, w, max_rows=max_rows, max_decode_rows=max_decode_rows, max_context=max_context)


@pytest.fixture(scope="module")
def long33():
    """A one-layer model of the 33B shape (with its embedding and lm_head) and a
    seeded cache of 131,072 positions (537 MB)."""
    m = tfl.Model(L1, gu.gpu_weights(L1, 11), max_rows=2048, max_decode_rows=16, max_context=LONG + 64)
    kv = m.kv(LONG + 64)
    K, V = synth.kv_contents(L1, 12, 0, LONG, "cuda")
    kv.write(0, 0, K, V)
    return m, kv, synth.bits(K), synth.bits(V)


def _attn_bound(orc, qb, pos, Kb, Vb, ref):
    """1 ulp of the output plus, times sum_t p_t |v_t|, the fp32 accumulation
    allowance sqrt(keys) 2^-24 and the representation error of the weights as
    bf16 hi + lo (2^-16 relative: |p - hi| <= 2^-8 p, and lo = bf16(p - hi) is
    within 2^-8 of p - hi, two roundings to 8 significant bits)."""
    absum = gu.bf16_to_f64(orc.attention(qb, pos, Kb, gu.abs_bits(Vb)))
    keys = (pos.astype(np.float64) + 1.0)[:, None]
    return gu.ulp_of(ref) + (np.sqrt(keys) * 2.0 ** -24 + 2.0 ** -16) * absum


def _check_attention(orc, got, qb, pos, Kb, Vb, what):
    n = int(pos.max()) + 1
    ref = orc.attention(qb, pos, Kb[:n], Vb[:n])
    bound = _attn_bound(orc, qb, pos, Kb[:n], Vb[:n], ref)
    return gu.assert_bound_gate(got.reshape(ref.shape), ref, bound, what)


# ---- decode attention at long contexts ----------------------------------------------

@pytest.mark.parametrize("R", [1, 2])
def test_33b_decode_attention_at_131k(orc, long33, R):
    """Decode attention of R rows at positions 131,000.. (256 units of 512 keys:
    the unstaged merge path with its 8-wide quarter loop)."""
    m, kv, Kb, Vb = long33
    pos0 = 131000
    q = synth.normal_bf16(61, R, (R, QD), 1.7, "cuda")
    out = torch.empty_like(q)
    tfl.tfl_layer_op(m, "attention", 0, q, out, kv, pos0)
    pos = np.arange(pos0, pos0 + R, dtype=np.int32)
    qb = synth.bits(q).reshape(R, L1.n_q, 128)
    _check_attention(orc, synth.bits(out), qb, pos, Kb, Vb, f"decode attention R={R} at {pos0}")


def test_33b_decode_window_16_rows_at_20k(orc, long33):
    """A 16-row window at positions 20,000..20,015: 40 units per row, past the
    32-unit limit of the staged merge."""
    m, kv, Kb, Vb = long33
    R, pos0 = 16, 20000
    q = synth.normal_bf16(62, 0, (R, QD), 1.7, "cuda")
    out = torch.empty_like(q)
    tfl.tfl_layer_op(m, "attention", 0, q, out, kv, pos0)
    pos = np.arange(pos0, pos0 + R, dtype=np.int32)
    _check_attention(orc, synth.bits(out), synth.bits(q).reshape(R, L1.n_q, 128), pos, Kb, Vb,
                     "16-row window at 20,000")


@pytest.mark.parametrize("R", [1, 2])
@pytest.mark.parametrize("pos0", [131000, 10000])
def test_33b_persistent_step_equals_per_launch_at_131k(long33, R, pos0):
    """The persistent decode step (the benchmark's launch configuration) and the
    launch per operation give the same logits, keys and values at 131,000
    positions, so the oracle gate of the per-operation attention above carries
    over to the persistent step.  Both positions give more attention units than
    CTAs (the step variant whose combine warps fold all but each CTA's last
    unit); at 10,000 most CTAs run one unit and a few two."""
    m, kv, _, _ = long33
    ids = synth.uniform_ids(63, R, L1.vocab, "cuda")
    k0, v0 = kv.read(0, pos0, R)       # the seeded rows the steps overwrite
    outs = []
    for persistent in (True, False):
        m.set_persistent(persistent)
        kv.reset(pos0)
        lg = torch.empty((R, L1.vocab), dtype=torch.bfloat16, device="cuda")
        m.decode_step([kv], ids, [R], lg)
        k, v = kv.read(0, pos0, R)
        outs.append((lg, k, v))
    m.set_persistent(True)
    assert m.status() == tfl.TFL_OK
    kv.write(0, pos0, k0, v0)
    kv.reset(LONG)
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---- prompt attention on full chunks -------------------------------------------------

SAMPLED = np.array([0, 1, 127, 128, 255, 256, 1023, 1500, 2046, 2047])


@pytest.mark.parametrize("pos0", [0, 129024])
def test_33b_prompt_attention_full_chunk(orc, long33, pos0):
    """A full 2,048-row prompt chunk of the 33B shape (56 query heads over 8 KV
    heads, G = 7) through the prompt attention kernel; sampled rows, every head,
    against the oracle."""
    m, kv, Kb, Vb = long33
    N = 2048
    q = synth.normal_bf16(64, pos0 // 1024, (N, QD), 1.7, "cuda")
    out = torch.empty_like(q)
    tfl.tfl_layer_op(m, "attention", 0, q, out, kv, pos0, prompt=True)
    pos = (pos0 + SAMPLED).astype(np.int32)
    qb = synth.bits(q)[SAMPLED].reshape(len(SAMPLED), L1.n_q, 128)
    _check_attention(orc, synth.bits(out)[SAMPLED], qb, pos, Kb, Vb, f"prompt chunk at {pos0}")


# ---- rising block maxima (the prompt kernel's lazy rescale) -----------------------------

def _rising(n_pos, n_kv, jump, seed):
    """Keys whose scores against q = 1 + N(0, 0.1^2) rise by about `jump` natural
    units from one 128-key block to the next: K_t = N(0,1) + c_t with
    c_t = (jump / sqrt(128)) floor(t / 128), so q . K_t / sqrt(128) is about
    jump floor(t / 128) + N(0, 1)."""
    K = synth.normal_bf16(seed, 0, (n_pos, n_kv, 128), 1.0, "cpu").float()
    c = (jump / 128.0 ** 0.5) * torch.floor(torch.arange(n_pos, dtype=torch.float32) / 128.0)
    K = (K + c[:, None, None]).to(torch.bfloat16)
    V = synth.normal_bf16(seed, 1, (n_pos, n_kv, 128), 1.0, "cpu")
    return K, V


def _rising_q(rows, n_q, seed):
    noise = synth.normal_bf16(seed, 2, (rows, n_q * 128), 0.1, "cpu").float()
    return (noise + 1.0).to(torch.bfloat16)


@pytest.mark.parametrize("pos0,rows", [(0, 1024), (300, 700), (900, 1)])
def test_prompt_attention_rising_block_maxima_tiny(orc, pos0, rows):
    """Block maxima rising by about 7 natural units (10 in log2 units, past the
    kernel's 2^8 rescale threshold) at every 128-key block: the running output in
    tensor memory is rescaled at each block boundary a row crosses."""
    m = _layer_model(TINY.with_layers(1), 1024 + 64, max_rows=1024)
    kv = m.kv(1024 + 64)
    K, V = _rising(1024, TINY.n_kv, 7.0, 85)
    kv.write(0, 0, K.cuda(), V.cuda())
    q = _rising_q(rows, TINY.n_q, 86 + pos0).cuda()
    out = torch.empty_like(q)
    tfl.tfl_layer_op(m, "attention", 0, q, out, kv, pos0, prompt=True)
    pos = np.arange(pos0, pos0 + rows, dtype=np.int32)
    qb = synth.bits(q).reshape(rows, TINY.n_q, 128)
    _check_attention(orc, synth.bits(out), qb, pos, synth.bits(K), synth.bits(V),
                     f"rising maxima, prompt pos0 {pos0} rows {rows}")


@pytest.mark.parametrize("R", [1, 2, 16])
def test_decode_attention_rising_block_maxima_tiny(orc, R):
    """The same key pattern through the decode attention (per-warp online
    softmax, then the merge of units whose maxima differ by tens of units)."""
    m = _layer_model(TINY.with_layers(1), 2048 + 64)
    kv = m.kv(2048 + 64)
    K, V = _rising(2048, TINY.n_kv, 7.0, 87)
    kv.write(0, 0, K.cuda(), V.cuda())
    pos0 = 2048 - R
    q = _rising_q(R, TINY.n_q, 88).cuda()
    out = torch.empty_like(q)
    tfl.tfl_layer_op(m, "attention", 0, q, out, kv, pos0)
    pos = np.arange(pos0, pos0 + R, dtype=np.int32)
    _check_attention(orc, synth.bits(out), synth.bits(q).reshape(R, TINY.n_q, 128), pos, synth.bits(K),
                     synth.bits(V), f"rising maxima, decode R={R}")
