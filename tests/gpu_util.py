"""Helpers shared by the GPU parity tests: building the same random-init model on
the GPU (for libtfl) and on the host (for the oracle), and the comparison gates."""
from __future__ import annotations

import numpy as np
import torch

from gqa_decoder_forward_gb300 import synth


def gpu_weights(shape, seed):
    return synth.model_weights(shape, seed, "cuda")


def layer_weights(shape, seed):
    """The decoder-layer tensors of a random-init model on the GPU; embedding,
    final norm and lm_head are small placeholders (never read by the layer-only
    entry points tfl_decode_hidden / tfl_prefill_hidden, nor by the oracle's layer)."""
    w = {k: [synth.layer_weight(shape, seed, l, k, "cuda") for l in range(shape.layers)] for k in synth.LAYER_KEYS}
    w["embed"] = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    w["final_norm"] = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    w["lm_head"] = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    return w


def host_weights(w):
    out = {k: synth.bits(w[k]) for k in ("embed", "final_norm", "lm_head")}
    for k in synth.LAYER_KEYS:
        out[k] = [synth.bits(t) for t in w[k]]
    return out


def oracle_model(orc, shape, hw, max_pos):
    c = orc.Config(shape.hidden, shape.layers, shape.n_q, shape.n_kv, shape.head_dim, shape.ffn, shape.vocab,
                   shape.rope_theta, shape.rms_eps)
    return orc.Model(c, hw, max_pos)


def ulp_key(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_dist(a, b) -> np.ndarray:
    """Distance in bf16 steps between two bit patterns (order-mapped)."""
    return np.abs(ulp_key(a) - ulp_key(b))


def bf16_to_f64(b) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ulp_of(b) -> np.ndarray:
    """bf16 spacing at each value (2^(e-8) for |x| in [2^(e-1), 2^e); 2^-133 at 0)."""
    v = np.abs(bf16_to_f64(b))
    e = np.frexp(v)[1]
    return np.where(v > 0, np.ldexp(1.0, np.maximum(e - 8, -133)), 2.0 ** -133)


def assert_hidden_gate(gpu_bits, ref_bits, what=""):
    """The hidden-state gate for a value with one rounding point:
    <= 1 bf16 ulp for >= 99.9% of elements, <= 4 ulp everywhere."""
    d = ulp_dist(gpu_bits, ref_bits)
    frac1 = float(np.mean(d <= 1))
    assert frac1 >= 0.999, f"{what}: only {frac1:.5f} within 1 ulp (max {d.max()})"
    assert d.max() <= 4, f"{what}: max ulp distance {d.max()}"
    return frac1, int(d.max())


def assert_bound_gate(gpu_bits, ref_bits, bound, what=""):
    """The same gate for a fused op with several rounding points: |gpu - ref| within
    the bound that 1 ulp at each of the op's rounding points gives (ulp of the
    output plus each internal point's ulp times the output's sensitivity to it),
    for >= 99.9% of elements, and within 4 bounds everywhere."""
    e = np.abs(bf16_to_f64(gpu_bits) - bf16_to_f64(ref_bits)) / bound
    frac1 = float(np.mean(e <= 1.0))
    assert frac1 >= 0.999, f"{what}: only {frac1:.5f} within the rounding-point bound (max {e.max():.2f})"
    assert e.max() <= 4.0, f"{what}: max error {e.max():.2f} rounding-point bounds"
    return frac1, float(e.max())


def kl_mean(ref_bits, gpu_bits) -> float:
    """Mean over rows of KL(ref || gpu), softmax in double of the bf16 logits."""
    a = bf16_to_f64(ref_bits)
    b = bf16_to_f64(gpu_bits)
    a = a - a.max(axis=-1, keepdims=True)
    b = b - b.max(axis=-1, keepdims=True)
    la = a - np.log(np.exp(a).sum(axis=-1, keepdims=True))
    lb = b - np.log(np.exp(b).sum(axis=-1, keepdims=True))
    return float(np.mean(np.sum(np.exp(la) * (la - lb), axis=-1)))


def bf16_step(x: float) -> float:
    """Spacing of bf16 numbers at |x| (0.125 below 32, 0.25 from 32 to 64, ...)."""
    e = np.frexp(abs(x))[1]
    return 2.0 ** (e - 8)


def near_tie(logits_bits_row, a: int, b: int) -> bool:
    """The near-tie rule of the pages' teacher-forced checks: ids a and b within one
    bf16 step of each other."""
    v = bf16_to_f64(logits_bits_row)
    hi = max(abs(v[a]), abs(v[b]))
    return abs(v[a] - v[b]) <= bf16_step(hi)


def to_torch_bits(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def oracle_chain(orc, shape, hw, layer, h_in, pos, K_prefix, V_prefix):
    """Every rounding point of one decoder layer, computed by the oracle's pinned
    primitives from h_in [R, H] at positions pos, over a cache whose first
    positions hold K_prefix / V_prefix ([P, n_kv, D] bf16 bits)."""
    R = h_in.shape[0]
    D = shape.head_dim
    top = int(pos.max()) + 1
    c, s = orc.rope_table(shape.rope_theta, D, top)
    ones_h = np.full(shape.hidden, 0x3F80, np.uint16)
    ch = {"h_in": h_in, "cos": c[pos], "sin": s[pos]}
    ch["y1"] = orc.rmsnorm(h_in, ones_h, shape.rms_eps)            # bf16(x * r)
    ch["xn1"] = orc.rmsnorm(h_in, hw["attn_norm"][layer], shape.rms_eps)
    ch["qp"] = orc.linear(hw["wq"][layer], ch["xn1"]).reshape(R, shape.n_q, D)
    ch["kp"] = orc.linear(hw["wk"][layer], ch["xn1"]).reshape(R, shape.n_kv, D)
    ch["qp_abs"] = orc.linear(abs_bits(hw["wq"][layer]), abs_bits(ch["xn1"])).reshape(R, shape.n_q, D)
    ch["kp_abs"] = orc.linear(abs_bits(hw["wk"][layer]), abs_bits(ch["xn1"])).reshape(R, shape.n_kv, D)
    ch["q"] = orc.rope_apply(ch["qp"], pos, c, s)
    ch["k"] = orc.rope_apply(ch["kp"], pos, c, s)
    ch["v"] = orc.linear(hw["wv"][layer], ch["xn1"]).reshape(R, shape.n_kv, D)
    ch["v_abs"] = orc.linear(abs_bits(hw["wv"][layer]), abs_bits(ch["xn1"])).reshape(R, shape.n_kv, D)
    P = K_prefix.shape[0]
    Kc = np.zeros((top, shape.n_kv, D), np.uint16)
    Vc = np.zeros_like(Kc)
    Kc[:P], Vc[:P] = K_prefix, V_prefix
    Kc[pos], Vc[pos] = ch["k"], ch["v"]
    ch["o"] = orc.attention(ch["q"], pos, Kc, Vc)
    ch["o_abs"] = orc.attention(ch["q"], pos, Kc, abs_bits(Vc))     # sum p |v| / l
    ch["n_keys"] = int(pos.max()) + 1
    ch["yo"] = orc.linear(hw["wo"][layer], ch["o"])
    ch["yo_abs"] = orc.linear(abs_bits(hw["wo"][layer]), abs_bits(ch["o"]))
    ch["h1"] = orc.residual_add(h_in, ch["yo"])
    ch["y2"] = orc.rmsnorm(ch["h1"], ones_h, shape.rms_eps)
    ch["xn2"] = orc.rmsnorm(ch["h1"], hw["ffn_norm"][layer], shape.rms_eps)
    ch["g"] = orc.linear(hw["wg"][layer], ch["xn2"])
    ch["u"] = orc.linear(hw["wu"][layer], ch["xn2"])
    ch["g_abs"] = orc.linear(abs_bits(hw["wg"][layer]), abs_bits(ch["xn2"]))
    ch["u_abs"] = orc.linear(abs_bits(hw["wu"][layer]), abs_bits(ch["xn2"]))
    ch["sg"] = orc.swiglu(ch["g"], np.full_like(ch["g"], 0x3F80))   # bf16(silu(g))
    ch["a"] = orc.swiglu(ch["g"], ch["u"])
    ch["yd"] = orc.linear(hw["wd"][layer], ch["a"])
    ch["yd_abs"] = orc.linear(abs_bits(hw["wd"][layer]), abs_bits(ch["a"]))
    ch["K"] = (shape.hidden, shape.n_q * D, shape.ffn)
    ch["h2"] = orc.residual_add(ch["h1"], ch["yd"])
    return ch


# ---- rounding-point bounds of the fused ops (all from oracle values) ---------------

def abs_bits(b):
    return np.asarray(b, np.uint16) & np.uint16(0x7FFF)


def acc_allowance(abs_sum_bits, K):
    """fp32 accumulation allowance of a K-term sum: sqrt(K) * 2^-24 * sum |terms|
    (the usual probabilistic bound on rounding errors of a floating-point sum);
    abs_sum_bits holds bf16(sum |terms|)."""
    return np.sqrt(K) * 2.0 ** -24 * bf16_to_f64(abs_sum_bits)

def _round_bits(v):
    f = np.asarray(v, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bound_norm(y, w, out):
    """out = bf16(w * y), y = bf16(x * r): ulp(out) + |w| ulp(y)."""
    return ulp_of(out) + np.abs(bf16_to_f64(w)) * ulp_of(y)


def bound_rope(pre, cos, sin, out, acc=0.0):
    """out_j = bf16(bf16(x_j c) + bf16(o_j s)) with x = pre (a rounded sum with
    accumulation allowance acc), o the rotate-half partner: ulp(out) + ulp of both
    products + |c| (ulp(x_j) + acc_j) + |s| (ulp(o_j) + acc_o)."""
    x = bf16_to_f64(pre)
    half = x.shape[-1] // 2
    rot = np.concatenate([-x[..., half:], x[..., :half]], axis=-1)
    c = np.concatenate([bf16_to_f64(cos)] * 2, axis=-1)[:, None, :]
    s = np.concatenate([bf16_to_f64(sin)] * 2, axis=-1)[:, None, :]
    ux = ulp_of(pre) + acc
    urot = np.concatenate([ux[..., half:], ux[..., :half]], axis=-1)
    up = lambda v: ulp_of(_round_bits(v))  # noqa: E731
    return ulp_of(out) + up(x * c) + up(rot * s) + np.abs(c) * ux + np.abs(s) * urot


def bound_residual(y, out, acc=0.0):
    """out = bf16(h + y), y a rounded sum with accumulation allowance acc:
    ulp(out) + ulp(y) + acc."""
    return ulp_of(out) + ulp_of(y) + acc


def bound_swiglu(g, u, sg, out, acc_g=0.0, acc_u=0.0):
    """out = bf16(sg * u), sg = bf16(silu(g)), g and u rounded projections with
    accumulation allowances acc_g, acc_u."""
    gv, uv, sv = bf16_to_f64(g), bf16_to_f64(u), bf16_to_f64(sg)
    sig = 1.0 / (1.0 + np.exp(-gv))
    dsilu = sig * (1.0 + gv * (1.0 - sig))
    return (ulp_of(out) + np.abs(uv) * ulp_of(sg) + np.abs(uv * dsilu) * (ulp_of(g) + acc_g)
            + np.abs(sv) * (ulp_of(u) + acc_u))


def bound_sum(out, acc):
    """A single rounded sum: ulp(out) + its accumulation allowance."""
    return ulp_of(out) + acc


def check_ops(tfl, model, kv, layer, ch, pos0, report=None, head=None, prompt=False):
    """Runs each decode op (prompt=True: each prompt-chunk op) on the oracle's
    input of that op and gates its output: single-rounding outputs with the
    plain ulp gate, fused ones with the rounding-point bound.  head = (orc, hw,
    shape) also checks the final norm and lm_head on the oracle's layer output."""
    R = ch["h_in"].shape[0]
    T = lambda a: to_torch_bits(np.ascontiguousarray(a).reshape(R, -1))  # noqa: E731
    res = {}

    def gate(name, gpu, ref, bound=None):
        g = synth.bits(gpu).reshape(ref.shape)
        if bound is None:
            res[name] = assert_hidden_gate(g, ref, f"layer {layer} {name}")
        else:
            res[name] = assert_bound_gate(g, ref, bound, f"layer {layer} {name}")

    out = torch.empty_like(T(ch["xn1"]))
    tfl.tfl_layer_op(model, "attn_norm", layer, T(ch["h_in"]), out, prompt=prompt)
    gate("attn_norm", out, ch["xn1"], bound_norm(ch["y1"], model_norm(model, "attn_norm", layer), ch["xn1"]))
    q = torch.empty_like(T(ch["q"]))
    tfl.tfl_layer_op(model, "qkv_rope", layer, T(ch["xn1"]), q, kv, pos0, prompt=prompt)
    H, QD, F = ch["K"]
    gate("qkv_rope.q", q, ch["q"],
         bound_rope(ch["qp"], ch["cos"], ch["sin"], ch["q"], acc_allowance(ch["qp_abs"], H)))
    k, v = kv.read(layer, pos0, R)
    gate("qkv_rope.k", k, ch["k"],
         bound_rope(ch["kp"], ch["cos"], ch["sin"], ch["k"], acc_allowance(ch["kp_abs"], H)))
    gate("qkv_rope.v", v, ch["v"], bound_sum(ch["v"], acc_allowance(ch["v_abs"], H)))
    # the attention reads the oracle's keys and values for the call's own rows
    kv.write(layer, pos0, to_torch_bits(ch["k"]), to_torch_bits(ch["v"]))
    o = torch.empty_like(T(ch["o"]))
    tfl.tfl_layer_op(model, "attention", layer, T(ch["q"]), o, kv, pos0, prompt=prompt)
    gate("attention", o, ch["o"], bound_sum(ch["o"], acc_allowance(ch["o_abs"], ch["n_keys"])))
    h = T(ch["h_in"]).clone()
    tfl.tfl_layer_op(model, "o_residual", layer, T(ch["o"]), h, prompt=prompt)
    gate("o_residual", h, ch["h1"], bound_residual(ch["yo"], ch["h1"], acc_allowance(ch["yo_abs"], QD)))
    xn2 = torch.empty_like(h)
    tfl.tfl_layer_op(model, "ffn_norm", layer, T(ch["h1"]), xn2, prompt=prompt)
    gate("ffn_norm", xn2, ch["xn2"], bound_norm(ch["y2"], model_norm(model, "ffn_norm", layer), ch["xn2"]))
    a = torch.empty_like(T(ch["a"]))
    tfl.tfl_layer_op(model, "gate_up", layer, T(ch["xn2"]), a, prompt=prompt)
    gate("gate_up", a, ch["a"], bound_swiglu(ch["g"], ch["u"], ch["sg"], ch["a"], acc_allowance(ch["g_abs"], H),
                                             acc_allowance(ch["u_abs"], H)))
    h = T(ch["h1"]).clone()
    tfl.tfl_layer_op(model, "down_residual", layer, T(ch["a"]), h, prompt=prompt)
    gate("down_residual", h, ch["h2"], bound_residual(ch["yd"], ch["h2"], acc_allowance(ch["yd_abs"], F)))
    if head is not None:
        orc, hw, shape = head
        ones_h = np.full(shape.hidden, 0x3F80, np.uint16)
        yf = orc.rmsnorm(ch["h2"], ones_h, shape.rms_eps)
        xnf = orc.rmsnorm(ch["h2"], hw["final_norm"], shape.rms_eps)
        out = torch.empty_like(T(ch["h2"]))
        tfl.tfl_layer_op(model, "final_norm", 0, T(ch["h2"]), out)
        gate("final_norm", out, xnf, bound_norm(yf, hw["final_norm"], xnf))
        lg = torch.empty((R, shape.vocab), dtype=torch.bfloat16, device="cuda")
        tfl.tfl_layer_op(model, "lm_head", 0, T(xnf), lg)
        lm = orc.linear(hw["lm_head"], xnf)
        lm_abs = orc.linear(abs_bits(hw["lm_head"]), abs_bits(xnf))
        gate("lm_head", lg, lm, bound_sum(lm, acc_allowance(lm_abs, shape.hidden)))
    torch.cuda.synchronize()
    if report is not None:
        report.update(res)
    return res


def model_norm(model, key, layer):
    return synth.bits(model.weights[key][layer])


def rel_rms(gpu_bits, ref_bits) -> float:
    g, r = bf16_to_f64(gpu_bits), bf16_to_f64(ref_bits)
    return float(np.sqrt(np.mean((g - r) ** 2) / np.mean(r ** 2)))


# A whole layer fed the oracle's layer input differs from the oracle's layer by
# the propagation of 1-ulp differences at its rounding points: two bf16 steps
# (2^-7 relative) of root-mean-square difference bound it.
LAYER_REL_RMS = 2.0 ** -7
