"""Seeded synthetic inputs: random-init bf16 weights, KV contents and token ids.

This module holds none of the decoder's arithmetic.  It only draws numbers, and it
draws them the same way on any device: a counter-based 32-bit integer hash of
(seed, tensor id, element index), evaluated with int64 tensor ops that are exact on
CPU and GPU alike.  A "normal" draw is an Irwin-Hall sum of four 16-bit uniforms
(mean 0, bounded at about 3.46 sigma), converted exactly to fp32, scaled by one
IEEE fp32 multiply and rounded to bf16 by torch's round-to-nearest-even cast, so a
tensor generated on ``cuda:0`` is bit-identical to the same tensor generated on the
CPU.  Both the CUDA path and the oracle consume these tensors.

Distributions follow the workloads of the 33B-shaped configurations: projections,
embeddings and lm_head N(0, 0.02); RMSNorm weights 1 + N(0, 0.1); seeded KV
contents N(0, 1.7^2); token ids uniform over the vocabulary.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

_M32 = 0xFFFFFFFF
_CHUNK = 1 << 26  # elements per generation chunk (bounds the int64 temporaries)
# sigma of a sum of four independent uniforms on {0..65535}
_IH_SIGMA = (4.0 * (65536.0 ** 2 - 1.0) / 12.0) ** 0.5


@dataclass(frozen=True)
class ModelShape:
    """Geometry of a dense Llama-family GQA decoder."""
    hidden: int
    layers: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float = 1.2e8
    rms_eps: float = 1e-5

    def with_layers(self, n: int) -> "ModelShape":
        return replace(self, layers=n)


# The 33B shape (Nanbeige4.3-33B: hidden 7168, 52 layers, 56 q / 8 KV heads of
# 128, FFN 22016, vocab 166,912, unscaled RoPE theta 1.2e8) and the tiny test model.
NANBEIGE_33B = ModelShape(7168, 52, 56, 8, 128, 22016, 166912)
TINY = ModelShape(1024, 2, 8, 1, 128, 2816, 4096)


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2^32 for 0 <= x < 2^32 without int64 overflow."""
    lo = (x * (c & 0xFFFF)) & _M32
    hi = ((x * (c >> 16)) & 0xFFFF) << 16
    return (lo + hi) & _M32


def _mix32(x: torch.Tensor) -> torch.Tensor:
    """A 32-bit integer finaliser (xorshift-multiply; constants of 'lowbias32')."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def _key(seed: int, tensor_id: int) -> int:
    t = torch.tensor([(seed * 0x9E3779B1 + tensor_id * 0x85EBCA77 + 0x165667B1) & _M32], dtype=torch.int64)
    return int(_mix32(_mix32(t))[0])


def _words(key: int, idx: torch.Tensor, lane: int) -> torch.Tensor:
    # mixing rounds over (low index word ^ key), then (high index word, lane)
    h = _mix32((idx & _M32) ^ key)
    return _mix32(h ^ (((idx >> 32) * 0x632BE5AB + lane * 0x9E3779B9 + 0x7F4A7C15) & _M32))


def _normal_f32(key: int, start: int, n: int, device) -> torch.Tensor:
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    a = _words(key, idx, 0)
    b = _words(key, idx, 1)
    s = (a & 0xFFFF) + (a >> 16) + (b & 0xFFFF) + (b >> 16) - 2 * 65535
    return s.to(torch.float32)  # exact: |s| < 2^18


def normal_bf16(seed: int, tensor_id: int, shape, std: float, device="cpu", mean: float = 0.0) -> torch.Tensor:
    """bf16 tensor of N(mean, std^2)-like values (Irwin-Hall of order 4)."""
    shape = tuple(int(s) for s in shape)
    numel = 1
    for s in shape:
        numel *= s
    key = _key(seed, tensor_id)
    out = torch.empty(numel, dtype=torch.bfloat16, device=device)
    scale = torch.tensor(std / _IH_SIGMA, dtype=torch.float32, device=device)
    shift = torch.tensor(mean, dtype=torch.float32, device=device)
    for st in range(0, numel, _CHUNK):
        n = min(_CHUNK, numel - st)
        v = _normal_f32(key, st, n, device) * scale
        if mean != 0.0:
            v = v + shift
        out[st:st + n] = v.to(torch.bfloat16)
    return out.view(shape)


def uniform_ids(seed: int, n: int, vocab: int, device="cpu", tensor_id: int = 7) -> torch.Tensor:
    """int32 token ids, uniform over [0, vocab)."""
    key = _key(seed, tensor_id)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    return (_words(key, idx, 2) % vocab).to(torch.int32)


# tensor ids inside one model's seed
_GLOBAL_IDS = {"embed": 0, "final_norm": 1, "lm_head": 2}
LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")


def layer_tensor_shapes(m: ModelShape) -> dict:
    qd, kd = m.n_q * m.head_dim, m.n_kv * m.head_dim
    return {"attn_norm": (m.hidden,), "wq": (qd, m.hidden), "wk": (kd, m.hidden), "wv": (kd, m.hidden),
            "wo": (m.hidden, qd), "ffn_norm": (m.hidden,), "wg": (m.ffn, m.hidden),
            "wu": (m.ffn, m.hidden), "wd": (m.hidden, m.ffn)}


def layer_weight(m: ModelShape, seed: int, layer: int, key: str, device="cpu",
                 std: float = 0.02, norm_std: float = 0.1) -> torch.Tensor:
    shape = layer_tensor_shapes(m)[key]
    tid = 16 + layer * 16 + LAYER_KEYS.index(key)
    if key.endswith("norm"):
        return normal_bf16(seed, tid, shape, norm_std, device, mean=1.0)
    return normal_bf16(seed, tid, shape, std, device)


def global_weight(m: ModelShape, seed: int, key: str, device="cpu",
                  std: float = 0.02, norm_std: float = 0.1) -> torch.Tensor:
    tid = _GLOBAL_IDS[key]
    if key == "final_norm":
        return normal_bf16(seed, tid, (m.hidden,), norm_std, device, mean=1.0)
    return normal_bf16(seed, tid, (m.vocab, m.hidden), std, device)


def model_weights(m: ModelShape, seed: int, device="cpu", std: float = 0.02, norm_std: float = 0.1) -> dict:
    """All weights of a random-init model: globals plus per-layer lists."""
    w = {k: global_weight(m, seed, k, device, std, norm_std) for k in _GLOBAL_IDS}
    for k in LAYER_KEYS:
        w[k] = [layer_weight(m, seed, l, k, device, std, norm_std) for l in range(m.layers)]
    return w


def kv_contents(m: ModelShape, seed: int, layer: int, n_pos: int, device="cpu", std: float = 1.7):
    """Seeded K and V contents for one layer: two bf16 [n_pos, n_kv, head_dim] tensors."""
    shape = (n_pos, m.n_kv, m.head_dim)
    k = normal_bf16(seed, 1 << 20 | layer * 2, shape, std, device)
    v = normal_bf16(seed, 1 << 20 | layer * 2 + 1, shape, std, device)
    return k, v


def hidden_rows(m: ModelShape, seed: int, rows: int, device="cpu", std: float = 0.02) -> torch.Tensor:
    """Residual-stream rows drawn like embedding rows (bf16 [rows, hidden])."""
    return normal_bf16(seed, 5, (rows, m.hidden), std, device)


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy), the oracle's input form."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
