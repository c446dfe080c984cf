"""Oracle: plain CPU forward of the bf16 GQA decoder — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` /
``--impl reference`` legs may import this package.  The CUDA library never loads it
and shares no code with it (see ``oracle.cpp`` for the arithmetic and the readings
of the pages it follows: the rounding points of the Metal llama family pull request,
"A llama family on Metal ... #1415", section "How").

This module only marshals numpy arrays (bf16 held as ``uint16`` bit patterns) into
the C++ oracle; it does no arithmetic of its own.

Parity status per function (what pins it; see tests/test_oracle_*.py):
  bf16 rounding ............ pinned (independent bit-twiddle + torch + brute force)
  rmsnorm .................. pinned (closed form, 2^k scaling, brute force)
  linear ................... pinned (one-hot columns, exact small integers, brute force);
                             fp32-sum mode pinned against numpy's sequential fp32
                             cumulative sum and a sum that fp32 visibly truncates
  rope table / apply ....... pinned (p = 0 identity, inv_freq[0] = 1, closed forms,
                             relative-position invariance, rotation really applied)
  attention ................ pinned (one key, equal keys, brute force, causality, MHA/MQA)
  swiglu ................... pinned (silu(0) = 0, large-g limit, brute force)
  argmax ................... pinned (brute force, planted ties and non-finite values)
  layer / forward .......... invariants only (step == window, resumed == fresh,
                             hand-composed components) — the whole-model forward on
                             random weights is "parity unpinned" beyond those.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile oracle.cpp into liboracle.so with g++ (plain -O2, no fast math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.orc_bf16_from_double.restype = ctypes.c_uint16
        L.orc_bf16_from_double.argtypes = [ctypes.c_double]
        L.orc_bf16_to_double.restype = ctypes.c_double
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_get_threads.restype = ctypes.c_int
        L.orc_argmax.restype = ctypes.c_int
        L.orc_sample.restype = ctypes.c_int
        L.orc_sample.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_double,
                                 ctypes.POINTER(ctypes.c_double), _i32p]
        L.orc_forward.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(t)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"expected bf16 bit patterns as uint16, got {a.dtype}"
    return a


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


def set_fp32_sums(on: bool) -> None:
    """Projection sums in fp32 (k increasing) instead of double; see orc_linear."""
    lib().orc_set_fp32_sums(1 if on else 0)


def get_fp32_sums() -> bool:
    return bool(lib().orc_get_fp32_sums())


class fp32_sums:
    """Context manager: projection sums in fp32 inside the block."""

    def __enter__(self):
        self._old = get_fp32_sums()
        set_fp32_sums(True)
        return self

    def __exit__(self, *exc):
        set_fp32_sums(self._old)


# ---- elementwise ------------------------------------------------------------

def bf16_round(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_round_array(_p(x, _f64p), ctypes.c_long(x.size), _p(out, _u16p))
    return out


def bf16_value(b) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    b = np.asarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def residual_add(h, y) -> np.ndarray:
    h = _u16(h).copy()
    y = _u16(y)
    assert h.shape == y.shape
    lib().orc_residual_add(_p(h, _u16p), _p(y, _u16p), ctypes.c_long(h.size))
    return h


def rmsnorm(x, w, eps: float) -> np.ndarray:
    x = _u16(x)
    w = _u16(w)
    H = x.shape[-1]
    rows = x.size // H
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(x, _u16p), _p(w, _u16p), rows, H, ctypes.c_double(eps), _p(out, _u16p))
    return out


def linear(W, x) -> np.ndarray:
    """out[r, n] = bf16(sum_k W[n, k] x[r, k]) with W [N, K] and x [..., K]."""
    W = _u16(W)
    x = _u16(x)
    N, K = W.shape
    assert x.shape[-1] == K
    rows = x.size // K
    out = np.empty(x.shape[:-1] + (N,), np.uint16)
    lib().orc_linear(_p(W, _u16p), N, K, _p(x, _u16p), rows, _p(out, _u16p))
    return out


def rope_inv_freq(theta: float, D: int) -> np.ndarray:
    out = np.empty(D // 2, np.float32)
    lib().orc_rope_inv_freq(ctypes.c_double(theta), D, _p(out, _f32p))
    return out


def rope_table(theta: float, D: int, n_pos: int):
    c = np.empty((n_pos, D // 2), np.uint16)
    s = np.empty((n_pos, D // 2), np.uint16)
    lib().orc_rope_table(ctypes.c_double(theta), D, n_pos, _p(c, _u16p), _p(s, _u16p))
    return c, s


def rope_apply(x, pos: Sequence[int], cos_t, sin_t) -> np.ndarray:
    """x [rows, nh, D] -> rotated copy; row r at position pos[r]."""
    x = _u16(x).copy()
    rows, nh, D = x.shape
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    assert pos.shape == (rows,)
    cos_t, sin_t = _u16(cos_t), _u16(sin_t)
    lib().orc_rope_apply(_p(x, _u16p), rows, nh, D, _p(pos, _i32p), _p(cos_t, _u16p), _p(sin_t, _u16p))
    return x


def attention(q, pos, Kc, Vc) -> np.ndarray:
    """q [rows, NQ, D]; Kc, Vc [n_pos, NKV, D]; returns [rows, NQ*D]."""
    q = _u16(q)
    Kc, Vc = _u16(Kc), _u16(Vc)
    rows, NQ, D = q.shape
    NKV = Kc.shape[1]
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    assert int(pos.max(initial=-1)) < Kc.shape[0]
    out = np.empty((rows, NQ * D), np.uint16)
    lib().orc_attention(_p(q, _u16p), _p(pos, _i32p), rows, NQ, NKV, D,
                        _p(Kc, _u16p), _p(Vc, _u16p), _p(out, _u16p))
    return out


def swiglu(g, u) -> np.ndarray:
    g, u = _u16(g), _u16(u)
    assert g.shape == u.shape
    out = np.empty_like(g)
    lib().orc_swiglu(_p(g, _u16p), _p(u, _u16p), ctypes.c_long(g.size), _p(out, _u16p))
    return out


def argmax(logits):
    """Returns (ids int32 [rows], status); status -1 when a row holds NaN/+-Inf."""
    logits = _u16(logits)
    V = logits.shape[-1]
    rows = logits.size // V
    ids = np.empty(rows, np.int32)
    st = lib().orc_argmax(_p(logits, _u16p), rows, V, _p(ids, _i32p))
    return ids, int(st)


def sample(logits, temperature: float, top_k: int, top_p: float, u):
    """Seeded draw per row (see orc_sample): returns (ids int32 [rows], status)."""
    logits = _u16(logits)
    V = logits.shape[-1]
    rows = logits.size // V
    uu = np.ascontiguousarray(np.asarray(u, np.float64).reshape(rows))
    ids = np.empty(rows, np.int32)
    st = lib().orc_sample(_p(logits, _u16p), rows, V, float(temperature), int(top_k), float(top_p),
                          uu.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), _p(ids, _i32p))
    return ids, int(st)


# ---- model --------------------------------------------------------------------

class _Config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("layers", ctypes.c_int), ("n_q", ctypes.c_int),
                ("n_kv", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double)]


class _Weights(ctypes.Structure):
    _fields_ = [("embed", _u16p), ("final_norm", _u16p), ("lm_head", _u16p)] + [
        (n, ctypes.POINTER(_u16p)) for n in
        ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")]


@dataclass
class Config:
    hidden: int
    layers: int
    n_q: int
    n_kv: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    rms_eps: float

    def c(self) -> _Config:
        return _Config(self.hidden, self.layers, self.n_q, self.n_kv, self.head_dim, self.ffn,
                       self.vocab, self.rope_theta, self.rms_eps)


_LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")


class Model:
    """Holds host weights (uint16 bf16 patterns) and a flat KV cache per layer.

    weights: dict with 'embed', 'final_norm', 'lm_head' and, for each key in
    _LAYER_KEYS, a list of per-layer arrays.
    """

    def __init__(self, cfg: Config, weights: dict, max_pos: int):
        self.cfg = cfg
        self.max_pos = int(max_pos)
        self._keep = {}
        w = _Weights()
        for k in ("embed", "final_norm", "lm_head"):
            a = _u16(weights[k])
            self._keep[k] = a
            setattr(w, k, _p(a, _u16p))
        for k in _LAYER_KEYS:
            arrs = [_u16(a) for a in weights[k]]
            assert len(arrs) == cfg.layers, k
            ptrs = (_u16p * cfg.layers)(*[_p(a, _u16p) for a in arrs])
            self._keep[k] = (arrs, ptrs)
            setattr(w, k, ctypes.cast(ptrs, ctypes.POINTER(_u16p)))
        self._w = w
        self._c = cfg.c()
        shape = (cfg.layers, self.max_pos, cfg.n_kv, cfg.head_dim)
        self.K = np.zeros(shape, np.uint16)
        self.V = np.zeros(shape, np.uint16)

    def forward(self, ids, pos, want_logits=True, want_trace=False):
        """Run rows ids[] at positions pos[]; returns (logits or None, trace or None)."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        rows = ids.size
        assert pos.shape == (rows,)
        logits = np.empty((rows, self.cfg.vocab), np.uint16) if want_logits else None
        trace = np.empty((self.cfg.layers + 1, rows, self.cfg.hidden), np.uint16) if want_trace else None
        st = lib().orc_forward(ctypes.byref(self._c), ctypes.byref(self._w), _p(self.K, _u16p),
                               _p(self.V, _u16p), self.max_pos, _p(ids, _i32p), _p(pos, _i32p), rows,
                               _p(logits, _u16p) if logits is not None else None,
                               _p(trace, _u16p) if trace is not None else None)
        if st != 0:
            raise ValueError("oracle: position outside the cache")
        return logits, trace

    def layer(self, layer: int, h, pos):
        """One decoder layer in place on a copy of h [rows, hidden]; returns the new h."""
        h = _u16(h).copy()
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        rows = h.shape[0]
        top = int(pos.max()) + 1
        c, s = rope_table(self.cfg.rope_theta, self.cfg.head_dim, top)
        lib().orc_layer(ctypes.byref(self._c), layer, ctypes.byref(self._w),
                        _p(self.K[layer], _u16p), _p(self.V[layer], _u16p),
                        _p(pos, _i32p), rows, _p(h, _u16p), _p(c, _u16p), _p(s, _u16p))
        return h

    def head(self, h):
        h = _u16(h)
        rows = h.shape[0]
        out = np.empty((rows, self.cfg.vocab), np.uint16)
        lib().orc_head(ctypes.byref(self._c), ctypes.byref(self._w), _p(h, _u16p), rows, _p(out, _u16p))
        return out
