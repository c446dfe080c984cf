"""Thin Python binding of libtfl.so (include/tfl.h).

Argument marshalling only: every step of the forward runs in the library's CUDA
kernels.  PyTorch supplies device memory (tensors whose data_ptr is passed through)
and streams.  Functions keep the C names; the small classes below only own the
tensors that back a model's workspace and KV buffers.

The library is required: importing this module without a built libtfl.so raises,
and nothing here falls back to another implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtfl.so")

TFL_OK = 0
TFL_E_GEOMETRY = -1
TFL_E_ARCH = -2
TFL_E_CAPACITY = -3
TFL_E_ARG = -4
TFL_E_CUDA = -5
TFL_E_NONFINITE = -6
TFL_E_WORKSPACE = -7
TFL_E_DEVICE = -8
TFL_KV_PAGE = 128

_vp = ctypes.c_void_p


class tfl_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("layers", ctypes.c_int), ("n_q", ctypes.c_int),
                ("n_kv", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_float),
                ("max_rows", ctypes.c_int), ("max_decode_rows", ctypes.c_int), ("max_context", ctypes.c_int)]


class tfl_draft_stats(ctypes.Structure):
    _fields_ = [("rounds", ctypes.c_longlong), ("drafted", ctypes.c_longlong), ("accepted", ctypes.c_longlong),
                ("target_rows", ctypes.c_longlong), ("drafter_rows", ctypes.c_longlong)]


class tfl_weights(ctypes.Structure):
    _fields_ = [("embed", _vp), ("final_norm", _vp), ("lm_head", _vp)] + [
        (n, ctypes.POINTER(_vp)) for n in
        ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd")]


# C symbol -> (restype, argtypes); every symbol include/tfl.h declares
SIGNATURES = {
    "tfl_qualify": (ctypes.c_int, [ctypes.POINTER(tfl_config), ctypes.c_char_p, ctypes.c_size_t]),
    "tfl_rope_table": (None, [ctypes.c_double, ctypes.c_int, _vp, _vp]),
    "tfl_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(tfl_config)]),
    "tfl_init": (ctypes.c_int, [ctypes.POINTER(tfl_config), ctypes.POINTER(tfl_weights), _vp, ctypes.c_size_t,
                                ctypes.POINTER(_vp)]),
    "tfl_free": (None, [_vp]),
    "tfl_last_error": (ctypes.c_char_p, []),
    "tfl_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "tfl_kv_bytes": (ctypes.c_size_t, [ctypes.POINTER(tfl_config), ctypes.c_int]),
    "tfl_kv_alloc": (ctypes.c_int, [_vp, ctypes.c_int, _vp, ctypes.c_size_t, ctypes.POINTER(_vp)]),
    "tfl_kv_free": (None, [_vp]),
    "tfl_kv_reset": (ctypes.c_int, [_vp, ctypes.c_int]),
    "tfl_kv_length": (ctypes.c_int, [_vp]),
    "tfl_kv_capacity": (ctypes.c_int, [_vp]),
    "tfl_kv_write": (ctypes.c_int, [_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]),
    "tfl_kv_read": (ctypes.c_int, [_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]),
    "tfl_decode_step": (ctypes.c_int, [_vp, ctypes.POINTER(_vp), ctypes.c_int, _vp, ctypes.POINTER(ctypes.c_int),
                                       _vp, _vp]),
    "tfl_prefill_chunk": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int, _vp, ctypes.c_int, _vp]),
    "tfl_argmax": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _vp, _vp]),
    "tfl_status": (ctypes.c_int, [_vp, _vp]),
    "tfl_wait_probe": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, _vp]),
    "tfl_decode_hidden": (ctypes.c_int, [_vp, ctypes.POINTER(_vp), ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                         _vp, _vp, _vp]),
    "tfl_prefill_hidden": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int, _vp, _vp]),
    "tfl_head": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _vp, _vp]),
    "tfl_layer_op": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, _vp, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                    _vp]),
    "tfl_attention_decode_noalloc": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]),
    "tfl_profile": (ctypes.c_int, [_vp, ctypes.c_int]),
    "tfl_set_persistent": (ctypes.c_int, [_vp, ctypes.c_int]),
    "tfl_kv_copy_prefix": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int, _vp]),
    "tfl_prefix_store_new": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(_vp)]),
    "tfl_prefix_store_free": (None, [_vp]),
    "tfl_prefix_store_put": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int32), ctypes.c_int, _vp]),
    "tfl_prefix_store_match": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_int32), ctypes.c_int,
                                              ctypes.POINTER(_vp), ctypes.POINTER(ctypes.c_int)]),
    "tfl_prefix_store_remove": (ctypes.c_int, [_vp, _vp]),
    "tfl_prefix_store_size": (ctypes.c_int, [_vp]),
    "tfl_sample": (ctypes.c_int, [_vp, _vp, ctypes.c_int, ctypes.c_float, ctypes.c_int, ctypes.c_float, _vp, _vp,
                                  _vp]),
    "tfl_step_phases": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_double), ctypes.c_int]),
    "tfl_drafted_workspace_bytes": (ctypes.c_size_t, [_vp, ctypes.c_int]),
    "tfl_decode_drafted": (ctypes.c_int, [_vp, _vp, _vp, _vp, ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                                          ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_int32), _vp,
                                          ctypes.c_size_t, _vp, _vp]),
    "tfl_copy_draft": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(ctypes.c_int32)]),
    "tfl_profile_read": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_long)]),
    "tfl_profile_kind": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


def lib():
    """Loads libtfl.so (built by gqa_decoder_forward_gb300.build); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run gqa_decoder_forward_gb300.build.build() first "
                               "(there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


class TflError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} [{code}]")
        self.code = code


def _check(code: int) -> int:
    if code != TFL_OK:
        raise TflError(code, lib().tfl_last_error().decode())
    return code


def _ptr(t) -> int | None:
    if t is None:
        return None
    assert isinstance(t, torch.Tensor) and t.is_contiguous(), "expected a contiguous tensor"
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def config(shape, max_rows=64, max_decode_rows=64, max_context=4096) -> tfl_config:
    return tfl_config(shape.hidden, shape.layers, shape.n_q, shape.n_kv, shape.head_dim, shape.ffn, shape.vocab,
                      shape.rope_theta, shape.rms_eps, max_rows, max_decode_rows, max_context)


# ---- host-only entry points -------------------------------------------------------

def tfl_qualify(cfg: tfl_config) -> tuple[int, str]:
    buf = ctypes.create_string_buffer(512)
    code = lib().tfl_qualify(ctypes.byref(cfg), buf, 512)
    return code, buf.value.decode()


def tfl_workspace_bytes(cfg: tfl_config) -> int:
    return int(lib().tfl_workspace_bytes(ctypes.byref(cfg)))


def tfl_kv_bytes(cfg: tfl_config, max_positions: int) -> int:
    return int(lib().tfl_kv_bytes(ctypes.byref(cfg), int(max_positions)))


def tfl_rope_table(theta: float, n_pos: int):
    import numpy as np
    c = np.empty((n_pos, 64), np.uint16)
    s = np.empty((n_pos, 64), np.uint16)
    lib().tfl_rope_table(theta, n_pos, c.ctypes.data, s.ctypes.data)
    return c, s


# ---- objects ----------------------------------------------------------------------

class Model:
    """tfl_init over caller-owned weights (dict of bf16 CUDA tensors as made by
    synth.model_weights) plus a workspace tensor this object allocates."""

    def __init__(self, shape, weights: dict, max_rows=64, max_decode_rows=64, max_context=4096):
        self.shape = shape
        self.cfg = config(shape, max_rows, max_decode_rows, max_context)
        self.weights = weights
        nbytes = tfl_workspace_bytes(self.cfg)
        if nbytes == 0:
            code, msg = tfl_qualify(self.cfg)
            raise TflError(code, msg)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        w = tfl_weights()
        w.embed, w.final_norm, w.lm_head = (_ptr(weights[k]) for k in ("embed", "final_norm", "lm_head"))
        self._arrays = {}
        for k in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "wg", "wu", "wd"):
            arr = (_vp * shape.layers)(*[_ptr(t) for t in weights[k]])
            self._arrays[k] = arr
            setattr(w, k, ctypes.cast(arr, ctypes.POINTER(_vp)))
        self._w = w
        h = _vp()
        _check(lib().tfl_init(ctypes.byref(self.cfg), ctypes.byref(w), _ptr(self.workspace), nbytes,
                              ctypes.byref(h)))
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None):
            lib().tfl_free(self.handle)
            self.handle = None

    def kv(self, max_positions: int) -> "KV":
        return KV(self, max_positions)

    def decode_step(self, kvs: Sequence["KV"], ids: torch.Tensor, rows: Sequence[int], logits: torch.Tensor,
                    stream=None):
        return tfl_decode_step(self, kvs, ids, rows, logits, stream)

    def set_persistent(self, enable: bool):
        """Decode steps of one or two rows as one persistent launch (default) or
        as a launch per operation; the results are bit-identical."""
        return _check(lib().tfl_set_persistent(self.handle, 1 if enable else 0))

    def prefill_chunk(self, kv: "KV", ids: torch.Tensor, logits=None, all_rows=False, stream=None):
        return tfl_prefill_chunk(self, kv, ids, logits, all_rows, stream)

    def argmax(self, logits: torch.Tensor, ids: torch.Tensor, stream=None):
        return tfl_argmax(self, logits, ids, stream)

    def sample(self, logits: torch.Tensor, temperature: float, top_k: int, top_p: float, u: torch.Tensor,
               ids: torch.Tensor, stream=None):
        """Seeded draw per row (u: float32 CUDA tensor of uniforms in [0, 1))."""
        assert u.dtype == torch.float32 and u.is_cuda and ids.dtype == torch.int32
        return _check(lib().tfl_sample(self.handle, _ptr(logits), logits.shape[0], float(temperature), int(top_k),
                                       float(top_p), _ptr(u), _ptr(ids), _stream(stream)))

    def status(self, stream=None) -> int:
        return lib().tfl_status(self.handle, _stream(stream))

    def decode_drafted(self, kv: "KV", context, n_tokens: int, draft_len: int, drafter: "Model" = None,
                       dkv: "KV" = None, stream=None):
        """Drafted greedy decode (tfl_decode_drafted): context = the tokens so far
        (host ints, the last one pending, length(kv) == len(context) - 1).
        Returns (numpy int32 [n_tokens] greedy ids, stats dict)."""
        return tfl_decode_drafted(self, kv, context, n_tokens, draft_len, drafter, dkv, stream)


class KV:
    def __init__(self, model: Model, max_positions: int):
        self.model = model
        nbytes = tfl_kv_bytes(model.cfg, max_positions)
        self.buffer = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        h = _vp()
        _check(lib().tfl_kv_alloc(model.handle, int(max_positions), _ptr(self.buffer), nbytes, ctypes.byref(h)))
        self.handle = h

    def __del__(self):
        if getattr(self, "handle", None):
            lib().tfl_kv_free(self.handle)
            self.handle = None

    @property
    def length(self) -> int:
        return int(lib().tfl_kv_length(self.handle))

    def reset(self, keep: int):
        _check(lib().tfl_kv_reset(self.handle, int(keep)))

    def write(self, layer: int, pos0: int, k: torch.Tensor, v: torch.Tensor, stream=None):
        _check(lib().tfl_kv_write(self.model.handle, self.handle, layer, pos0, k.shape[0], _ptr(k), _ptr(v),
                                  _stream(stream)))

    def read(self, layer: int, pos0: int, n: int, stream=None):
        s = self.model.shape
        k = torch.empty((n, s.n_kv, s.head_dim), dtype=torch.bfloat16, device="cuda")
        v = torch.empty_like(k)
        _check(lib().tfl_kv_read(self.model.handle, self.handle, layer, pos0, n, _ptr(k), _ptr(v),
                                 _stream(stream)))
        return k, v


# ---- device entry points (C names) --------------------------------------------------

def _kv_array(kvs):
    return (_vp * len(kvs))(*[kv.handle for kv in kvs])


def tfl_decode_step(model: Model, kvs, ids, rows, logits, stream=None):
    assert ids.dtype == torch.int32 and logits.dtype == torch.bfloat16
    r = (ctypes.c_int * len(rows))(*rows)
    return _check(lib().tfl_decode_step(model.handle, _kv_array(kvs), len(kvs), _ptr(ids), r, _ptr(logits),
                                        _stream(stream)))


def tfl_decode_hidden(model: Model, kvs, rows, h_in, h_out, stream=None):
    r = (ctypes.c_int * len(rows))(*rows)
    return _check(lib().tfl_decode_hidden(model.handle, _kv_array(kvs), len(kvs), r, _ptr(h_in), _ptr(h_out),
                                          _stream(stream)))


def tfl_prefill_chunk(model: Model, kv: KV, ids, logits=None, all_rows=False, stream=None):
    assert ids.dtype == torch.int32
    return _check(lib().tfl_prefill_chunk(model.handle, kv.handle, _ptr(ids), ids.numel(), _ptr(logits),
                                          1 if all_rows else 0, _stream(stream)))


def tfl_prefill_hidden(model: Model, kv: KV, h_in, h_out, stream=None):
    return _check(lib().tfl_prefill_hidden(model.handle, kv.handle, _ptr(h_in), h_in.shape[0], _ptr(h_out),
                                           _stream(stream)))


def tfl_head(model: Model, h, logits, stream=None):
    return _check(lib().tfl_head(model.handle, _ptr(h), h.shape[0], _ptr(logits), _stream(stream)))


def tfl_argmax(model: Model, logits, ids, stream=None):
    return _check(lib().tfl_argmax(model.handle, _ptr(logits), logits.shape[0], _ptr(ids), _stream(stream)))


def tfl_status(model: Model, stream=None) -> int:
    return int(lib().tfl_status(model.handle, _stream(stream)))


def tfl_wait_probe(model: Model, which: int, spin_limit: int, stream=None):
    """Runs one bounded device wait (0: grid barrier, 1: mbarrier) on an event
    that never happens; tfl_status then reports TFL_E_DEVICE."""
    return _check(lib().tfl_wait_probe(model.handle, int(which), int(spin_limit), _stream(stream)))


TFL_OP_PROMPT = 0x100
OPS = {"attn_norm": 0, "qkv_rope": 1, "attention": 2, "o_residual": 3, "ffn_norm": 4, "gate_up": 5,
       "down_residual": 6, "final_norm": 7, "lm_head": 8, "norm_qkv_rope": 9, "norm_gate_up": 10,
       "norm_lm_head": 11}


def tfl_layer_op(model: Model, op: str, layer: int, inp: torch.Tensor, out: torch.Tensor, kv: "KV" = None,
                 pos0: int = 0, stream=None, prompt: bool = False):
    """One op of the decode path (prompt=True: of the prompt-chunk path)."""
    code = OPS[op] | (TFL_OP_PROMPT if prompt else 0)
    return _check(lib().tfl_layer_op(model.handle, code, layer, kv.handle if kv is not None else None, pos0,
                                     inp.shape[0], _ptr(inp), _ptr(out), _stream(stream)))


def tfl_attention_decode_noalloc(kv: "KV", layer: int, pos0: int, q: torch.Tensor, out: torch.Tensor, stream=None):
    """Decode attention with the library's fixed scratch (no allocation, no workspace)."""
    return _check(lib().tfl_attention_decode_noalloc(kv.handle, layer, pos0, q.shape[0], _ptr(q), _ptr(out),
                                                     _stream(stream)))


def tfl_profile(model: Model, enable: bool):
    return _check(lib().tfl_profile(model.handle, 1 if enable else 0))


def tfl_kv_copy_prefix(model: Model, src: "KV", dst: "KV", n: int, stream=None):
    """Copies positions [0, n) of every layer from src to dst; length(dst) = n."""
    _check(lib().tfl_kv_copy_prefix(model.handle, src.handle, dst.handle, n, _stream(stream)))


class PrefixStore:
    """Host index of caches holding prompt prefixes (tfl_prefix_store_*); the
    caches stay owned by the caller (KV objects are kept referenced here)."""

    def __init__(self, max_entries: int):
        h = _vp()
        _check(lib().tfl_prefix_store_new(max_entries, ctypes.byref(h)))
        self.handle = h
        self._kvs = {}

    def __del__(self):
        if getattr(self, "handle", None):
            lib().tfl_prefix_store_free(self.handle)
            self.handle = None

    @staticmethod
    def _tok(tokens):
        t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        return t, t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

    def put(self, tokens, kv: "KV"):
        t, p = self._tok(tokens)
        _check(lib().tfl_prefix_store_put(self.handle, p, len(t), kv.handle))
        self._kvs[kv.handle.value if hasattr(kv.handle, "value") else kv.handle] = kv

    def match(self, tokens):
        """(KV or None, matched token count)."""
        t, p = self._tok(tokens)
        h, n = _vp(), ctypes.c_int()
        _check(lib().tfl_prefix_store_match(self.handle, p, len(t), ctypes.byref(h), ctypes.byref(n)))
        return (self._kvs.get(h.value) if h.value else None), n.value

    def remove(self, kv: "KV"):
        _check(lib().tfl_prefix_store_remove(self.handle, kv.handle))
        self._kvs.pop(kv.handle.value if hasattr(kv.handle, "value") else kv.handle, None)

    def __len__(self):
        return lib().tfl_prefix_store_size(self.handle)


def tfl_copy_draft(tokens, max_draft: int) -> np.ndarray:
    """Copy-draft guesses for the tokens so far (host only)."""
    t = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    out = np.zeros(max(max_draft, 1), np.int32)
    n = _check_count(lib().tfl_copy_draft(t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(t), int(max_draft),
                                          out.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))))
    return out[:n]


def _check_count(code: int) -> int:
    if code < 0:
        raise TflError(code, lib().tfl_last_error().decode())
    return code


def tfl_decode_drafted(model: Model, kv: KV, context, n_tokens: int, draft_len: int, drafter: Model = None,
                       dkv: KV = None, stream=None):
    ctx = np.ascontiguousarray(np.asarray(context, dtype=np.int32))
    out = np.full(int(n_tokens), -1, np.int32)
    nbytes = int(lib().tfl_drafted_workspace_bytes(model.handle, int(draft_len)))
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    st = tfl_draft_stats()
    i32 = ctypes.POINTER(ctypes.c_int32)
    code = lib().tfl_decode_drafted(model.handle, kv.handle, drafter.handle if drafter is not None else None,
                                    dkv.handle if dkv is not None else None, int(draft_len),
                                    ctx.ctypes.data_as(i32), len(ctx), int(n_tokens), out.ctypes.data_as(i32),
                                    _ptr(ws), nbytes, ctypes.byref(st), _stream(stream))
    stats = {k: int(getattr(st, k)) for k, _ in tfl_draft_stats._fields_}
    if code != TFL_OK:
        err = TflError(code, lib().tfl_last_error().decode())
        err.ids, err.stats = out, stats
        raise err
    return out, stats


STEP_PHASES = ("qkv", "attention", "merge", "o", "gate_up", "down", "barrier", "head", "total")


def tfl_step_phases(model: Model) -> dict:
    """{phase: microseconds} of the last persistent decode step run while profiling."""
    out = (ctypes.c_double * len(STEP_PHASES))()
    _check(lib().tfl_step_phases(model.handle, out, len(STEP_PHASES)))
    return {k: round(v, 3) for k, v in zip(STEP_PHASES, out)}


def tfl_profile_read(model: Model) -> dict:
    """{family name: (total ms, launches)} recorded since the last read."""
    names = []
    while True:
        n = lib().tfl_profile_kind(len(names))
        if n is None:
            break
        names.append(n.decode())
    ms = (ctypes.c_double * len(names))()
    cnt = (ctypes.c_long * len(names))()
    _check(lib().tfl_profile_read(model.handle, len(names), ms, cnt))
    return {names[i]: (ms[i], cnt[i]) for i in range(len(names))}
