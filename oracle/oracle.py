"""ctypes binding of the float64 C oracle (pm_oracle.c).

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the bench's
CPU-baseline leg.  Builds `_build/liborc.so` with gcc + OpenMP on first use.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from typing import Dict, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "pm_oracle.c")]
_HDR = os.path.join(_HERE, "pm_oracle.h")
_OUT = os.path.join(_HERE, "_build", "liborc.so")
_lock = threading.Lock()
_lib = None

ORC_OK, ORC_ERR_ARG, ORC_ERR_INVALID_ID = 0, 1, 2


class orc_config(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("D", "H", "dh", "ffn", "n_layers", "ctx", "text_in", "text_out",
                                         "audio_in", "n_streams")] + [
        ("delays", C.c_int * 64), ("init_text", C.c_int), ("init_audio", C.c_int),
        ("eps", C.c_double), ("rope_theta", C.c_double)] + [
        (n, C.c_int) for n in ("dep_D", "dep_H", "dep_dh", "dep_ffn", "dep_layers", "dep_steps", "dep_ctx",
                               "dep_card", "dep_text_in", "dep_audio_in", "pinned_ring")]


class orc_sampling(C.Structure):
    _fields_ = [("temperature", C.c_double), ("top_k", C.c_int), ("seed", C.c_uint64)]


def build(force: bool = False) -> str:
    """Compile the oracle to a shared library (plain C11, -O2, OpenMP)."""
    newest = max(os.path.getmtime(p) for p in _SRC + [_HDR])
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= newest:
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp] + _SRC + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OUT)
    return _OUT


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = C.CDLL(path)
            d, i, u16p, dp, i32p = C.c_double, C.c_int, C.POINTER(C.c_uint16), C.POINTER(C.c_double), C.POINTER(C.c_int32)
            L.orc_bf16_to_double.restype = d
            L.orc_bf16_to_double.argtypes = [C.c_uint16]
            L.orc_matvec.argtypes = [u16p, i, i, dp, dp]
            L.orc_rmsnorm.argtypes = [dp, u16p, i, d, dp]
            L.orc_rope.argtypes = [dp, i, C.c_long, d]
            L.orc_silu.restype = d
            L.orc_silu.argtypes = [d]
            L.orc_attend.argtypes = [dp, C.POINTER(dp), C.POINTER(dp), i, i, dp]
            L.orc_argmax.restype = i
            L.orc_argmax.argtypes = [dp, i]
            L.orc_tensor_count.restype = i
            L.orc_tensor_count.argtypes = [C.POINTER(orc_config)]
            L.orc_create.restype = C.c_void_p
            L.orc_create.argtypes = [C.POINTER(orc_config), C.POINTER(u16p), i]
            L.orc_destroy.argtypes = [C.c_void_p]
            L.orc_validate_ids.restype = i
            L.orc_validate_ids.argtypes = [C.POINTER(orc_config), i32p]
            L.orc_embed.argtypes = [C.c_void_p, i32p, dp]
            L.orc_stream_new.restype = C.c_void_p
            L.orc_stream_new.argtypes = [C.c_void_p]
            L.orc_stream_free.argtypes = [C.c_void_p, C.c_void_p]
            L.orc_stream_set_position.argtypes = [C.c_void_p, C.c_void_p, C.c_long]
            L.orc_stream_load_kv.argtypes = [C.c_void_p, C.c_void_p, i, C.c_long, C.c_long, u16p, u16p]
            L.orc_stream_position.restype = C.c_long
            L.orc_stream_position.argtypes = [C.c_void_p]
            L.orc_delay_assemble.restype = i
            L.orc_delay_assemble.argtypes = [C.c_void_p, C.c_void_p, i32p, i32p]
            L.orc_frame_step.restype = i
            L.orc_frame_step.argtypes = [C.c_void_p, C.c_void_p, i32p, dp, dp, dp, i32p]
            L.orc_set_threads.restype = i
            L.orc_set_threads.argtypes = [i]
            L.orc_frame_forward.restype = i
            L.orc_frame_forward.argtypes = [C.c_void_p, C.c_void_p, i32p, dp, dp, dp, i32p]
            L.orc_full_sequence.restype = i
            L.orc_full_sequence.argtypes = [C.c_void_p, i, i32p, dp, dp, i32p]
            L.orc_depformer_step.restype = i
            L.orc_depformer_step.argtypes = [C.c_void_p, dp, C.c_int32, i32p, dp, i32p]
            L.orc_ring_labels.argtypes = [C.c_long, C.c_long, C.POINTER(C.c_long)]
            L.orc_visible_positions.restype = i
            L.orc_visible_positions.argtypes = [C.c_long, C.c_long, i, C.POINTER(C.c_long)]
            u64p = C.POINTER(C.c_uint64)
            L.orc_philox4x64.argtypes = [u64p, u64p, u64p]
            L.orc_uniform24.restype = d
            L.orc_uniform24.argtypes = [C.c_uint64, C.c_uint64, C.c_uint64, C.c_uint64]
            L.orc_sample_topk.restype = i
            L.orc_sample_topk.argtypes = [dp, i, d, i, C.c_uint64, C.c_uint64, C.c_uint64, C.c_uint64, dp, dp]
            L.orc_depformer_step_sampled.restype = i
            L.orc_depformer_step_sampled.argtypes = [C.c_void_p, dp, C.c_int32, i32p, C.POINTER(orc_sampling),
                                                     C.c_uint64, C.c_uint64, dp, i32p, dp]
            _lib = L
    return _lib


def _dp(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_double))


def _u16p(a: np.ndarray):
    assert a.dtype == np.uint16 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_uint16))


def _i32p(a: np.ndarray):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_int32))


def make_config(shape: dict, depformer: bool = True) -> orc_config:
    c = orc_config()
    for k in ("D", "H", "dh", "ffn", "n_layers", "ctx", "text_in", "text_out", "audio_in", "n_streams",
              "init_text", "init_audio", "dep_D", "dep_H", "dep_dh", "dep_ffn", "dep_steps", "dep_ctx",
              "dep_card", "dep_text_in", "dep_audio_in"):
        setattr(c, k, int(shape[k]))
    c.dep_layers = int(shape["dep_layers"]) if depformer else 0
    c.pinned_ring = int(shape.get("pinned_ring", 0))
    c.eps = float(shape["eps"])
    c.rope_theta = float(shape["rope_theta"])
    for i, d in enumerate(shape["delays"]):
        c.delays[i] = int(d)
    return c


class Oracle:
    """A model over borrowed bf16 weight arrays (uint16) in the canonical tensor order."""

    def __init__(self, shape: dict, tensors: Sequence[np.ndarray], depformer: bool = True):
        self.L = lib()
        self.shape = dict(shape)
        self.cfg = make_config(shape, depformer)
        self._keep = [np.ascontiguousarray(t, dtype=np.uint16) for t in tensors]
        n = len(self._keep)
        if self.L.orc_tensor_count(C.byref(self.cfg)) != n:
            raise ValueError(f"expected {self.L.orc_tensor_count(C.byref(self.cfg))} tensors, got {n}")
        arr = (C.POINTER(C.c_uint16) * n)(*[_u16p(t) for t in self._keep])
        self._ptrs = arr
        self.h = self.L.orc_create(C.byref(self.cfg), arr, n)
        if not self.h:
            raise RuntimeError("orc_create failed")

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.L.orc_destroy(h)
            self.h = None

    def new_stream(self) -> "OracleStream":
        return OracleStream(self)

    def embed(self, inputs: np.ndarray) -> np.ndarray:
        x = np.zeros(self.shape["D"], np.float64)
        self.L.orc_embed(self.h, _i32p(np.ascontiguousarray(inputs, np.int32)), _dp(x))
        return x

    def full_sequence(self, ids: np.ndarray):
        T = ids.shape[0]
        ids = np.ascontiguousarray(ids, np.int32)
        hid = np.zeros((T, self.shape["D"]), np.float64)
        lg = np.zeros((T, self.shape["text_out"]), np.float64)
        am = np.zeros(T, np.int32)
        rc = self.L.orc_full_sequence(self.h, T, _i32p(ids), _dp(hid), _dp(lg), _i32p(am))
        if rc != ORC_OK:
            raise ValueError(f"orc_full_sequence rc={rc}")
        return hid, lg, am

    def depformer_step(self, hidden: np.ndarray, text_tok: int, supplied: np.ndarray):
        Q, V = self.shape["dep_steps"], self.shape["dep_card"]
        lg = np.zeros((Q, V), np.float64)
        codes = np.zeros(Q, np.int32)
        rc = self.L.orc_depformer_step(self.h, _dp(np.ascontiguousarray(hidden, np.float64)), int(text_tok),
                                       _i32p(np.ascontiguousarray(supplied, np.int32)), _dp(lg), _i32p(codes))
        if rc != ORC_OK:
            raise ValueError(f"orc_depformer_step rc={rc}")
        return lg, codes

    def depformer_step_sampled(self, hidden: np.ndarray, text_tok: int, supplied: np.ndarray, temperature: float,
                               top_k: int, seed: int, pos: int, row: int):
        """Codes sampled where none is supplied; returns logits, codes and pick margins."""
        Q, V = self.shape["dep_steps"], self.shape["dep_card"]
        lg = np.zeros((Q, V), np.float64)
        codes = np.zeros(Q, np.int32)
        margins = np.zeros(Q, np.float64)
        smp = orc_sampling(float(temperature), int(top_k), int(seed) & (2**64 - 1))
        rc = self.L.orc_depformer_step_sampled(self.h, _dp(np.ascontiguousarray(hidden, np.float64)), int(text_tok),
                                               _i32p(np.ascontiguousarray(supplied, np.int32)), C.byref(smp),
                                               int(pos), int(row), _dp(lg), _i32p(codes), _dp(margins))
        if rc != ORC_OK:
            raise ValueError(f"orc_depformer_step_sampled rc={rc}")
        return lg, codes, margins


class OracleStream:
    """One conversation's incremental-decode state (position, ID history, K/V by position)."""

    def __init__(self, model: Oracle):
        self.m = model
        self.L = model.L
        self.h = self.L.orc_stream_new(model.h)

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.L.orc_stream_free(self.m.h, h)
            self.h = None

    @property
    def pos(self) -> int:
        return int(self.L.orc_stream_position(self.h))

    def set_position(self, pos: int) -> None:
        self.L.orc_stream_set_position(self.m.h, self.h, int(pos))

    def load_kv(self, layer: int, first: int, k: np.ndarray, v: np.ndarray) -> None:
        """k, v: bf16 bits [H, n, dh]."""
        k = np.ascontiguousarray(k, np.uint16)
        v = np.ascontiguousarray(v, np.uint16)
        n = k.shape[1]
        self.L.orc_stream_load_kv(self.m.h, self.h, int(layer), int(first), int(n), _u16p(k), _u16p(v))

    def delay_assemble(self, ids: np.ndarray) -> np.ndarray:
        out = np.zeros(self.m.shape["n_streams"], np.int32)
        rc = self.L.orc_delay_assemble(self.m.h, self.h, _i32p(np.ascontiguousarray(ids, np.int32)), _i32p(out))
        if rc != ORC_OK:
            raise ValueError(f"invalid ids rc={rc}")
        return out

    def step(self, ids: np.ndarray, want_logits: bool = True):
        """Returns (hidden [D], residual [D], logits [text_out] or None, argmax)."""
        D = self.m.shape["D"]
        hid = np.zeros(D, np.float64)
        res = np.zeros(D, np.float64)
        lg = np.zeros(self.m.shape["text_out"], np.float64) if want_logits else None
        am = np.zeros(1, np.int32)
        rc = self.L.orc_frame_step(self.m.h, self.h, _i32p(np.ascontiguousarray(ids, np.int32)), _dp(hid),
                                   _dp(res), _dp(lg) if lg is not None else None, _i32p(am))
        if rc != ORC_OK:
            raise ValueError(f"orc_frame_step rc={rc}")
        return hid, res, lg, int(am[0])


    def forward(self, inputs: np.ndarray, want_logits: bool = True):
        """One frame from already-delayed inputs (no delay assembly).  Returns (hidden [D],
        residual [D], logits [text_out] or None, argmax)."""
        D = self.m.shape["D"]
        hid = np.zeros(D, np.float64)
        res = np.zeros(D, np.float64)
        lg = np.zeros(self.m.shape["text_out"], np.float64) if want_logits else None
        am = np.zeros(1, np.int32)
        rc = self.L.orc_frame_forward(self.m.h, self.h, _i32p(np.ascontiguousarray(inputs, np.int32)), _dp(hid),
                                      _dp(res), _dp(lg) if lg is not None else None, _i32p(am))
        if rc != ORC_OK:
            raise ValueError(f"orc_frame_forward rc={rc}")
        return hid, res, lg, int(am[0])


# --- scalar steps (pins) ----------------------------------------------------

def matvec(W: np.ndarray, x: np.ndarray) -> np.ndarray:
    W = np.ascontiguousarray(W, np.uint16)
    y = np.zeros(W.shape[0], np.float64)
    lib().orc_matvec(_u16p(W), W.shape[0], W.shape[1], _dp(np.ascontiguousarray(x, np.float64)), _dp(y))
    return y


def rmsnorm(x: np.ndarray, alpha_bits: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.zeros_like(x)
    lib().orc_rmsnorm(_dp(x), _u16p(np.ascontiguousarray(alpha_bits, np.uint16)), x.size, eps, _dp(out))
    return out


def rope(v: np.ndarray, pos: int, theta: float = 1e4) -> np.ndarray:
    v = np.array(v, np.float64, copy=True)
    lib().orc_rope(_dp(v), v.size, int(pos), theta)
    return v


def silu(g: float) -> float:
    return float(lib().orc_silu(float(g)))


def attend(q: np.ndarray, keys: np.ndarray, vals: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float64)
    keys = np.ascontiguousarray(keys, np.float64)
    vals = np.ascontiguousarray(vals, np.float64)
    n, dh = keys.shape
    kp = (C.POINTER(C.c_double) * n)(*[_dp(keys[i]) for i in range(n)])
    vp = (C.POINTER(C.c_double) * n)(*[_dp(vals[i]) for i in range(n)])
    o = np.zeros(dh, np.float64)
    lib().orc_attend(_dp(q), kp, vp, n, dh, _dp(o))
    return o


def set_threads(n: int) -> int:
    """Threads of the oracle's OpenMP loops from now on; returns the previous count."""
    return int(lib().orc_set_threads(int(n)))


def argmax(v: np.ndarray) -> int:
    v = np.ascontiguousarray(v, np.float64)
    return int(lib().orc_argmax(_dp(v), v.size))


# --- sampling ----------------------------------------------------------------

def philox4x64(counter, key) -> list:
    """Philox4x64-10 block of a 4-word counter under a 2-word key."""
    ctr = (C.c_uint64 * 4)(*[int(v) & (2**64 - 1) for v in counter])
    k = (C.c_uint64 * 2)(*[int(v) & (2**64 - 1) for v in key])
    out = (C.c_uint64 * 4)()
    lib().orc_philox4x64(ctr, k, out)
    return [int(v) for v in out]


def uniform24(seed: int, c0: int, c1: int, c2: int) -> float:
    return float(lib().orc_uniform24(int(seed) & (2**64 - 1), int(c0), int(c1), int(c2)))


def sample_topk(logits: np.ndarray, temperature: float, top_k: int, seed: int, c0: int, c1: int, c2: int):
    """Returns (token, margin, cut_gap) of temperature / top-k sampling of one row."""
    lg = np.ascontiguousarray(logits, np.float64)
    mg = C.c_double()
    gap = C.c_double()
    tok = lib().orc_sample_topk(_dp(lg), lg.size, float(temperature), int(top_k), int(seed) & (2**64 - 1), int(c0),
                                int(c1), int(c2), C.byref(mg), C.byref(gap))
    return int(tok), float(mg.value), float(gap.value)


# --- ring position labels ----------------------------------------------------

def ring_labels(capacity: int, end_offset: int) -> list:
    out = (C.c_long * int(capacity))()
    lib().orc_ring_labels(int(capacity), int(end_offset), out)
    return [int(v) for v in out]


def visible_positions(pos: int, capacity: int, pinned: bool) -> list:
    out = (C.c_long * int(capacity))()
    n = lib().orc_visible_positions(int(pos), int(capacity), int(bool(pinned)), out)
    return [int(out[i]) for i in range(n)]
