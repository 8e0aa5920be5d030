"""Thin ctypes binding of `libpm.so` (declared in include/pm.h).

Argument marshalling only: every step of the decode path runs in the library's CUDA
kernels.  There is no fallback: if the library cannot be loaded, importing fails.
PyTorch tensors are accepted wherever the C ABI takes a pointer (`.data_ptr()` is
passed); the caller keeps the tensors alive.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional, Sequence

from . import build as _build

PM_OK, PM_ERR_ARG, PM_ERR_INVALID_ID, PM_ERR_CUDA, PM_ERR_TIMEOUT, PM_ERR_STATE, PM_ERR_OOM, PM_ERR_UNSUPPORTED = range(8)
PM_ID_NONE, PM_ID_UNGENERATED, PM_ID_FEEDBACK = -1, -2, -3
PM_MAX_STREAMS = 32
STATUS_NAMES = {0: "PM_OK", 1: "PM_ERR_ARG", 2: "PM_ERR_INVALID_ID", 3: "PM_ERR_CUDA", 4: "PM_ERR_TIMEOUT",
                5: "PM_ERR_STATE", 6: "PM_ERR_OOM", 7: "PM_ERR_UNSUPPORTED"}

# every symbol include/pm.h declares
EXPORTS = ["pm_kv_cache_bytes", "pm_create", "pm_reset", "pm_set_positions", "pm_get_positions",
           "pm_frame_step", "pm_depformer_step", "pm_profile_frame", "pm_device_status", "pm_last_error",
           "pm_destroy", "pm_text_head_noalloc", "pm_set_sampling", "pm_sample", "pm_snapshot_bytes",
           "pm_snapshot", "pm_restore", "pm_prefill", "pm_set_wait_budget", "pm_generator_step"]
# every symbol include/pm_mimi.h declares
MIMI_EXPORTS = ["pm_mimi_tensor_count", "pm_mimi_create", "pm_mimi_decode", "pm_mimi_reset", "pm_mimi_status",
                "pm_mimi_get_frames", "pm_mimi_last_error", "pm_mimi_destroy", "pm_mimi_profile",
                "pm_mimi_encoder_tensor_count", "pm_mimi_encoder_create", "pm_mimi_encode", "pm_mimi_encode_profile",
                "pm_mimi_set_wait_budget"]
MIMI_KINDS = {0: "front", 1: "in_proj", 2: "attention", 3: "out_proj", 4: "lin1", 5: "lin2", 6: "conv_first",
              7: "convtr", 8: "res_conv1", 9: "res_conv2", 10: "conv_last", 11: "finish", 12: "down",
              13: "resample", 14: "rvq"}
PM_WAIT_BUDGET_DEFAULT = 0xFFFFFFFF
KERNEL_KINDS = {0: "embed", 1: "qkv_rope", 2: "attention", 3: "out_proj", 4: "linear_in_swiglu",
                5: "linear_out", 6: "text_head", 7: "frame_program", 8: "text_sample"}


class pm_config(C.Structure):
    _fields_ = [("B_max", C.c_int), ("D", C.c_int), ("H", C.c_int), ("dh", C.c_int), ("ffn", C.c_int),
                ("n_layers", C.c_int), ("ctx", C.c_int), ("text_in", C.c_int), ("text_out", C.c_int),
                ("audio_in", C.c_int), ("n_streams", C.c_int), ("delays", C.c_int * PM_MAX_STREAMS),
                ("init_text", C.c_int), ("init_audio", C.c_int), ("eps", C.c_float), ("rope_theta", C.c_float),
                ("dep_D", C.c_int), ("dep_H", C.c_int), ("dep_dh", C.c_int), ("dep_ffn", C.c_int),
                ("dep_layers", C.c_int), ("dep_steps", C.c_int), ("dep_ctx", C.c_int), ("dep_card", C.c_int),
                ("dep_text_in", C.c_int), ("dep_audio_in", C.c_int), ("flags", C.c_uint)]

PM_FLAG_FRAME_PROGRAM = 1
PM_FLAG_PINNED_RING = 2
PM_FLAG_DEPFORMER_CHAIN = 4
PM_FLAG_BATCHED_TCGEN05 = 8


_PP = C.POINTER(C.c_void_p)

PM_MIMI_MAX_B = 8
PM_MIMI_MAX_RATIOS = 8


class pm_mimi_config(C.Structure):
    _fields_ = [("B_max", C.c_int), ("dim", C.c_int), ("cb_dim", C.c_int), ("card", C.c_int), ("n_q", C.c_int),
                ("n_layers", C.c_int), ("heads", C.c_int), ("ffn", C.c_int), ("ctx", C.c_int),
                ("n_filters", C.c_int), ("n_ratios", C.c_int), ("ratios", C.c_int * PM_MIMI_MAX_RATIOS),
                ("kernel", C.c_int), ("last_kernel", C.c_int), ("res_kernel", C.c_int), ("compress", C.c_int),
                ("up_kernel", C.c_int), ("up_stride", C.c_int), ("ln_eps", C.c_float), ("rope_theta", C.c_float)]


class pm_temporal_weights(C.Structure):
    _fields_ = [("text_emb", C.c_void_p), ("audio_emb", C.c_void_p * (PM_MAX_STREAMS - 1)),
                ("norm1", _PP), ("in_proj", _PP), ("out_proj", _PP), ("norm2", _PP), ("linear_in", _PP),
                ("linear_out", _PP), ("out_norm", C.c_void_p), ("text_linear", C.c_void_p)]


class pm_depformer_weights(C.Structure):
    _fields_ = [("dep_in", _PP), ("text_emb", C.c_void_p), ("audio_emb", _PP), ("norm1", _PP), ("in_proj", _PP),
                ("out_proj", _PP), ("norm2", _PP), ("linear_in", _PP), ("linear_out", _PP), ("heads", _PP)]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libpm.so (compiling it first if the sources are newer)."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        vp, i32p, fp = C.c_void_p, C.POINTER(C.c_int32), C.c_void_p
        L.pm_kv_cache_bytes.restype = C.c_size_t
        L.pm_kv_cache_bytes.argtypes = [C.POINTER(pm_config)]
        L.pm_create.restype = C.c_int
        L.pm_create.argtypes = [C.POINTER(pm_config), C.POINTER(pm_temporal_weights),
                                C.POINTER(pm_depformer_weights), vp, vp, C.POINTER(C.c_void_p)]
        L.pm_reset.restype = C.c_int
        L.pm_reset.argtypes = [vp, vp]
        L.pm_set_positions.restype = C.c_int
        L.pm_set_positions.argtypes = [vp, C.c_int, vp]
        L.pm_get_positions.restype = C.c_int
        L.pm_get_positions.argtypes = [vp, vp]
        L.pm_frame_step.restype = C.c_int
        L.pm_frame_step.argtypes = [vp, C.c_int, vp, vp, vp, vp]
        L.pm_depformer_step.restype = C.c_int
        L.pm_depformer_step.argtypes = [vp, C.c_int, vp, vp, vp, vp, vp]
        L.pm_profile_frame.restype = C.c_int
        L.pm_profile_frame.argtypes = [vp, C.c_int, vp, vp, vp, vp, vp, vp, C.c_int, C.POINTER(C.c_int)]
        L.pm_device_status.restype = C.c_int
        L.pm_device_status.argtypes = [vp]
        L.pm_last_error.restype = C.c_char_p
        L.pm_last_error.argtypes = [vp]
        L.pm_text_head_noalloc.restype = C.c_int
        L.pm_text_head_noalloc.argtypes = [C.c_int, C.c_int, C.c_int, vp, vp, vp, C.c_float, vp, vp, vp, vp, vp]
        L.pm_generator_step.restype = C.c_int
        L.pm_generator_step.argtypes = [vp, C.c_int, vp, vp, vp, vp, vp, vp]
        L.pm_set_wait_budget.restype = C.c_int
        L.pm_set_wait_budget.argtypes = [vp, C.c_uint32]
        L.pm_set_sampling.restype = C.c_int
        L.pm_set_sampling.argtypes = [vp, C.c_float, C.c_int, C.c_float, C.c_int, C.c_ulonglong]
        L.pm_sample.restype = C.c_int
        L.pm_sample.argtypes = [vp, C.c_int, vp, C.c_int, C.c_int, C.c_float, C.c_int, C.c_ulonglong,
                                C.c_longlong, C.c_int, vp]
        L.pm_prefill.restype = C.c_int
        L.pm_prefill.argtypes = [vp, C.c_int, C.c_int, vp, vp, vp, vp]
        L.pm_snapshot_bytes.restype = C.c_size_t
        L.pm_snapshot_bytes.argtypes = [C.POINTER(pm_config)]
        L.pm_snapshot.restype = C.c_int
        L.pm_snapshot.argtypes = [vp, C.c_int, vp]
        L.pm_restore.restype = C.c_int
        L.pm_restore.argtypes = [vp, C.c_int, vp]
        L.pm_destroy.restype = None
        L.pm_destroy.argtypes = [vp]
        mp = C.POINTER(pm_mimi_config)
        L.pm_mimi_tensor_count.restype = C.c_int
        L.pm_mimi_tensor_count.argtypes = [mp]
        L.pm_mimi_create.restype = C.c_int
        L.pm_mimi_create.argtypes = [mp, vp, C.c_int, vp, C.POINTER(C.c_void_p)]
        L.pm_mimi_decode.restype = C.c_int
        L.pm_mimi_decode.argtypes = [vp, C.c_int, vp, vp]
        L.pm_mimi_reset.restype = C.c_int
        L.pm_mimi_reset.argtypes = [vp, vp]
        L.pm_mimi_status.restype = C.c_int
        L.pm_mimi_status.argtypes = [vp]
        L.pm_mimi_get_frames.restype = C.c_int
        L.pm_mimi_get_frames.argtypes = [vp, vp]
        L.pm_mimi_last_error.restype = C.c_char_p
        L.pm_mimi_last_error.argtypes = [vp]
        L.pm_mimi_profile.restype = C.c_int
        L.pm_mimi_profile.argtypes = [vp, C.c_int, vp, vp, vp, vp, C.c_int, C.POINTER(C.c_int)]
        L.pm_mimi_encoder_tensor_count.restype = C.c_int
        L.pm_mimi_encoder_tensor_count.argtypes = [mp]
        L.pm_mimi_encoder_create.restype = C.c_int
        L.pm_mimi_encoder_create.argtypes = [mp, vp, C.c_int, vp, C.POINTER(C.c_void_p)]
        L.pm_mimi_encode.restype = C.c_int
        L.pm_mimi_encode.argtypes = [vp, C.c_int, vp, vp, vp]
        L.pm_mimi_encode_profile.restype = C.c_int
        L.pm_mimi_encode_profile.argtypes = [vp, C.c_int, vp, vp, vp, vp, vp, C.c_int, C.POINTER(C.c_int)]
        L.pm_mimi_set_wait_budget.restype = C.c_int
        L.pm_mimi_set_wait_budget.argtypes = [vp, C.c_uint32]
        L.pm_mimi_destroy.restype = None
        L.pm_mimi_destroy.argtypes = [vp]
        _lib = L
    return _lib


class PMError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _ptr(x) -> Optional[int]:
    """Pointer of a torch tensor / numpy array / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(type(x))


def make_config(shape: dict, B_max: int, depformer: bool = True, flags: int = 0) -> pm_config:
    c = pm_config()
    c.B_max = int(B_max)
    c.flags = int(flags) | (PM_FLAG_PINNED_RING if shape.get("pinned_ring") else 0)
    for k in ("D", "H", "dh", "ffn", "n_layers", "ctx", "text_in", "text_out", "audio_in", "n_streams",
              "init_text", "init_audio", "dep_D", "dep_H", "dep_dh", "dep_ffn", "dep_steps", "dep_ctx",
              "dep_card", "dep_text_in", "dep_audio_in"):
        setattr(c, k, int(shape[k]))
    c.dep_layers = int(shape["dep_layers"]) if depformer else 0
    c.eps = float(shape["eps"])
    c.rope_theta = float(shape["rope_theta"])
    for i, d in enumerate(shape["delays"]):
        c.delays[i] = int(d)
    return c


def pm_kv_cache_bytes(cfg: pm_config) -> int:
    return int(lib().pm_kv_cache_bytes(C.byref(cfg)))


class Context:
    """Owns one pm_ctx.  `weights` maps the PyTorch parameter names of the inventory
    (see inputs.tensor_specs) to device tensors; `kv_cache` is a device tensor of
    pm_kv_cache_bytes bytes."""

    def __init__(self, shape: dict, weights: Dict[str, object], kv_cache, B_max: int = 1,
                 depformer: bool = True, stream: int = 0, flags: int = 0):
        L = lib()
        self.L = L
        self.shape = dict(shape)
        self.cfg = make_config(shape, B_max, depformer, flags)
        s = self.shape
        self._keep: List[object] = []

        def arr(names: Sequence[str]):
            a = (C.c_void_p * max(1, len(names)))(*[_ptr(weights[n]) for n in names])
            self._keep.append(a)
            return C.cast(a, _PP)

        tw = pm_temporal_weights()
        tw.text_emb = _ptr(weights["text_emb"])
        for i in range(s["n_streams"] - 1):
            tw.audio_emb[i] = _ptr(weights[f"emb.{i}"])
        Lr = range(s["n_layers"])
        tw.norm1 = arr([f"layers.{l}.norm1" for l in Lr])
        tw.in_proj = arr([f"layers.{l}.in_proj" for l in Lr])
        tw.out_proj = arr([f"layers.{l}.out_proj" for l in Lr])
        tw.norm2 = arr([f"layers.{l}.norm2" for l in Lr])
        tw.linear_in = arr([f"layers.{l}.linear_in" for l in Lr])
        tw.linear_out = arr([f"layers.{l}.linear_out" for l in Lr])
        tw.out_norm = _ptr(weights["out_norm"])
        tw.text_linear = _ptr(weights["text_linear"])
        dwp = None
        if depformer:
            Q, J = s["dep_steps"], s["dep_layers"]
            dw = pm_depformer_weights()
            dw.dep_in = arr([f"depformer_in.{q}" for q in range(Q)])
            dw.text_emb = _ptr(weights["depformer_text_emb"])
            dw.audio_emb = arr([f"depformer_emb.{q}" for q in range(Q - 1)])
            dw.norm1 = arr([f"depformer.{j}.norm1" for j in range(J)])
            dw.in_proj = arr([f"depformer.{j}.in_proj" for j in range(J)])
            dw.out_proj = arr([f"depformer.{j}.out_proj" for j in range(J)])
            dw.norm2 = arr([f"depformer.{j}.norm2" for j in range(J)])
            dw.linear_in = arr([f"depformer.{j}.gating.{q}.linear_in" for j in range(J) for q in range(Q)])
            dw.linear_out = arr([f"depformer.{j}.gating.{q}.linear_out" for j in range(J) for q in range(Q)])
            dw.heads = arr([f"linears.{q}" for q in range(Q)])
            self._dw = dw
            dwp = C.byref(dw)
        self._tw = tw
        self.kv_cache = kv_cache
        h = C.c_void_p()
        st = L.pm_create(C.byref(self.cfg), C.byref(tw), dwp, _ptr(kv_cache), stream or None, C.byref(h))
        if st != PM_OK:
            raise PMError(st, L.pm_last_error(None).decode())
        self.h = h

    def _check(self, st: int):
        if st != PM_OK:
            raise PMError(st, self.L.pm_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self.L.pm_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self, mask=None):
        m = None
        if mask is not None:
            m = (C.c_int32 * self.cfg.B_max)(*[int(v) for v in mask])
        self._check(self.L.pm_reset(self.h, m))

    def set_positions(self, pos: Sequence[int]):
        a = (C.c_int32 * len(pos))(*[int(p) for p in pos])
        self._check(self.L.pm_set_positions(self.h, len(pos), a))

    def get_positions(self) -> List[int]:
        a = (C.c_int32 * self.cfg.B_max)()
        self._check(self.L.pm_get_positions(self.h, a))
        return list(a)

    def frame_step(self, B: int, ids, text_logits=None, hidden=None, text_token=None) -> None:
        self._check(self.L.pm_frame_step(self.h, int(B), _ptr(ids), _ptr(text_logits), _ptr(hidden),
                                         _ptr(text_token)))

    def prefill(self, stream: int, T: int, ids, text_logits=None, hidden=None, text_token=None) -> None:
        """T frames of one stream in batched passes (ids [T][n_streams], host or device)."""
        self._check(self.L.pm_prefill(self.h, int(stream), int(T), _ptr(ids), _ptr(text_logits), _ptr(hidden),
                                      _ptr(text_token)))

    def depformer_step(self, B: int, hidden=None, text_tok=None, supplied=None, logits=None, codes=None) -> None:
        self._check(self.L.pm_depformer_step(self.h, int(B), _ptr(hidden), _ptr(text_tok), _ptr(supplied),
                                             _ptr(logits), _ptr(codes)))

    def set_sampling(self, text_temperature: float, text_top_k: int, audio_temperature: float, audio_top_k: int,
                     seed: int) -> None:
        """Temperature / top-k sampling of the text token and the depth codes (<= 0 / <= 1:
        greedy)."""
        self._check(self.L.pm_set_sampling(self.h, float(text_temperature), int(text_top_k),
                                           float(audio_temperature), int(audio_top_k),
                                           int(seed) & (2**64 - 1)))

    def sample(self, B: int, logits, V: int, ld: int, temperature: float, top_k: int, seed: int, position: int,
               substep: int, tokens) -> None:
        """Standalone sampling of B rows of device logits into `tokens` (device int32)."""
        self._check(self.L.pm_sample(self.h, int(B), _ptr(logits), int(V), int(ld), float(temperature), int(top_k),
                                     int(seed) & (2**64 - 1), int(position), int(substep), _ptr(tokens)))

    def snapshot_bytes(self) -> int:
        return int(self.L.pm_snapshot_bytes(C.byref(self.cfg)))

    def snapshot(self, stream: int, dst) -> None:
        """Stream `stream`'s decode state into the device buffer `dst`."""
        self._check(self.L.pm_snapshot(self.h, int(stream), _ptr(dst)))

    def restore(self, stream: int, src) -> None:
        self._check(self.L.pm_restore(self.h, int(stream), _ptr(src)))

    def profile_frame(self, B: int, ids, text_logits=None, hidden=None, text_token=None):
        """One frame with per-launch device times: list of (kind name, ms)."""
        n_max = 3 + 5 * self.shape["n_layers"]
        ms = (C.c_float * n_max)()
        kind = (C.c_int32 * n_max)()
        n = C.c_int(0)
        self._check(self.L.pm_profile_frame(self.h, int(B), _ptr(ids), _ptr(text_logits), _ptr(hidden),
                                            _ptr(text_token), ms, kind, n_max, C.byref(n)))
        return [(KERNEL_KINDS[kind[i]], float(ms[i])) for i in range(n.value)]

    def device_status(self) -> int:
        return int(self.L.pm_device_status(self.h))

    def generator_step(self, B: int, provided=None, out=None, out_valid=None, text_logits=None, hidden=None,
                       depth_logits=None) -> None:
        """One generator step (token ring + provided ring): aligned output codes into `out`."""
        if provided is not None and not hasattr(provided, "data_ptr"):
            import numpy as np
            provided = np.ascontiguousarray(provided, dtype=np.int32)
        self._check(self.L.pm_generator_step(self.h, int(B), _ptr(provided), _ptr(out), _ptr(out_valid),
                                             _ptr(text_logits), _ptr(hidden), _ptr(depth_logits)))

    def set_wait_budget(self, polls: int = PM_WAIT_BUDGET_DEFAULT) -> None:
        """Poll budget of the bounded waits (0: the next frame's waits run out at once)."""
        self._check(self.L.pm_set_wait_budget(self.h, int(polls) & 0xFFFFFFFF))


def pm_text_head_noalloc(B: int, D: int, V: int, residual, out_norm, text_linear, eps: float,
                         hidden=None, logits=None, token=None, status=None, stream: int = 0) -> int:
    """Final RMSNorm + text head + greedy token without a context or any device
    allocation (scratch in a static device array; B <= 64).  Returns the pm_status of the
    call; `status` (int32 [1], optional) receives the device-side outcome."""
    return int(lib().pm_text_head_noalloc(int(B), int(D), int(V), _ptr(residual), _ptr(out_norm),
                                          _ptr(text_linear), float(eps), _ptr(hidden), _ptr(logits), _ptr(token),
                                          _ptr(status), stream or None))


def upload_weights(weights: Dict[str, object], device: str = "cuda") -> Dict[str, object]:
    """Copy bf16 bit arrays (numpy uint16) to device tensors of dtype bfloat16."""
    import numpy as np
    import torch
    out = {}
    for k, v in weights.items():
        t = torch.from_numpy(np.ascontiguousarray(v).view(np.int16))
        out[k] = t.to(device, non_blocking=False).view(torch.bfloat16)
    return out


def alloc_kv_cache(cfg: pm_config, device: str = "cuda"):
    """A zeroed device buffer of pm_kv_cache_bytes(cfg) bytes, viewed as bf16
    [n_layers, 2, B_max, H, ctx, dh]."""
    import torch
    shape = (cfg.n_layers, 2, cfg.B_max, cfg.H, cfg.ctx, cfg.dh)
    return torch.zeros(shape, dtype=torch.bfloat16, device=device)


# ------------------------------------------------------------------------------------
# streaming Mimi decoder (include/pm_mimi.h)
# ------------------------------------------------------------------------------------

MIMI_DEFAULT = dict(dim=512, cb_dim=256, card=2048, n_q=8, n_layers=8, heads=8, ffn=2048, ctx=250, n_filters=64,
                    ratios=[8, 6, 5, 4], kernel=7, last_kernel=3, res_kernel=3, compress=2, up_kernel=4,
                    up_stride=2, ln_eps=1e-5, rope_theta=1e4)


def make_mimi_config(shape: dict, B_max: int) -> pm_mimi_config:
    s = dict(MIMI_DEFAULT)
    s.update(shape)
    c = pm_mimi_config()
    c.B_max = int(B_max)
    for k in ("dim", "cb_dim", "card", "n_q", "n_layers", "heads", "ffn", "ctx", "n_filters", "kernel",
              "last_kernel", "res_kernel", "compress", "up_kernel", "up_stride"):
        setattr(c, k, int(s[k]))
    c.n_ratios = len(s["ratios"])
    for i, r in enumerate(s["ratios"]):
        c.ratios[i] = int(r)
    c.ln_eps = float(s["ln_eps"])
    c.rope_theta = float(s["rope_theta"])
    return c


def mimi_tensor_names(shape: dict) -> List[str]:
    """Tensor names in the canonical order of include/pm_mimi.h."""
    s = dict(MIMI_DEFAULT)
    s.update(shape)
    n = [f"q.codebook.{j}" for j in range(s["n_q"])] + ["q.sem.out", "q.ac.out", "up.weight"]
    for l in range(s["n_layers"]):
        n += [f"tr.{l}.{k}" for k in ("norm1.w", "norm1.b", "in_proj", "out_proj", "scale1", "norm2.w", "norm2.b",
                                      "lin1", "lin2", "scale2")]
    n += ["dec.0.w", "dec.0.b"]
    for i in range(len(s["ratios"])):
        n += [f"dec.up{i}.w", f"dec.up{i}.b", f"dec.res{i}.w1", f"dec.res{i}.b1", f"dec.res{i}.w2", f"dec.res{i}.b2"]
    return n + ["dec.out.w", "dec.out.b"]


def mimi_frame_samples(shape: dict) -> int:
    s = dict(MIMI_DEFAULT)
    s.update(shape)
    n = int(s["up_stride"])
    for r in s["ratios"]:
        n *= int(r)
    return n


def mimi_encoder_tensor_names(shape: dict) -> List[str]:
    """Tensor names in the encoder's canonical order of include/pm_mimi.h."""
    s = dict(MIMI_DEFAULT)
    s.update(shape)
    n = ["enc.0.w", "enc.0.b"]
    for i in range(len(s["ratios"])):
        n += [f"enc.res{i}.w1", f"enc.res{i}.b1", f"enc.res{i}.w2", f"enc.res{i}.b2", f"enc.down{i}.w", f"enc.down{i}.b"]
    n += ["enc.out.w", "enc.out.b"]
    for l in range(s["n_layers"]):
        n += [f"etr.{l}.{k}" for k in ("norm1.w", "norm1.b", "in_proj", "out_proj", "scale1", "norm2.w", "norm2.b",
                                       "lin1", "lin2", "scale2")]
    return n + ["ds.weight", "q.sem.in", "q.ac.in"] + [f"q.codebook.{j}" for j in range(s["n_q"])]


class _MimiContext:
    """Owns one pm_mimi_ctx (decoder or encoder).  `weights` maps the canonical tensor
    names to bf16 device tensors; the context holds a reference to each, since the library
    reads them on every call."""

    _encoder = False

    def __init__(self, shape: dict, weights: Dict[str, object], B_max: int = 1, stream: int = 0):
        L = lib()
        self.L = L
        self.cfg = make_mimi_config(shape, B_max)
        self.frame_samples = mimi_frame_samples(shape)
        if self._encoder:
            names, count, create = (mimi_encoder_tensor_names(shape), L.pm_mimi_encoder_tensor_count,
                                    L.pm_mimi_encoder_create)
        else:
            names, count, create = mimi_tensor_names(shape), L.pm_mimi_tensor_count, L.pm_mimi_create
        n = count(C.byref(self.cfg))
        if n != len(names):
            raise PMError(PM_ERR_ARG, f"unsupported Mimi configuration (tensor count {n})")
        self._weights = [weights[k] for k in names]
        self._ptrs = (C.c_void_p * len(names))(*[_ptr(w) for w in self._weights])
        h = C.c_void_p()
        st = create(C.byref(self.cfg), self._ptrs, len(names), stream or None, C.byref(h))
        if st != PM_OK:
            raise PMError(st, L.pm_mimi_last_error(None).decode())
        self.h = h

    def _check(self, st: int):
        if st != PM_OK:
            raise PMError(st, self.L.pm_mimi_last_error(self.h).decode())

    def _timed(self, fn, *args):
        n_max = 8 + 5 * self.cfg.n_layers + 3 * self.cfg.n_ratios
        ms = (C.c_float * n_max)()
        kind = (C.c_int32 * n_max)()
        n = C.c_int(0)
        self._check(fn(self.h, *args, ms, kind, n_max, C.byref(n)))
        return [(MIMI_KINDS[kind[i]], float(ms[i])) for i in range(n.value)]

    def reset(self, mask=None) -> None:
        m = None
        if mask is not None:
            m = (C.c_int32 * self.cfg.B_max)(*[int(v) for v in mask])
        self._check(self.L.pm_mimi_reset(self.h, m))

    def status(self) -> int:
        return int(self.L.pm_mimi_status(self.h))

    def set_wait_budget(self, polls: int = PM_WAIT_BUDGET_DEFAULT) -> None:
        """Poll budget of the encoder's bounded waits (0: they give up at once)."""
        self._check(self.L.pm_mimi_set_wait_budget(self.h, int(polls) & 0xFFFFFFFF))

    def frames(self) -> List[int]:
        a = (C.c_int32 * self.cfg.B_max)()
        self._check(self.L.pm_mimi_get_frames(self.h, a))
        return list(a)

    def close(self):
        if getattr(self, "h", None):
            self.L.pm_mimi_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _i32(a):
    if a is not None and not hasattr(a, "data_ptr"):
        import numpy as np
        a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _f32(a):
    if a is not None and not hasattr(a, "data_ptr"):
        import numpy as np
        a = np.ascontiguousarray(a, dtype=np.float32)
    return a


class MimiDecoder(_MimiContext):
    """Streaming decoder: codes -> PCM (include/pm_mimi.h)."""

    def decode(self, B: int, codes, pcm) -> None:
        """Next frame of streams 0..B-1: codes [B][n_q] int32 (host or device), pcm
        [B][frame_samples] fp32 (device or host-mapped)."""
        self._check(self.L.pm_mimi_decode(self.h, int(B), _ptr(_i32(codes)), _ptr(pcm)))

    def profile(self, B: int, codes, pcm):
        """One decode with per-launch device times: list of (kind name, ms)."""
        return self._timed(self.L.pm_mimi_profile, int(B), _ptr(_i32(codes)), _ptr(pcm))


class MimiEncoder(_MimiContext):
    """Streaming encoder: PCM -> codes (include/pm_mimi.h)."""

    _encoder = True

    def encode(self, B: int, pcm, codes, latent=None) -> None:
        """Next frame of streams 0..B-1: pcm [B][frame_samples] fp32 (host or device),
        codes [B][n_q] int32 and latent [B][dim] fp32 out (device or host-mapped)."""
        self._check(self.L.pm_mimi_encode(self.h, int(B), _ptr(_f32(pcm)), _ptr(codes), _ptr(latent)))

    def profile(self, B: int, pcm, codes, latent=None):
        """One encode with per-launch device times: list of (kind name, ms)."""
        return self._timed(self.L.pm_mimi_encode_profile, int(B), _ptr(_f32(pcm)), _ptr(codes), _ptr(latent))
