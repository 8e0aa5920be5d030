"""Shared helpers of the GPU parity tests: build a model on both sides from the same
seeded bf16 bits, run frames through the C ABI, compare with the oracle.

Tolerances (stated by the decode-step workload): final hidden state within
max|diff| / max|ref| <= 2e-2; logits relative L2 <= 1e-2; greedy tokens bit-exact where the
oracle's top-2 gap exceeds 1e-2 (elsewhere both sides are fed the oracle's token).
"""
from __future__ import annotations

import json
import os

import numpy as np

from full_duplex_speech_moshi_gb300 import inputs as I

HIDDEN_TOL = 2e-2
LOGITS_TOL = 1e-2
GAP_MIN = 1e-2


def small_shape(**over):
    """Mid-size shapes: several GEMV tiles per CTA, ragged unit ranges, K = 2816 and
    768 paths, a 32-frame ring."""
    base = dict(D=1024, H=8, dh=128, ffn=2816, n_layers=2, ctx=32, text_in=1001, text_out=1000,
                audio_in=129, init_text=1000, init_audio=128, dep_D=512, dep_H=8, dep_dh=64,
                dep_ffn=768, dep_layers=2, dep_steps=16, dep_ctx=8, dep_card=128,
                dep_text_in=1001, dep_audio_in=129)
    base.update(over)
    return I.ModelShape(**base)


def hidden_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(gpu - ref)) / max(np.max(np.abs(ref)), 1e-30))


def logits_rel_l2(gpu: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30))


def top2_gap(ref: np.ndarray) -> float:
    s = np.sort(ref)
    return float(s[-1] - s[-2])


class Pair:
    """The same model on the GPU (through the C ABI) and in the oracle."""

    def __init__(self, shape: I.ModelShape, B_max: int = 1, depformer: bool = True, weights=None, flags: int = 0):
        import torch
        from full_duplex_speech_moshi_gb300 import pm
        from oracle import oracle as O
        self.torch = torch
        self.pm = pm
        self.shape = shape
        self.W = weights if weights is not None else I.make_weights(shape, depformer=depformer)
        specs = I.tensor_specs(shape, depformer)
        self.orc = O.Oracle(shape.asdict(), [self.W[n] for n, _, _ in specs], depformer=depformer)
        self.Wd = pm.upload_weights({n: self.W[n] for n, _, _ in specs})
        self.cfg = pm.make_config(shape.asdict(), B_max, depformer, flags)
        self.kv = pm.alloc_kv_cache(self.cfg)
        self.ctx = pm.Context(shape.asdict(), self.Wd, self.kv, B_max=B_max, depformer=depformer,
                              stream=torch.cuda.current_stream().cuda_stream, flags=flags)
        self.B_max = B_max
        self.streams = [self.orc.new_stream() for _ in range(B_max)]
        dev = "cuda"
        s = shape
        self.logits = torch.zeros((B_max, s.text_out), dtype=torch.float32, device=dev)
        self.hidden = torch.zeros((B_max, s.D), dtype=torch.float32, device=dev)
        self.token = torch.zeros((B_max,), dtype=torch.int32, device=dev)
        if depformer:
            self.dlogits = torch.zeros((B_max, s.dep_steps, s.dep_card), dtype=torch.float32, device=dev)
            self.dcodes = torch.zeros((B_max, s.dep_steps), dtype=torch.int32, device=dev)

    def close(self):
        self.ctx.close()

    def gpu_frame(self, ids: np.ndarray, B: int | None = None):
        """ids int32 [B, n_streams] (host).  Returns numpy hidden, logits, token."""
        B = B or ids.shape[0]
        self.ctx.frame_step(B, np.ascontiguousarray(ids, np.int32), self.logits, self.hidden, self.token)
        self.torch.cuda.synchronize()
        return (self.hidden[:B].double().cpu().numpy(), self.logits[:B].double().cpu().numpy(),
                self.token[:B].cpu().numpy())

    def oracle_frame(self, ids: np.ndarray):
        outs = [self.streams[b].step(ids[b]) for b in range(ids.shape[0])]
        return (np.stack([o[0] for o in outs]), np.stack([o[2] for o in outs]), np.array([o[3] for o in outs]))

    def check_frame(self, g, r, where=""):
        gh, gl, gt = g
        rh, rl, rt = r
        for b in range(gh.shape[0]):
            he = hidden_err(gh[b], rh[b])
            le = logits_rel_l2(gl[b], rl[b])
            assert he <= HIDDEN_TOL, f"{where} b={b} hidden err {he:.3e}"
            assert le <= LOGITS_TOL, f"{where} b={b} logits rel L2 {le:.3e}"
            if top2_gap(rl[b]) > GAP_MIN:
                assert int(gt[b]) == int(rt[b]), f"{where} b={b} token {gt[b]} vs oracle {rt[b]}"
        return max(hidden_err(gh[b], rh[b]) for b in range(gh.shape[0]))


def record_parity(name: str, **values) -> None:
    """Append one JSON line of measured parity figures (worst errors over a run) to the
    file named by PM_PARITY_LOG, when that variable is set; print it either way."""
    line = json.dumps({"case": name, **values})
    print(line)
    path = os.environ.get("PM_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")


class Worst:
    """Running worst hidden error / logits relative L2 of a parity run, and how many greedy
    decisions the oracle's near-tie let the two sides take differently (lockstep)."""

    def __init__(self):
        self.hidden = 0.0
        self.logits = 0.0
        self.frames = 0
        self.forced = 0

    def add(self, he: float, le: float) -> None:
        self.hidden = max(self.hidden, he)
        self.logits = max(self.logits, le)
        self.frames += 1

    def asdict(self) -> dict:
        return {"frames": self.frames, "worst_hidden_err": self.hidden, "worst_logits_rel_l2": self.logits,
                "near_tie_tokens_fed_from_oracle": self.forced}

