"""A second, independent float64 statement of the decode step in NumPy, for tiny shapes.

TEST INFRASTRUCTURE ONLY.  It evaluates a whole sequence of frames at once (every layer
over all T positions, attention with an explicit T x T mask matrix) and the depformer
as a loop, written from "PersonaPlex native LM audit" (clockless-atlas
personaplex-research page) sections 3 and 4, separately from the C oracle, so that the
two can be compared (incremental decode vs full recompute, C vs NumPy).
"""
from __future__ import annotations

import numpy as np


def widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64, exactly."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _norm(x: np.ndarray, alpha: np.ndarray, eps: float) -> np.ndarray:
    return alpha * x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def _rope_table(T: int, dh: int, theta: float):
    j = np.arange(dh // 2, dtype=np.float64)
    freq = np.exp(-np.log(theta) * 2.0 * j / dh)
    ang = np.arange(T, dtype=np.float64)[:, None] * freq[None, :]
    return np.cos(ang), np.sin(ang)


def _rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    # x [T, H, dh]; pairs are adjacent coordinates (2j, 2j+1)
    a = x[..., 0::2]
    b = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * cos[:, None, :] - b * sin[:, None, :]
    out[..., 1::2] = a * sin[:, None, :] + b * cos[:, None, :]
    return out


def _silu(g: np.ndarray) -> np.ndarray:
    return g / (1.0 + np.exp(-g))


def temporal_sequence(s: dict, W: dict, ids: np.ndarray):
    """ids int [T, n_streams] (undelayed, frames 0..T-1 from reset).
    Returns hidden [T, D], logits [T, text_out]."""
    T = ids.shape[0]
    D, H, dh, F = s["D"], s["H"], s["dh"], s["ffn"]
    # delays: stream k at frame t reads frame t - delay_k, or its initial ID
    inp = np.empty_like(ids)
    for k, d in enumerate(s["delays"]):
        init = s["init_text"] if k == 0 else s["init_audio"]
        for t in range(T):
            inp[t, k] = ids[t - d, k] if t - d >= 0 else init
    tables = [widen(W["text_emb"])] + [widen(W[f"emb.{i}"]) for i in range(s["n_streams"] - 1)]
    x = np.zeros((T, D))
    for k, tab in enumerate(tables):
        for t in range(T):
            if inp[t, k] != -1:
                x[t] += tab[inp[t, k]]
    cos, sin = _rope_table(T, dh, s["rope_theta"])
    tpos = np.arange(T)
    delta = tpos[:, None] - tpos[None, :]
    allowed = (delta >= 0) & (delta < s["ctx"])
    for l in range(s["n_layers"]):
        u = _norm(x, widen(W[f"layers.{l}.norm1"]), s["eps"])
        qkv = u @ widen(W[f"layers.{l}.in_proj"]).T
        q = _rope(qkv[:, :D].reshape(T, H, dh), cos, sin)
        k = _rope(qkv[:, D:2 * D].reshape(T, H, dh), cos, sin)
        v = qkv[:, 2 * D:].reshape(T, H, dh)
        sc = np.einsum("thd,shd->hts", q, k) / np.sqrt(dh)
        sc = np.where(allowed[None], sc, -np.inf)
        sc = sc - sc.max(axis=-1, keepdims=True)
        p = np.exp(sc)
        p = p / p.sum(axis=-1, keepdims=True)
        o = np.einsum("hts,shd->thd", p, v).reshape(T, D)
        y = x + o @ widen(W[f"layers.{l}.out_proj"]).T
        vn = _norm(y, widen(W[f"layers.{l}.norm2"]), s["eps"])
        gz = vn @ widen(W[f"layers.{l}.linear_in"]).T
        x = y + (_silu(gz[:, :F]) * gz[:, F:]) @ widen(W[f"layers.{l}.linear_out"]).T
    h = _norm(x, widen(W["out_norm"]), s["eps"])
    logits = h @ widen(W["text_linear"]).T
    return h, logits


def depformer(s: dict, W: dict, hidden: np.ndarray, text_tok: int, supplied: np.ndarray):
    """One frame of the depformer; returns logits [Q, card], codes [Q]."""
    Dd, Hd, dd, Fd, Q = s["dep_D"], s["dep_H"], s["dep_dh"], s["dep_ffn"], s["dep_steps"]
    J = s["dep_layers"]
    Kc = [np.zeros((Q, Dd)) for _ in range(J)]
    Vc = [np.zeros((Q, Dd)) for _ in range(J)]
    logits = np.zeros((Q, s["dep_card"]))
    codes = np.zeros(Q, np.int64)
    prev = int(text_tok)
    for q in range(Q):
        z = widen(W[f"depformer_in.{q}"]) @ hidden
        emb = W["depformer_text_emb"] if q == 0 else W[f"depformer_emb.{q - 1}"]
        z = z + widen(emb[prev])
        for j in range(J):
            u = _norm(z, widen(W[f"depformer.{j}.norm1"]), s["eps"])
            wq = widen(W[f"depformer.{j}.in_proj"])[q * 3 * Dd:(q + 1) * 3 * Dd]
            qkv = wq @ u
            Kc[j][q] = qkv[Dd:2 * Dd]
            Vc[j][q] = qkv[2 * Dd:]
            lo = max(0, q - s["dep_ctx"] + 1)
            o = np.zeros(Dd)
            for h in range(Hd):
                qh = qkv[h * dd:(h + 1) * dd]
                kh = Kc[j][lo:q + 1, h * dd:(h + 1) * dd]
                vh = Vc[j][lo:q + 1, h * dd:(h + 1) * dd]
                sc = kh @ qh / np.sqrt(dd)
                p = np.exp(sc - sc.max())
                o[h * dd:(h + 1) * dd] = (p / p.sum()) @ vh
            z = z + widen(W[f"depformer.{j}.out_proj"])[q * Dd:(q + 1) * Dd] @ o
            vn = _norm(z, widen(W[f"depformer.{j}.norm2"]), s["eps"])
            gz = widen(W[f"depformer.{j}.gating.{q}.linear_in"]) @ vn
            z = z + widen(W[f"depformer.{j}.gating.{q}.linear_out"]) @ (_silu(gz[:Fd]) * gz[Fd:])
        logits[q] = widen(W[f"linears.{q}"]) @ z
        best = int(np.argmax(logits[q]))
        codes[q] = supplied[q] if supplied[q] >= 0 else best
        prev = int(codes[q])
    return logits, codes
