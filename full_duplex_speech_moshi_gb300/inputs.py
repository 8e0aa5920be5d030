"""Seeded synthetic inputs for the Moshi/PersonaPlex per-frame decode step.

This module is the only code shared by the GPU path's tests and bench and by the
oracle's tests.  It holds shapes, seeds and random draws, and none of the decode
step's arithmetic.

Model shapes follow "PersonaPlex native LM audit" (clockless-atlas personaplex-research
page), sections 3-5 (temporal block, depth block, parameter inventory).  Random-init
distributions follow the workload statement of the decode benchmark: linear weights
~N(0, 0.02) in bf16, embedding tables ~N(0, 1) in bf16, RMSNorm scales 1 + 0.1*N(0, 1)
(so that scale application is exercised), per-frame IDs with text = pad ID 3 with
probability 0.65 (else uniform 0..31999) and audio uniform 0..2047 with 10% set to -1.

Draws are bf16 bit patterns (uint16).  A normal draw is made by an inverse-CDF table:
a uniform 16-bit index picks one of 65536 equiprobable quantiles of N(mean, std), each
rounded to nearest-even bf16.  Every tensor is cut into fixed chunks, each with its own
PCG64 stream keyed by (seed, chunk), so results do not depend on the thread count.
"""
from __future__ import annotations

import os
import statistics
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, asdict
from typing import Dict, List, Tuple

import numpy as np

# ----------------------------------------------------------------------------
# configurations
# ----------------------------------------------------------------------------

DELAYS_17 = [0, 0, 1, 1, 1, 1, 1, 1, 1, 0, 1, 1, 1, 1, 1, 1, 1]


@dataclass
class ModelShape:
    """Dimensions of the temporal stack and depformer (all integers are element counts)."""
    D: int = 4096
    H: int = 32
    dh: int = 128
    ffn: int = 11264          # gated hidden width (2*16896/3)
    n_layers: int = 32
    ctx: int = 3000
    text_in: int = 32001      # text embedding rows (32000 = initial text ID)
    text_out: int = 32000     # text head rows
    audio_in: int = 2049      # audio embedding rows (2048 = initial audio ID)
    n_streams: int = 17
    delays: List[int] = field(default_factory=lambda: list(DELAYS_17))
    init_text: int = 32000
    init_audio: int = 2048
    eps: float = 1e-8
    rope_theta: float = 1e4
    # depformer
    dep_D: int = 1024
    dep_H: int = 16
    dep_dh: int = 64
    dep_ffn: int = 2816       # gated hidden width (2*4224/3)
    dep_layers: int = 6
    dep_steps: int = 16
    dep_ctx: int = 8
    dep_card: int = 2048      # depth head rows
    dep_text_in: int = 32001
    dep_audio_in: int = 2049
    # 1: attention windows follow the pinned ring's position labels instead of the declared
    # mask (a full ring hides its oldest key)
    pinned_ring: int = 0

    def asdict(self) -> dict:
        return asdict(self)


FULL = ModelShape()


def tiny_shape(**over) -> ModelShape:
    """A small model with the same structure, used by fast parity tests."""
    base = dict(D=256, H=2, dh=128, ffn=512, n_layers=2, ctx=16, text_in=301, text_out=300,
                audio_in=65, init_text=300, init_audio=64, dep_D=256, dep_H=4, dep_dh=64,
                dep_ffn=256, dep_layers=2, dep_steps=16, dep_ctx=8, dep_card=64,
                dep_text_in=301, dep_audio_in=65)
    base.update(over)
    return ModelShape(**base)


# ----------------------------------------------------------------------------
# tensor inventory (names, shapes, distributions)
# ----------------------------------------------------------------------------

EMB, LINEAR, NORM = "emb", "linear", "norm"


def tensor_specs(s: ModelShape, depformer: bool = True) -> List[Tuple[str, Tuple[int, ...], str]]:
    """Canonical tensor order; weights are [out, in] as stored by PyTorch.

    The order is the layout contract used by the oracle's C API and by the tests that
    build the GPU context: index i of this list gets seed 1000 + i.
    """
    out: List[Tuple[str, Tuple[int, ...], str]] = []
    out.append(("text_emb", (s.text_in, s.D), EMB))
    for i in range(s.n_streams - 1):
        out.append((f"emb.{i}", (s.audio_in, s.D), EMB))
    for l in range(s.n_layers):
        out.append((f"layers.{l}.norm1", (s.D,), NORM))
        out.append((f"layers.{l}.in_proj", (3 * s.D, s.D), LINEAR))
        out.append((f"layers.{l}.out_proj", (s.D, s.D), LINEAR))
        out.append((f"layers.{l}.norm2", (s.D,), NORM))
        out.append((f"layers.{l}.linear_in", (2 * s.ffn, s.D), LINEAR))
        out.append((f"layers.{l}.linear_out", (s.D, s.ffn), LINEAR))
    out.append(("out_norm", (s.D,), NORM))
    out.append(("text_linear", (s.text_out, s.D), LINEAR))
    if depformer:
        Q = s.dep_steps
        for q in range(Q):
            out.append((f"depformer_in.{q}", (s.dep_D, s.D), LINEAR))
        out.append(("depformer_text_emb", (s.dep_text_in, s.dep_D), EMB))
        for q in range(Q - 1):
            out.append((f"depformer_emb.{q}", (s.dep_audio_in, s.dep_D), EMB))
        for j in range(s.dep_layers):
            out.append((f"depformer.{j}.norm1", (s.dep_D,), NORM))
            out.append((f"depformer.{j}.in_proj", (Q * 3 * s.dep_D, s.dep_D), LINEAR))
            out.append((f"depformer.{j}.out_proj", (Q * s.dep_D, s.dep_D), LINEAR))
            out.append((f"depformer.{j}.norm2", (s.dep_D,), NORM))
            for q in range(Q):
                out.append((f"depformer.{j}.gating.{q}.linear_in", (2 * s.dep_ffn, s.dep_D), LINEAR))
            for q in range(Q):
                out.append((f"depformer.{j}.gating.{q}.linear_out", (s.dep_D, s.dep_ffn), LINEAR))
        for q in range(Q):
            out.append((f"linears.{q}", (s.dep_card, s.dep_D), LINEAR))
    return out


# ----------------------------------------------------------------------------
# random draws
# ----------------------------------------------------------------------------

_CHUNK = 1 << 22
_TABLES: Dict[Tuple[float, float], np.ndarray] = {}


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to nearest-even bf16 and return the 16-bit patterns."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_table(mean: float, std: float) -> np.ndarray:
    key = (mean, std)
    if key not in _TABLES:
        nd = statistics.NormalDist(mean, std)
        q = np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)], dtype=np.float64)
        _TABLES[key] = _f32_to_bf16_bits(q.astype(np.float32))
    return _TABLES[key]


def _fill_chunk(out: np.ndarray, table: np.ndarray, seed: int, chunk: int) -> None:
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, chunk])))
    lo = chunk * _CHUNK
    hi = min(out.size, lo + _CHUNK)
    idx = g.integers(0, 65536, size=hi - lo, dtype=np.uint16)
    out[lo:hi] = table[idx]


def normal_bf16(shape, mean: float, std: float, seed: int, pool: ThreadPoolExecutor | None = None) -> np.ndarray:
    """bf16 bits of a seeded N(mean, std) draw of the given shape."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    table = _normal_table(mean, std)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    if pool is None or nchunks == 1:
        for c in range(nchunks):
            _fill_chunk(out, table, seed, c)
    else:
        list(pool.map(lambda c: _fill_chunk(out, table, seed, c), range(nchunks)))
    return out.reshape(shape)


_DIST = {EMB: (0.0, 1.0), LINEAR: (0.0, 0.02), NORM: (1.0, 0.1)}


def make_weights(s: ModelShape, depformer: bool = True, base_seed: int = 1000,
                 threads: int | None = None) -> Dict[str, np.ndarray]:
    """All tensors of `tensor_specs(s)` as bf16 bit arrays (uint16), keyed by name."""
    specs = tensor_specs(s, depformer)
    threads = threads or min(32, os.cpu_count() or 1)
    out: Dict[str, np.ndarray] = {}
    with ThreadPoolExecutor(threads) as pool:
        for i, (name, shape, kind) in enumerate(specs):
            mean, std = _DIST[kind]
            out[name] = normal_bf16(shape, mean, std, base_seed + i, pool)
    return out


def make_ids(s: ModelShape, T: int, B: int = 1, seed: int = 2000, pad_id: int = 3,
             pad_prob: float = 0.65, audio_card: int = 2048, drop_prob: float = 0.10) -> np.ndarray:
    """Per-frame undelayed token IDs, int32 [T, B, n_streams].

    Stream 0 is text: `pad_id` with probability `pad_prob`, else uniform over the text
    vocabulary below the initial ID.  Streams 1.. are audio: uniform 0..audio_card-1,
    each replaced by -1 (no input) with probability `drop_prob`.
    """
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, B, T])))
    ids = np.empty((T, B, s.n_streams), dtype=np.int32)
    text_hi = min(s.init_text, s.text_in - 1)
    is_pad = g.random((T, B)) < pad_prob
    txt = g.integers(0, text_hi, size=(T, B))
    ids[:, :, 0] = np.where(is_pad, min(pad_id, text_hi - 1), txt)
    card = min(audio_card, s.init_audio)
    aud = g.integers(0, card, size=(T, B, s.n_streams - 1))
    drop = g.random((T, B, s.n_streams - 1)) < drop_prob
    ids[:, :, 1:] = np.where(drop, -1, aud)
    return ids


def make_supplied_codes(s: ModelShape, T: int, B: int = 1, seed: int = 4000, n_generated: int = 8) -> np.ndarray:
    """Depformer supplied codes, int32 [T, B, dep_steps]: -1 (generate) for the first
    `n_generated` positions, uniform 0..dep_card-1 for the rest."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, B, T])))
    sup = g.integers(0, s.dep_card, size=(T, B, s.dep_steps)).astype(np.int32)
    sup[:, :, :n_generated] = -1
    return sup


def make_cache_lengths(B: int, lo: int = 64, hi: int = 3000, seed: int = 3000) -> np.ndarray:
    """Per-stream prefilled cache lengths, uniform lo..hi inclusive."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, B])))
    return g.integers(lo, hi + 1, size=B).astype(np.int32)


def make_kv_history(s: ModelShape, n_pos: int, seed: int, layer: int, stream: int,
                    pool: ThreadPoolExecutor | None = None) -> Tuple[np.ndarray, np.ndarray]:
    """Seeded stand-in K/V history for one (layer, stream): bf16 bits [H, n_pos, dh] each,
    ~N(0, 1).  Attention cost does not depend on cache contents, and both sides read
    the same bits."""
    k = normal_bf16((s.H, n_pos, s.dh), 0.0, 1.0, seed * 1000003 + layer * 1009 + stream * 2 + 0, pool)
    v = normal_bf16((s.H, n_pos, s.dh), 0.0, 1.0, seed * 1000003 + layer * 1009 + stream * 2 + 1, pool)
    return k, v


def make_weights_device(s: ModelShape, depformer: bool = True, seed: int = 1000, device: str = "cuda"):
    """Seeded weights of the same shapes and distributions drawn directly on the device
    with torch's generator (bf16 by nearest-even rounding of fp32 draws).  Used where only
    timing matters and host copies would cost more than the measurement (the bench)."""
    import torch
    g = torch.Generator(device=device)
    out = {}
    for i, (name, shape, kind) in enumerate(tensor_specs(s, depformer)):
        mean, std = _DIST[kind]
        g.manual_seed(seed + i)
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        t.mul_(std).add_(mean)
        out[name] = t.to(torch.bfloat16)
        del t
    return out


# ----------------------------------------------------------------------------
# Mimi decoder ("PersonaPlex native LM audit", chapter "Exact Mimi codec construction")
# ----------------------------------------------------------------------------

MIMI_FULL = dict(dim=512, cb_dim=256, card=2048, n_q=8, n_layers=8, heads=8, ffn=2048, ctx=250, n_filters=64,
                 ratios=[8, 6, 5, 4], kernel=7, last_kernel=3, res_kernel=3, compress=2, up_kernel=4,
                 up_stride=2, ln_eps=1e-5, rope_theta=1e4)

# the smallest shape the GPU kernels take (dim a multiple of 256) that still has two
# transformer blocks, a window the test outruns in a few frames and two SEANet stages
MIMI_SMALL = dict(MIMI_FULL, dim=256, cb_dim=32, card=64, n_layers=2, heads=4, ffn=512, ctx=6, n_filters=8,
                  ratios=[4, 3])


def mimi_tensor_specs(shape: dict) -> List[Tuple[str, Tuple[int, ...]]]:
    """Names and shapes of the decoder's tensors in their canonical order (PyTorch
    layouts: Linear [out, in], Conv1d [out, in, k], ConvTranspose1d [in, out, k])."""
    s = dict(MIMI_FULL)
    s.update(shape)
    t = [(f"q.codebook.{j}", (s["card"], s["cb_dim"])) for j in range(s["n_q"])]
    t += [("q.sem.out", (s["dim"], s["cb_dim"])), ("q.ac.out", (s["dim"], s["cb_dim"])),
          ("up.weight", (s["dim"], 1, s["up_kernel"]))]
    d, f = s["dim"], s["ffn"]
    for l in range(s["n_layers"]):
        p = f"tr.{l}."
        t += [(p + "norm1.w", (d,)), (p + "norm1.b", (d,)), (p + "in_proj", (3 * d, d)), (p + "out_proj", (d, d)),
              (p + "scale1", (d,)), (p + "norm2.w", (d,)), (p + "norm2.b", (d,)), (p + "lin1", (f, d)),
              (p + "lin2", (d, f)), (p + "scale2", (d,))]
    C = s["n_filters"] * 2 ** len(s["ratios"])
    t += [("dec.0.w", (C, d, s["kernel"])), ("dec.0.b", (C,))]
    for i, r in enumerate(s["ratios"]):
        co = C // 2
        h = co // s["compress"]
        t += [(f"dec.up{i}.w", (C, co, 2 * r)), (f"dec.up{i}.b", (co,)), (f"dec.res{i}.w1", (h, co, s["res_kernel"])),
              (f"dec.res{i}.b1", (h,)), (f"dec.res{i}.w2", (co, h, 1)), (f"dec.res{i}.b2", (co,))]
        C = co
    return t + [("dec.out.w", (1, C, s["last_kernel"])), ("dec.out.b", (1,))]


def make_mimi_weights(shape: dict, base_seed: int = 5000, layer_scale: float = 0.05,
                      threads: int | None = None) -> Dict[str, np.ndarray]:
    """bf16 bits of every decoder tensor: codebooks N(0, 1); LayerNorm weights
    1 + 0.1 N(0, 1); LayerScale layer_scale (1 + 0.1 N(0, 1)); biases (LayerNorm biases
    included) N(0, 0.02); matrices and kernels N(0, 1 / fan), fan = the product of all
    dimensions after the first (so activations keep their scale through the stack).
    Tensor i of the canonical order gets seed base_seed + i."""
    threads = threads or min(32, os.cpu_count() or 1)
    out: Dict[str, np.ndarray] = {}
    with ThreadPoolExecutor(threads) as pool:
        for i, (name, sh) in enumerate(mimi_tensor_specs(shape)):
            if name.startswith("q.codebook"):
                mean, std = 0.0, 1.0
            elif name.endswith(("norm1.w", "norm2.w")):
                mean, std = 1.0, 0.1
            elif name.endswith(("scale1", "scale2")):
                mean, std = layer_scale, 0.1 * layer_scale
            elif len(sh) == 1:
                mean, std = 0.0, 0.02
            else:
                mean, std = 0.0, float(1.0 / np.sqrt(np.prod(sh[1:])))
            out[name] = normal_bf16(sh, mean, std, base_seed + i, pool)
    return out


def make_mimi_codes(shape: dict, T: int, B: int = 1, seed: int = 6000) -> np.ndarray:
    """Code frames [T][B][n_q], each code uniform over 0..card-1."""
    s = dict(MIMI_FULL)
    s.update(shape)
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, T, B])))
    return g.integers(0, s["card"], size=(T, B, s["n_q"]), dtype=np.int64).astype(np.int32)


def mimi_encoder_tensor_specs(shape: dict) -> List[Tuple[str, Tuple[int, ...]]]:
    """Names and shapes of the encoder's tensors in their canonical order: the SEANet
    encoder (stages in the reversed ratio order), the encoder transformer, the latent
    downsampler, the quantizer input projections, then the codebooks."""
    s = dict(MIMI_FULL)
    s.update(shape)
    d, f, C = s["dim"], s["ffn"], s["n_filters"]
    t = [("enc.0.w", (C, 1, s["kernel"])), ("enc.0.b", (C,))]
    for i, r in enumerate(reversed(s["ratios"])):
        h = C // s["compress"]
        t += [(f"enc.res{i}.w1", (h, C, s["res_kernel"])), (f"enc.res{i}.b1", (h,)), (f"enc.res{i}.w2", (C, h, 1)),
              (f"enc.res{i}.b2", (C,)), (f"enc.down{i}.w", (2 * C, C, 2 * r)), (f"enc.down{i}.b", (2 * C,))]
        C *= 2
    t += [("enc.out.w", (d, C, s["last_kernel"])), ("enc.out.b", (d,))]
    for l in range(s["n_layers"]):
        p = f"etr.{l}."
        t += [(p + "norm1.w", (d,)), (p + "norm1.b", (d,)), (p + "in_proj", (3 * d, d)), (p + "out_proj", (d, d)),
              (p + "scale1", (d,)), (p + "norm2.w", (d,)), (p + "norm2.b", (d,)), (p + "lin1", (f, d)),
              (p + "lin2", (d, f)), (p + "scale2", (d,))]
    t += [("ds.weight", (d, d, s["up_kernel"])), ("q.sem.in", (s["cb_dim"], d)), ("q.ac.in", (s["cb_dim"], d))]
    return t + [(f"q.codebook.{j}", (s["card"], s["cb_dim"])) for j in range(s["n_q"])]


def make_mimi_encoder_weights(shape: dict, base_seed: int = 7000, codebook_seed: int = 5000,
                              layer_scale: float = 0.05, threads: int | None = None) -> Dict[str, np.ndarray]:
    """bf16 bits of every encoder tensor with the distributions of make_mimi_weights; tensor
    i of the encoder order gets seed base_seed + i, except the codebooks, drawn exactly as
    make_mimi_weights(shape, codebook_seed) draws them, so that one set of tables serves the
    encoder and the decoder."""
    threads = threads or min(32, os.cpu_count() or 1)
    out: Dict[str, np.ndarray] = {}
    with ThreadPoolExecutor(threads) as pool:
        for i, (name, sh) in enumerate(mimi_encoder_tensor_specs(shape)):
            if name.startswith("q.codebook"):
                out[name] = normal_bf16(sh, 0.0, 1.0, codebook_seed + int(name.rsplit(".", 1)[1]), pool)
                continue
            if name.endswith(("norm1.w", "norm2.w")):
                mean, std = 1.0, 0.1
            elif name.endswith(("scale1", "scale2")):
                mean, std = layer_scale, 0.1 * layer_scale
            elif len(sh) == 1:
                mean, std = 0.0, 0.02
            else:
                mean, std = 0.0, float(1.0 / np.sqrt(np.prod(sh[1:])))
            out[name] = normal_bf16(sh, mean, std, base_seed + i, pool)
    return out


def make_mimi_pcm(n_samples: int, B: int = 1, seed: int = 8000, rate: int = 24000) -> np.ndarray:
    """Seeded speech-band stand-in [B][n_samples] float32: per stream five sines (80-3000 Hz,
    amplitudes 0.02-0.2, random phases) under a 3 Hz syllable-rate envelope, plus white noise
    of standard deviation 0.01."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, n_samples, B])))
    t = np.arange(n_samples) / rate
    out = np.zeros((B, n_samples))
    for b in range(B):
        f = g.uniform(80.0, 3000.0, 5)
        a = g.uniform(0.02, 0.2, 5)
        ph = g.uniform(0.0, 2 * np.pi, 5)
        env = 0.6 + 0.4 * np.sin(2 * np.pi * 3.0 * t + g.uniform(0.0, 2 * np.pi))
        out[b] = env * (a[:, None] * np.sin(2 * np.pi * f[:, None] * t[None, :] + ph[:, None])).sum(0)
        out[b] += 0.01 * g.standard_normal(n_samples)
    return out.astype(np.float32)
