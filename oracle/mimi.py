"""Float64 statement of the Mimi decoder: codes -> 24 kHz PCM.

TEST INFRASTRUCTURE ONLY: used by the tests and the bench's CPU leg, never by the library.

Follows "PersonaPlex native LM audit", chapter "Exact Mimi codec construction":
  - "Complete encode/decode order" (DECODE): semantic code lookup -> semantic output
    projection 256 -> 512, plus the sum of the seven acoustic lookups -> acoustic output
    projection; learned depthwise ConvTranspose1d 512 -> 512, kernel 4, stride 2, no bias;
    decoder transformer; SEANet decoder;
  - "Split quantizer: exact paths and active capacity": decoded = W_sem,out e0[code0] +
    W_ac,out sum_{j=1..7} e_j[code_j], output projections bias-free [512, 256];
  - "Both codec transformer stacks": per block LayerNorm(512, eps 1e-5) -> multi-head
    self-attention (8 heads x 64, bias-free in/out projections) -> LayerScale -> + x ->
    LayerNorm -> Linear 512 -> 2048 -> GELU -> Linear 2048 -> 512 -> LayerScale -> +;
    causal, window 0 <= q - k < 250, RoPE max period 10000;
  - "SEANet decoder, every stage": D0 Conv1d 512 -> 1024 k7; per stage (ratios 8, 6, 5,
    4) ELU -> ConvTranspose1d (C -> C/2, kernel 2r, stride r) then the residual block
    x + Conv(C/2, C, k1)(ELU(Conv(C, C/2, k3)(ELU(x)))); D5 ELU -> Conv1d 64 -> 1 k3; no
    final activation; every convolution has a bias, dilation 1, groups 1;
  - "Stateful streaming, padding and dependency boundaries": causal convolutions pad
    kernel - stride zeros on the left; causal transposed convolutions trim kernel - stride
    positions from the right.  Streaming emits exactly these values frame by frame.

and the ENCODE order of the same chapter:
  - "SEANet encoder, every stage": E0 Conv1d 1 -> 64 k7; per stage (the loader's ratios
    reversed: 4, 5, 6, 8) the residual block x + Conv(C/2, C, k1)(ELU(Conv(C, C/2, k3)(ELU(x))))
    then ELU -> Conv1d C -> 2C, kernel 2r, stride r; E5 ELU -> Conv1d 1024 -> 512 k3; every
    convolution with a bias;
  - the encoder transformer (a separate stack of the same construction);
  - "Learned resampling around the quantizer": Conv1d 512 -> 512, kernel 4, stride 2, no
    bias, causal left padding of 2 positions by replicating the first position;
  - "Split quantizer": the same latent through the semantic input projection (256 x 512,
    bias-free) to the nearest vector of codebook 0, and through the acoustic input projection
    to a residual chain over codebooks 1..7 (code_j = nearest to r_{j-1}, r_j = r_{j-1} -
    e_j[code_j]); semantic then acoustic indices.
  - "Stateful streaming, padding and dependency boundaries": a strided causal convolution
    pads kernel - stride zeros on the left (the SEANet convolutions) or replicates the first
    position (the latent downsampler).

These are the non-streaming causal computations over whole sequences; streaming encoders
and decoders must reproduce them frame by frame.  Readings where the chapter is silent:
RoPE rotates adjacent coordinate pairs (2j, 2j+1) of each 64-wide head with frequencies
exp(-ln(10000) * 2j / 64), as the temporal transformer's RoPE is described; the
attention scale is 1/sqrt(64); GELU is the exact erf form; ELU has alpha 1; the
transformer positions count the 25 Hz grid from 0 at reset; the codebooks are used as
given tables [2048][256] (the effective vectors of the quantizer's state); "nearest" is the
smallest Euclidean distance, the lowest index on an exact tie.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, asdict
from typing import Dict, List, Sequence, Tuple

import numpy as np


@dataclass
class MimiShape:
    dim: int = 512          # latent / transformer width
    cb_dim: int = 256       # codebook vector width
    card: int = 2048        # entries per codebook
    n_q: int = 8            # active codebooks: 1 semantic + 7 acoustic
    n_layers: int = 8
    heads: int = 8
    ffn: int = 2048
    ctx: int = 250          # attention window (positions)
    n_filters: int = 64
    ratios: List[int] = field(default_factory=lambda: [8, 6, 5, 4])
    kernel: int = 7         # D0
    last_kernel: int = 3    # D5
    res_kernel: int = 3
    compress: int = 2
    up_kernel: int = 4      # latent upsampler 12.5 -> 25 Hz
    up_stride: int = 2
    ln_eps: float = 1e-5
    rope_theta: float = 1e4

    @property
    def hop(self) -> int:
        return int(np.prod(self.ratios))

    @property
    def frame_samples(self) -> int:
        return self.hop * self.up_stride

    def asdict(self) -> dict:
        return asdict(self)


def tensor_specs(s: MimiShape) -> List[Tuple[str, Tuple[int, ...]]]:
    """Canonical decoder tensors: name and shape (PyTorch layouts: Conv1d [out, in, k],
    ConvTranspose1d [in, out/groups, k], Linear [out, in])."""
    t = [("q.codebook.0", (s.card, s.cb_dim))]
    t += [(f"q.codebook.{j}", (s.card, s.cb_dim)) for j in range(1, s.n_q)]
    t += [("q.sem.out", (s.dim, s.cb_dim)), ("q.ac.out", (s.dim, s.cb_dim)),
          ("up.weight", (s.dim, 1, s.up_kernel))]
    for l in range(s.n_layers):
        p = f"tr.{l}."
        t += [(p + "norm1.w", (s.dim,)), (p + "norm1.b", (s.dim,)), (p + "in_proj", (3 * s.dim, s.dim)),
              (p + "out_proj", (s.dim, s.dim)), (p + "scale1", (s.dim,)), (p + "norm2.w", (s.dim,)),
              (p + "norm2.b", (s.dim,)), (p + "lin1", (s.ffn, s.dim)), (p + "lin2", (s.dim, s.ffn)),
              (p + "scale2", (s.dim,))]
    C = s.n_filters * 2 ** len(s.ratios)
    t += [("dec.0.w", (C, s.dim, s.kernel)), ("dec.0.b", (C,))]
    for i, r in enumerate(s.ratios):
        co = C // 2
        h = co // s.compress
        t += [(f"dec.up{i}.w", (C, co, 2 * r)), (f"dec.up{i}.b", (co,)),
              (f"dec.res{i}.w1", (h, co, s.res_kernel)), (f"dec.res{i}.b1", (h,)),
              (f"dec.res{i}.w2", (co, h, 1)), (f"dec.res{i}.b2", (co,))]
        C = co
    t += [("dec.out.w", (1, C, s.last_kernel)), ("dec.out.b", (1,))]
    return t


def encoder_tensor_specs(s: MimiShape) -> List[Tuple[str, Tuple[int, ...]]]:
    """Canonical encoder tensors (same layout conventions): the SEANet encoder, the encoder
    transformer, the latent downsampler, the two quantizer input projections, then the
    codebooks the decoder also reads."""
    t = [("enc.0.w", (s.n_filters, 1, s.kernel)), ("enc.0.b", (s.n_filters,))]
    C = s.n_filters
    for i, r in enumerate(reversed(s.ratios)):
        h = C // s.compress
        t += [(f"enc.res{i}.w1", (h, C, s.res_kernel)), (f"enc.res{i}.b1", (h,)), (f"enc.res{i}.w2", (C, h, 1)),
              (f"enc.res{i}.b2", (C,)), (f"enc.down{i}.w", (2 * C, C, 2 * r)), (f"enc.down{i}.b", (2 * C,))]
        C *= 2
    t += [("enc.out.w", (s.dim, C, s.last_kernel)), ("enc.out.b", (s.dim,))]
    for l in range(s.n_layers):
        p = f"etr.{l}."
        t += [(p + "norm1.w", (s.dim,)), (p + "norm1.b", (s.dim,)), (p + "in_proj", (3 * s.dim, s.dim)),
              (p + "out_proj", (s.dim, s.dim)), (p + "scale1", (s.dim,)), (p + "norm2.w", (s.dim,)),
              (p + "norm2.b", (s.dim,)), (p + "lin1", (s.ffn, s.dim)), (p + "lin2", (s.dim, s.ffn)),
              (p + "scale2", (s.dim,))]
    t += [("ds.weight", (s.dim, s.dim, s.up_kernel)), ("q.sem.in", (s.cb_dim, s.dim)), ("q.ac.in", (s.cb_dim, s.dim))]
    t += [(f"q.codebook.{j}", (s.card, s.cb_dim)) for j in range(s.n_q)]
    return t


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------------------------
# scalar steps
# ------------------------------------------------------------------------------------

def elu(x: np.ndarray) -> np.ndarray:
    return np.where(x > 0, x, np.expm1(np.minimum(x, 0.0)))


def gelu(x: np.ndarray) -> np.ndarray:
    erf = np.vectorize(math.erf)
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def layer_norm(x: np.ndarray, w: np.ndarray, b: np.ndarray, eps: float) -> np.ndarray:
    """x [..., n]: (x - mean) / sqrt(var + eps) * w + b, biased variance."""
    m = x.mean(-1, keepdims=True)
    v = ((x - m) ** 2).mean(-1, keepdims=True)
    return (x - m) / np.sqrt(v + eps) * w + b


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate adjacent pairs (2j, 2j+1) of a head vector by pos * exp(-ln(theta) 2j / d)."""
    d = v.shape[-1]
    out = v.copy()
    for j in range(d // 2):
        a = pos * math.exp(-math.log(theta) * 2 * j / d)
        c, s_ = math.cos(a), math.sin(a)
        x0, x1 = v[..., 2 * j], v[..., 2 * j + 1]
        out[..., 2 * j] = x0 * c - x1 * s_
        out[..., 2 * j + 1] = x0 * s_ + x1 * c
    return out


def conv1d_causal(x: np.ndarray, w: np.ndarray, b: np.ndarray) -> np.ndarray:
    """x [Cin][T], w [Cout][Cin][k], stride 1: y[t] = b + sum_j w[:, :, j] x[t - (k-1) + j],
    zeros before the first sample."""
    k = w.shape[2]
    T = x.shape[1]
    xp = np.concatenate([np.zeros((x.shape[0], k - 1)), x], axis=1)
    y = np.zeros((w.shape[0], T))
    for j in range(k):
        y += w[:, :, j] @ xp[:, j:j + T]
    return y + b[:, None]


def convtr_causal(x: np.ndarray, w: np.ndarray, b: np.ndarray, stride: int) -> np.ndarray:
    """x [Cin][T], w [Cin][Cout][k]: the full transposed convolution (input t adds
    w[:, :, j]^T x[t] at output t * stride + j, length (T - 1) stride + k), trimmed by
    k - stride on the right (length T * stride), plus the bias."""
    k = w.shape[2]
    T = x.shape[1]
    full = np.zeros((w.shape[1], (T - 1) * stride + k))
    for j in range(k):
        full[:, j:j + (T - 1) * stride + 1:stride] += w[:, :, j].T @ x
    return full[:, :T * stride] + b[:, None]


def convtr_depthwise_causal(x: np.ndarray, w: np.ndarray, stride: int) -> np.ndarray:
    """Depthwise (groups = channels) transposed convolution without bias, trimmed the same
    way: x [C][T], w [C][1][k]."""
    k = w.shape[2]
    T = x.shape[1]
    full = np.zeros((x.shape[0], (T - 1) * stride + k))
    for j in range(k):
        full[:, j:j + (T - 1) * stride + 1:stride] += w[:, 0, j][:, None] * x
    return full[:, :T * stride]


def rvq_decode(codebooks: Sequence[np.ndarray], codes: Sequence[int]) -> np.ndarray:
    """Sum of the looked-up vectors of one residual quantizer."""
    out = np.zeros(codebooks[0].shape[1])
    for cb, c in zip(codebooks, codes):
        out = out + cb[int(c)]
    return out


def conv1d_causal_strided(x: np.ndarray, w: np.ndarray, b, stride: int, replicate: bool = False) -> np.ndarray:
    """x [Cin][T] (T a multiple of stride), w [Cout][Cin][k]: left padding of k - stride
    positions (zeros, or copies of the first position), then y[t] = b + sum_j w[:, :, j]
    x_pad[t * stride + j] for t < T / stride."""
    k = w.shape[2]
    T = x.shape[1]
    pad = np.repeat(x[:, :1], k - stride, axis=1) if replicate else np.zeros((x.shape[0], k - stride))
    xp = np.concatenate([pad, x], axis=1)
    n = T // stride
    y = np.zeros((w.shape[0], n))
    for j in range(k):
        y += w[:, :, j] @ xp[:, j:j + (n - 1) * stride + 1:stride]
    return y if b is None else y + b[:, None]


def nearest(codebook: np.ndarray, v: np.ndarray) -> Tuple[int, float]:
    """Index of the codebook row nearest to v (lowest index on an exact tie) and the gap
    between the second-smallest and the smallest squared distance."""
    d = ((codebook - v[None, :]) ** 2).sum(axis=1)
    i = int(np.argmin(d))
    return i, float(np.partition(d, 1)[1] - d[i]) if len(d) > 1 else float("inf")


def rvq_encode(codebooks: Sequence[np.ndarray], v: np.ndarray, forced: Sequence[int] = None):
    """Residual quantisation of v: per level the nearest row to the current residual, then
    the residual minus that row.  forced[j] >= 0 takes that code instead (the caller's choice
    at a near tie).  Returns (codes, gaps, final residual)."""
    r = np.array(v, dtype=np.float64)
    codes, gaps = [], []
    for j, cb in enumerate(codebooks):
        i, g = nearest(cb, r)
        if forced is not None and forced[j] >= 0:
            i = int(forced[j])
        codes.append(i)
        gaps.append(g)
        r = r - cb[i]
    return codes, gaps, r


def transformer_stack(W: Dict[str, np.ndarray], prefix: str, s: MimiShape, x: np.ndarray) -> np.ndarray:
    """One codec transformer stack ("Both codec transformer stacks") over x [dim][T] at 25 Hz,
    positions 0..T-1 -> [dim][T]."""
    X = x.T.copy()  # [T][dim]
    T = X.shape[0]
    H, dh = s.heads, s.dim // s.heads
    for l in range(s.n_layers):
        p = f"{prefix}{l}."
        u = layer_norm(X, W[p + "norm1.w"], W[p + "norm1.b"], s.ln_eps)
        qkv = u @ W[p + "in_proj"].T
        q, k, v = qkv[:, :s.dim], qkv[:, s.dim:2 * s.dim], qkv[:, 2 * s.dim:]
        o = np.zeros((T, s.dim))
        for h in range(H):
            sl = slice(h * dh, (h + 1) * dh)
            qh = np.stack([rope(q[t, sl], t, s.rope_theta) for t in range(T)])
            kh = np.stack([rope(k[t, sl], t, s.rope_theta) for t in range(T)])
            for t in range(T):
                lo = max(0, t - s.ctx + 1)
                sc = kh[lo:t + 1] @ qh[t] / math.sqrt(dh)
                pr = np.exp(sc - sc.max())
                pr /= pr.sum()
                o[t, sl] = pr @ v[lo:t + 1, sl]
        X = X + (o @ W[p + "out_proj"].T) * W[p + "scale1"]
        u = layer_norm(X, W[p + "norm2.w"], W[p + "norm2.b"], s.ln_eps)
        f = gelu(u @ W[p + "lin1"].T) @ W[p + "lin2"].T
        X = X + f * W[p + "scale2"]
    return X.T


# ------------------------------------------------------------------------------------
# the decoder
# ------------------------------------------------------------------------------------

class MimiDecoderOracle:
    def __init__(self, shape: MimiShape, weights_bf16: Dict[str, np.ndarray]):
        self.s = shape
        self.W = {n: bf16_to_f64(weights_bf16[n]).reshape(sh) for n, sh in tensor_specs(shape)}

    def latent(self, codes: np.ndarray) -> np.ndarray:
        """codes [T][n_q] -> latent [dim][T] at 12.5 Hz (split quantizer decode)."""
        s, W = self.s, self.W
        cbs = [W[f"q.codebook.{j}"] for j in range(s.n_q)]
        out = np.zeros((s.dim, codes.shape[0]))
        for t in range(codes.shape[0]):
            sem = rvq_decode(cbs[:1], codes[t, :1])
            ac = rvq_decode(cbs[1:], codes[t, 1:])
            out[:, t] = W["q.sem.out"] @ sem + W["q.ac.out"] @ ac
        return out

    def transformer(self, x: np.ndarray) -> np.ndarray:
        """x [dim][T] at 25 Hz, positions 0..T-1 -> [dim][T]."""
        return transformer_stack(self.W, "tr.", self.s, x)

    def seanet(self, z: np.ndarray) -> np.ndarray:
        """z [dim][T] at 25 Hz -> PCM [T * hop]."""
        s, W = self.s, self.W
        x = conv1d_causal(z, W["dec.0.w"], W["dec.0.b"])
        for i, r in enumerate(s.ratios):
            x = convtr_causal(elu(x), W[f"dec.up{i}.w"], W[f"dec.up{i}.b"], r)
            y = conv1d_causal(elu(x), W[f"dec.res{i}.w1"], W[f"dec.res{i}.b1"])
            x = x + conv1d_causal(elu(y), W[f"dec.res{i}.w2"], W[f"dec.res{i}.b2"])
        return conv1d_causal(elu(x), W["dec.out.w"], W["dec.out.b"])[0]

    def decode(self, codes: np.ndarray) -> np.ndarray:
        """codes [T][n_q] (frames from reset) -> PCM [T * frame_samples]."""
        codes = np.asarray(codes)
        lat = self.latent(codes)
        up = convtr_depthwise_causal(lat, self.W["up.weight"], self.s.up_stride)
        return self.seanet(self.transformer(up))


# ------------------------------------------------------------------------------------
# the encoder
# ------------------------------------------------------------------------------------

class MimiEncoderOracle:
    def __init__(self, shape: MimiShape, weights_bf16: Dict[str, np.ndarray]):
        self.s = shape
        self.W = {n: bf16_to_f64(weights_bf16[n]).reshape(sh) for n, sh in encoder_tensor_specs(shape)}

    def seanet(self, pcm: np.ndarray) -> np.ndarray:
        """PCM [N] (N a multiple of the hop) -> [dim][N / hop] at 25 Hz."""
        s, W = self.s, self.W
        x = conv1d_causal(np.asarray(pcm, np.float64)[None, :], W["enc.0.w"], W["enc.0.b"])
        for i, r in enumerate(reversed(s.ratios)):
            y = conv1d_causal(elu(x), W[f"enc.res{i}.w1"], W[f"enc.res{i}.b1"])
            x = x + conv1d_causal(elu(y), W[f"enc.res{i}.w2"], W[f"enc.res{i}.b2"])
            x = conv1d_causal_strided(elu(x), W[f"enc.down{i}.w"], W[f"enc.down{i}.b"], r)
        return conv1d_causal(elu(x), W["enc.out.w"], W["enc.out.b"])

    def transformer(self, x: np.ndarray) -> np.ndarray:
        return transformer_stack(self.W, "etr.", self.s, x)

    def downsample(self, x: np.ndarray) -> np.ndarray:
        """[dim][T] at 25 Hz -> [dim][T / 2] at 12.5 Hz (replicated left padding, no bias)."""
        return conv1d_causal_strided(x, self.W["ds.weight"], None, self.s.up_stride, replicate=True)

    def latent(self, pcm: np.ndarray) -> np.ndarray:
        """PCM [N] (N a multiple of the frame) -> the unquantised latent [F][dim]."""
        return self.downsample(self.transformer(self.seanet(pcm))).T

    def quantize(self, e: np.ndarray, forced: Sequence[int] = None):
        """One latent [dim] -> (codes [n_q], gaps [n_q]): codebook 0 on the semantic
        projection, codebooks 1.. as a residual chain on the acoustic projection."""
        s, W = self.s, self.W
        cbs = [W[f"q.codebook.{j}"] for j in range(s.n_q)]
        f0 = None if forced is None else forced[:1]
        fa = None if forced is None else forced[1:]
        c0, g0, _ = rvq_encode(cbs[:1], W["q.sem.in"] @ e, f0)
        ca, ga, _ = rvq_encode(cbs[1:], W["q.ac.in"] @ e, fa)
        return c0 + ca, g0 + ga

    def encode(self, pcm: np.ndarray) -> np.ndarray:
        """PCM [N] from reset -> codes [F][n_q]."""
        return np.array([self.quantize(e)[0] for e in self.latent(pcm)], dtype=np.int64)
