"""Pins of the Mimi decoder oracle (oracle/mimi.py) against what the pages and the
mathematics fix:

- tensor shapes: the decoder groups sum to the page's printed parameter totals
  (tests/golden/mimi_inventory.json);
- residual VQ decode: the explainer's worked 3-level example reconstructs x exactly from
  its codes (tests/golden/rvq_worked_example.json);
- causal convolution: a single channel equals numpy.convolve truncated to the causal
  part; a delta kernel at tap j delays by k-1-j samples;
- causal transposed convolution: equals numpy.convolve of the zero-stuffed input, trimmed
  to T * stride; the depthwise upsampler is the per-channel case;
- ELU, GELU, LayerNorm closed forms; RoPE keeps pair norms and turns (1, 0) by exactly
  pos radians in pair 0;
- attention: a one-position sequence passes v through; the window: a key ctx positions
  back has no effect;
- the decoder is causal: decoding T + 2 frames reproduces the first T frames' samples;
- encoder: the SEANet encoder, the encoder transformer and the dense downsampler sum to
  the page's totals; the explainer's worked example quantises to its printed codes and
  residual norms; a strided causal convolution equals the subsampled truncated
  convolution (zero padding) and the replicate-padded downsampler repeats the first
  position; exact ties take the lowest index; the acoustic chain does not depend on the
  semantic branch; the encoder is causal frame by frame.
"""
import json
import math
import os

import numpy as np

from oracle import mimi as M

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf16(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def tiny_mimi_shape(**over):
    base = dict(dim=64, cb_dim=32, card=16, n_q=8, n_layers=2, heads=2, ffn=128, ctx=6, n_filters=4,
                ratios=[4, 3], kernel=7, last_kernel=3, res_kernel=3, compress=2)
    base.update(over)
    return M.MimiShape(**base)


def random_weights(s, seed=1, ls=0.05, specs=None):
    rng = np.random.default_rng(seed)
    W = {}
    for n, sh in (specs if specs is not None else M.tensor_specs(s)):
        if n.startswith("q.codebook"):
            v = rng.standard_normal(sh)
        elif n.endswith(("norm1.w", "norm2.w")):
            v = 1 + 0.1 * rng.standard_normal(sh)
        elif n.endswith(("scale1", "scale2")):
            v = ls * (1 + 0.1 * rng.standard_normal(sh))
        elif len(sh) == 1:
            v = 0.02 * rng.standard_normal(sh)
        else:
            fan = sh[1] * (sh[2] if len(sh) == 3 else 1)
            v = rng.standard_normal(sh) / math.sqrt(fan)
        W[n] = _bf16(v)
    return W


def test_decoder_shapes_match_the_page_inventory():
    g = json.load(open(os.path.join(GOLDEN, "mimi_inventory.json")))
    s = M.MimiShape()
    specs = dict(M.tensor_specs(s))
    n = lambda pred: sum(int(np.prod(sh)) for k, sh in specs.items() if pred(k))
    assert n(lambda k: k.startswith("dec.")) == g["seanet_decoder_params"]
    assert n(lambda k: k.startswith("tr.")) == g["decoder_transformer_params"]
    assert n(lambda k: k.startswith("tr.0.")) == g["transformer_block_params"]
    # the decoder's two output projections are half of the four quantizer projections
    assert 2 * n(lambda k: k in ("q.sem.out", "q.ac.out")) == g["four_quantizer_projections_params"]
    assert n(lambda k: k == "up.weight") == g["depthwise_upsampler_params"]
    assert specs["q.codebook.0"] == (g["codebook_entries"], g["codebook_dim"])
    assert s.frame_samples == 1920 and s.hop == 960   # 24 kHz / 12.5 Hz, 24 kHz / 25 Hz


def test_rvq_decode_reconstructs_the_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "rvq_worked_example.json")))
    books = [np.array(c, np.float64) for c in g["codebooks"]]
    rec = M.rvq_decode(books, g["codes_zero_based"])
    assert np.allclose(rec, g["reconstruction"], atol=1e-15)
    # and the residual norms after each level, as printed (4 decimals)
    x = np.array(g["x"])
    r = x.copy()
    for lvl, (cb, c) in enumerate(zip(books, g["codes_zero_based"])):
        assert int(((cb - r) ** 2).sum(1).argmin()) == c
        r = r - cb[c]
        assert abs(np.linalg.norm(r) - g["error_norms"][lvl]) < 5e-5


def test_conv1d_causal_is_truncated_convolution():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 23))
    w = rng.standard_normal((1, 1, 7))
    y = M.conv1d_causal(x, w, np.zeros(1))[0]
    # y[t] = sum_j w[j] x[t - 6 + j]  ==  (x * reversed w)[t] of the full convolution
    ref = np.convolve(x[0], w[0, 0][::-1])[:23]
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-13)
    # a delta at tap j delays by k - 1 - j; the bias is added everywhere
    for j in range(7):
        d = np.zeros((1, 1, 7))
        d[0, 0, j] = 1.0
        y = M.conv1d_causal(x, d, np.array([0.5]))[0]
        sh = 6 - j
        assert np.allclose(y[sh:], x[0, :23 - sh] + 0.5) and np.allclose(y[:sh], 0.5)


def test_convtr_causal_is_upsampled_convolution():
    rng = np.random.default_rng(4)
    for k, st in ((16, 8), (12, 6), (10, 5), (8, 4), (4, 2)):
        x = rng.standard_normal((1, 9))
        w = rng.standard_normal((1, 1, k))
        y = M.convtr_causal(x, w, np.zeros(1), st)[0]
        z = np.zeros(9 * st)
        z[::st] = x[0]
        ref = np.convolve(z, w[0, 0])[:9 * st]
        assert y.shape == (9 * st,) and np.allclose(y, ref, rtol=1e-13, atol=1e-13)
        # multi-channel: channel mixing is w[ci, co, j]^T
        x2 = rng.standard_normal((3, 5))
        w2 = rng.standard_normal((3, 2, k))
        y2 = M.convtr_causal(x2, w2, np.zeros(2), st)
        for co in range(2):
            acc = np.zeros(5 * st)
            for ci in range(3):
                zz = np.zeros(5 * st)
                zz[::st] = x2[ci]
                acc += np.convolve(zz, w2[ci, co])[:5 * st]
            assert np.allclose(y2[co], acc, rtol=1e-12, atol=1e-12)
    # depthwise: channel c alone with its own taps
    x = rng.standard_normal((4, 6))
    w = rng.standard_normal((4, 1, 4))
    y = M.convtr_depthwise_causal(x, w, 2)
    for c in range(4):
        assert np.allclose(y[c], M.convtr_causal(x[c:c + 1], w[c:c + 1], np.zeros(1), 2)[0])


def test_pointwise_closed_forms():
    assert M.elu(np.array([2.0]))[0] == 2.0
    assert abs(M.elu(np.array([math.log(0.5)]))[0] + 0.5) < 1e-15
    assert abs(M.elu(np.array([-50.0]))[0] + 1.0) < 1e-15
    g = M.gelu(np.array([0.0, 1.3, -1.3, 3.0]))
    assert g[0] == 0.0 and abs((g[1] - g[2]) - 1.3) < 1e-15     # GELU(x) - GELU(-x) = x
    assert abs(g[3] - 3.0 * 0.5 * (1 + math.erf(3.0 / math.sqrt(2)))) < 1e-15
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, 40)) * 4 + 2
    y = M.layer_norm(x, np.ones(40), np.zeros(40), 0.0)
    assert np.allclose(y.mean(-1), 0, atol=1e-13) and np.allclose((y ** 2).mean(-1), 1, atol=1e-12)
    c = M.layer_norm(np.full((1, 8), 3.0), np.full(8, 2.0), np.full(8, 0.25), 1e-5)
    assert np.allclose(c, 0.25)                                     # a constant row -> the bias
    v = rng.standard_normal(64)
    r = M.rope(v, 7, 1e4)
    assert np.allclose(np.hypot(r[0::2], r[1::2]), np.hypot(v[0::2], v[1::2]))
    e = np.zeros(64)
    e[0] = 1.0
    r = M.rope(e, 5, 1e4)
    assert abs(r[0] - math.cos(5)) < 1e-15 and abs(r[1] - math.sin(5)) < 1e-15 and np.all(r[2:] == 0)


def test_attention_single_position_and_window():
    s = tiny_mimi_shape(n_layers=1, ctx=3)
    W = random_weights(s, seed=6)
    # zero out the FFN so the block is x + scale * attention
    W["tr.0.lin2"][...] = 0
    O = M.MimiDecoderOracle(s, W)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((s.dim, 1))
    y = O.transformer(x)
    Wd = O.W
    u = M.layer_norm(x.T, Wd["tr.0.norm1.w"], Wd["tr.0.norm1.b"], s.ln_eps)
    v = (u @ Wd["tr.0.in_proj"].T)[:, 2 * s.dim:]
    assert np.allclose(y.T, x.T + (v @ Wd["tr.0.out_proj"].T) * Wd["tr.0.scale1"], rtol=1e-12, atol=1e-12)
    # a position ctx or more steps back never changes the output
    x = rng.standard_normal((s.dim, 8))
    y = O.transformer(x)
    x2 = x.copy()
    x2[:, 1] += 5.0
    y2 = O.transformer(x2)
    assert np.array_equal(y[:, 4:], y2[:, 4:]) and not np.allclose(y[:, 1:4], y2[:, 1:4])


def test_decoder_is_causal_frame_by_frame():
    s = tiny_mimi_shape()
    O = M.MimiDecoderOracle(s, random_weights(s, seed=8))
    codes = np.random.default_rng(9).integers(0, s.card, (5, s.n_q))
    a = O.decode(codes[:3])
    b = O.decode(codes)
    assert a.shape == (3 * s.frame_samples,) and b.shape == (5 * s.frame_samples,)
    assert np.allclose(a, b[:a.size], rtol=0, atol=1e-12 * np.abs(b).max())  # (BLAS blocking may differ)
    assert np.all(np.isfinite(b)) and np.std(b) > 0


# ------------------------------------------------------------------------------------
# encoder
# ------------------------------------------------------------------------------------

def test_encoder_shapes_match_the_page_inventory():
    g = json.load(open(os.path.join(GOLDEN, "mimi_inventory.json")))
    s = M.MimiShape()
    specs = dict(M.encoder_tensor_specs(s))
    n = lambda pred: sum(int(np.prod(sh)) for k, sh in specs.items() if pred(k))
    assert n(lambda k: k.startswith("enc.")) == g["seanet_encoder_params"]
    assert n(lambda k: k.startswith("etr.")) == g["encoder_transformer_params"]
    assert n(lambda k: k == "ds.weight") == g["dense_latent_downsampler_params"]
    # the encoder's two input projections are the other half of the four projections
    assert 2 * n(lambda k: k in ("q.sem.in", "q.ac.in")) == g["four_quantizer_projections_params"]
    # the encoder downsamples by the reversed ratios: 4, 5, 6, 8
    assert [specs[f"enc.down{i}.w"][2] // 2 for i in range(4)] == [4, 5, 6, 8]


def test_rvq_encode_reproduces_the_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "rvq_worked_example.json")))
    books = [np.array(c, np.float64) for c in g["codebooks"]]
    codes, gaps, r = M.rvq_encode(books, np.array(g["x"]))
    assert codes == g["codes_zero_based"]
    assert np.allclose(np.array(g["x"]) - r, g["reconstruction"], atol=1e-15)
    assert np.linalg.norm(r) < 1e-15 and all(gg > 0 for gg in gaps)
    # a forced code replaces the choice and the chain continues from it
    codes2, _, r2 = M.rvq_encode(books, np.array(g["x"]), forced=[1, -1, -1])
    assert codes2[0] == 1 and np.allclose(r2, np.array(g["x"]) - books[0][1] - books[1][codes2[1]] - books[2][codes2[2]])


def test_nearest_takes_the_lowest_index_on_an_exact_tie():
    cb = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 0.0], [0.0, 1.0]])
    assert M.nearest(cb, np.array([0.0, 1.0]))[0] == 1
    i, gap = M.nearest(cb, np.array([0.5, 0.5]))   # all four at the same distance
    assert i == 0 and gap == 0.0


def test_strided_convolution_and_replicate_padding():
    rng = np.random.default_rng(21)
    for k, st in ((8, 4), (10, 5), (12, 6), (16, 8), (4, 2)):
        x = rng.standard_normal((1, 6 * st))
        w = rng.standard_normal((1, 1, k))
        y = M.conv1d_causal_strided(x, w, np.array([0.25]), st)[0]
        full = np.convolve(np.concatenate([np.zeros(k - st), x[0]]), w[0, 0][::-1], mode="valid")
        assert y.shape == (6,) and np.allclose(y, full[::st][:6] + 0.25, rtol=1e-13, atol=1e-13)
    # replicate: a constant input gives the constant sum of the taps everywhere
    w = rng.standard_normal((3, 2, 4))
    c = np.array([[1.5], [-0.5]])
    y = M.conv1d_causal_strided(np.repeat(c, 8, axis=1), w, None, 2, replicate=True)
    assert np.allclose(y, (w.sum(2) @ c).repeat(4, axis=1), rtol=1e-13)
    # and the first output sees x0 three times, then x1
    x = rng.standard_normal((2, 6))
    y0 = M.conv1d_causal_strided(x, w, None, 2, replicate=True)[:, 0]
    assert np.allclose(y0, (w[:, :, 0] + w[:, :, 1] + w[:, :, 2]) @ x[:, 0] + w[:, :, 3] @ x[:, 1], rtol=1e-13)


def _tiny_encoder(seed):
    s = tiny_mimi_shape()
    return s, M.MimiEncoderOracle(s, random_weights(s, seed=seed, specs=M.encoder_tensor_specs(s)))


def test_acoustic_chain_ignores_the_semantic_branch():
    s, E = _tiny_encoder(22)
    e = np.random.default_rng(23).standard_normal(s.dim)
    codes, _ = E.quantize(e)
    E.W["q.codebook.0"] = E.W["q.codebook.0"][::-1].copy()   # a different semantic table
    E.W["q.sem.in"] = -E.W["q.sem.in"]
    codes2, _ = E.quantize(e)
    assert codes2[1:] == codes[1:]


def test_encoder_is_causal_frame_by_frame():
    s, E = _tiny_encoder(24)
    pcm = np.random.default_rng(25).standard_normal(5 * s.frame_samples) * 0.3
    a = E.latent(pcm[:3 * s.frame_samples])
    b = E.latent(pcm)
    assert a.shape == (3, s.dim) and b.shape == (5, s.dim)
    assert np.allclose(a, b[:3], rtol=0, atol=1e-12 * np.abs(b).max())
    assert np.array_equal(E.encode(pcm[:3 * s.frame_samples]), E.encode(pcm)[:3])
