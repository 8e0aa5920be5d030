"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test states the passage it follows ("PersonaPlex native LM audit" = clockless-atlas
personaplex-research page, P1 below; sections as printed there).  Structured weights are
chosen so that a dropped term, a wrong sign or index, or a transposed operand changes
the checked value.
"""
import json
import math
import os

import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I
from oracle import oracle as O
from oracle import tiny_reference as TR

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(x):
    """float -> bf16 bits (values used here are exactly representable)."""
    b = np.asarray(x, np.float32).view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (b >> 16).astype(np.uint16)


def tiny_model(shape=None, depformer=True, mutate=None):
    s = shape or I.tiny_shape()
    W = I.make_weights(s, depformer=depformer)
    if mutate:
        mutate(W, s)
    specs = I.tensor_specs(s, depformer)
    tensors = [W[name] for name, _, _ in specs]
    return s, W, O.Oracle(s.asdict(), tensors, depformer=depformer)


# --------------------------------------------------------------------------
# shapes: P1 section 5 inventory, section 6 cache sizes
# --------------------------------------------------------------------------

def test_inventory_matches_page():
    g = json.load(open(os.path.join(GOLDEN, "personaplex_inventory.json")))
    specs = I.tensor_specs(I.FULL)
    assert len(specs) == g["total_tensors"]
    total = sum(int(np.prod(sh)) for _, sh, _ in specs)
    assert total == g["total_params"]
    # the 8-position constructor from P1 section 2
    s8 = I.ModelShape(dep_steps=8)
    total8 = sum(int(np.prod(sh)) for _, sh, _ in I.tensor_specs(s8))
    assert total8 == g["params_with_8_depth_positions"]
    assert total - total8 == g["difference_8_vs_16"]
    # per-family sums
    fam = {}
    for name, sh, _ in specs:
        if name.startswith("emb."):
            k = "emb.*.weight"
        elif name == "text_emb":
            k = "text_emb.weight"
        elif name == "text_linear":
            k = "text_linear.weight"
        elif name.startswith("layers.") and name.endswith("in_proj"):
            k = "transformer.layers.*.self_attn.in_proj_weight"
        elif name.startswith("layers.") and name.endswith("out_proj"):
            k = "transformer.layers.*.self_attn.out_proj.weight"
        elif name.startswith("layers.") and name.endswith("linear_in"):
            k = "transformer.layers.*.gating.linear_in.weight"
        elif name.startswith("layers.") and name.endswith("linear_out"):
            k = "transformer.layers.*.gating.linear_out.weight"
        elif (name.startswith("layers.") and "norm" in name) or name == "out_norm":
            k = "temporal norm alphas"
        elif name.startswith("depformer_in."):
            k = "depformer_in.*.weight"
        elif name.startswith("depformer_emb."):
            k = "depformer_emb.*.weight"
        elif name == "depformer_text_emb":
            k = "depformer_text_emb.weight"
        elif name.startswith("depformer.") and name.endswith("in_proj"):
            k = "depformer.layers.*.self_attn.in_proj_weight"
        elif name.startswith("depformer.") and name.endswith("out_proj"):
            k = "depformer.layers.*.self_attn.out_proj.weight"
        elif name.startswith("depformer.") and name.endswith("linear_in"):
            k = "depformer.layers.*.gating.*.linear_in.weight"
        elif name.startswith("depformer.") and name.endswith("linear_out"):
            k = "depformer.layers.*.gating.*.linear_out.weight"
        elif name.startswith("depformer.") and "norm" in name:
            k = "depth norm alphas"
        elif name.startswith("linears."):
            k = "linears.*.weight"
        else:
            raise AssertionError(name)
        c, p = fam.get(k, (0, 0))
        fam[k] = (c + 1, p + int(np.prod(sh)))
    for f in g["families"]:
        assert fam[f["pattern"]] == (f["count"], f["params"]), f["pattern"]


def test_cache_sizes_match_pages():
    g = json.load(open(os.path.join(GOLDEN, "personaplex_inventory.json")))
    s = I.FULL
    per_layer = 2 * 1 * s.H * s.ctx * s.dh * 2  # [2,B,32,3000,128] bf16, B=1
    assert per_layer == g["temporal_kv_bytes_per_layer_bf16_B1"]
    assert per_layer * s.n_layers == g["temporal_kv_bytes_32_layers_bf16_B1"]
    assert 2 * 1 * s.dep_H * s.dep_steps * s.dep_dh * 2 * s.dep_layers == g["depth_kv_bytes_6_layers_bf16_B1"]
    assert 2 * s.D * 2 == g["kv_bytes_per_position_per_layer"]
    assert 2 * s.D * 2 * s.n_layers == g["kv_bytes_per_position_32_layers"]
    assert 2 * g["temporal_ffn_configured"] // 3 == s.ffn == g["temporal_ffn_hidden"]
    assert 2 * g["depth_ffn_configured"] // 3 == s.dep_ffn == g["depth_ffn_hidden"]


# --------------------------------------------------------------------------
# scalar steps
# --------------------------------------------------------------------------

def test_bf16_widening_exact():
    L = O.lib()
    assert L.orc_bf16_to_double(0x3F80) == 1.0
    assert L.orc_bf16_to_double(0xBF80) == -1.0
    assert L.orc_bf16_to_double(0x4049) == 3.140625
    assert L.orc_bf16_to_double(0x0000) == 0.0


def test_matvec_orientation():
    # W is [out, in]: one nonzero at (r=2, c=5) maps x[5] to y[2] only.
    W = np.zeros((3, 7), np.uint16)
    W[2, 5] = bf16(1.5)
    x = np.arange(7, dtype=np.float64) + 1.0
    y = O.matvec(W, x)
    assert np.array_equal(y, [0.0, 0.0, 1.5 * 6.0])


def test_rmsnorm_closed_form():
    # P1 connector section 2: RMSNorm(x; g, e) = g * x / sqrt(mean x^2 + e); eps 1e-8 (P1 section 3)
    n, eps = 64, 1e-8
    alpha = bf16(np.full(n, 1.25, np.float32))
    for c in (3.0, -0.5, 1e-5):
        y = O.rmsnorm(np.full(n, c), alpha, eps)
        assert np.allclose(y, 1.25 * c / math.sqrt(c * c + eps), rtol=1e-14, atol=0)
    # no mean subtraction: a constant vector does not normalise to zero
    assert abs(O.rmsnorm(np.full(n, 2.0), alpha, eps)[0]) > 1.0
    # eps is inside the sqrt: x = 0 maps to exactly 0, tiny x is damped by eps
    assert np.all(O.rmsnorm(np.zeros(n), alpha, eps) == 0.0)
    # scale invariance up to the eps term
    rng = np.random.default_rng(0)
    x = rng.standard_normal(n)
    assert np.allclose(O.rmsnorm(7.0 * x, alpha, eps), O.rmsnorm(x, alpha, eps), rtol=1e-7)
    # per-coordinate scale: unit alpha gives mean(y^2) = 1 (up to eps)
    y = O.rmsnorm(x, bf16(np.ones(n, np.float32)), eps)
    assert abs(np.mean(y * y) - 1.0) < 1e-7


def test_rope_pairs_frequency_and_sign():
    # P1 section 3: period 10,000, all 128 coordinates in adjacent pairs,
    # f_j = exp(-log(10000) * 2j / 128).
    dh = 128
    v = np.zeros(dh)
    v[0] = 1.0
    r = O.rope(v, 1)
    # pair (0,1), j = 0: f = 1, angle 1 rad; coordinate 0 rotates into coordinate 1, never 64
    assert np.allclose(r[:2], [math.cos(1.0), math.sin(1.0)], atol=1e-15)
    assert np.all(r[2:] == 0.0)
    # pair (64,65), j = 32: f = 1e4^(-1/2) = 0.01; at pos 100 the angle is 1 rad
    v = np.zeros(dh)
    v[64] = 1.0
    r = O.rope(v, 100)
    assert np.allclose(r[64:66], [math.cos(1.0), math.sin(1.0)], atol=1e-12)
    # second coordinate of a pair: (0, 1) -> (-sin, cos)
    v = np.zeros(dh)
    v[1] = 1.0
    r = O.rope(v, 1)
    assert np.allclose(r[:2], [-math.sin(1.0), math.cos(1.0)], atol=1e-15)


def test_rope_identity_norm_and_shift_invariance():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    assert np.array_equal(O.rope(q, 0), q)
    r = O.rope(q, 777)
    assert np.allclose(r[0::2] ** 2 + r[1::2] ** 2, q[0::2] ** 2 + q[1::2] ** 2, rtol=1e-12)
    for p, pp, sh in ((5, 2, 11), (2999, 1, 3000), (40, 40, 123456)):
        a = O.rope(q, p) @ O.rope(k, pp)
        b = O.rope(q, p + sh) @ O.rope(k, pp + sh)
        assert abs(a - b) < 1e-9 * (1 + abs(a))


def test_silu_identities():
    assert O.silu(0.0) == 0.0
    for x in (0.3, 1.0, 2.5, 7.0):
        # x*sigma(x) - (-x)*sigma(-x) = x
        assert abs(O.silu(x) - O.silu(-x) - x) < 1e-14
    # sigma(ln 3) = 3/4
    assert abs(O.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15


def test_attention_single_key_and_scale():
    rng = np.random.default_rng(2)
    dh = 128
    q = rng.standard_normal(dh)
    k = rng.standard_normal((1, dh))
    v = rng.standard_normal((1, dh))
    assert np.allclose(O.attend(q, k, v), v[0], rtol=0, atol=0)  # one key: softmax = 1
    # two keys, scores a/sqrt(dh) and 0 with a = sqrt(dh)*ln 3 -> weights 3/4, 1/4
    q = np.zeros(dh)
    q[0] = math.sqrt(dh) * math.log(3.0)
    k = np.zeros((2, dh))
    k[0, 0] = 1.0
    v = np.zeros((2, dh))
    v[0, 0] = 1.0
    v[1, 1] = 1.0
    o = O.attend(q, k, v)
    assert abs(o[0] - 0.75) < 1e-14 and abs(o[1] - 0.25) < 1e-14


def test_argmax_lowest_index_on_ties():
    assert O.argmax(np.array([1.0, 3.0, 2.0, 3.0])) == 1
    assert O.argmax(np.array([-1.0, -1.0])) == 0


# --------------------------------------------------------------------------
# embedding sum and IDs: P1 section 3 "Input embedding sum"
# --------------------------------------------------------------------------

def test_embedding_sum_zero_and_exact_rows():
    s, W, M = tiny_model(depformer=False)
    allneg = np.full(s.n_streams, -1, np.int32)
    assert np.all(M.embed(allneg) == 0.0)
    one = allneg.copy()
    one[5] = 7
    assert np.array_equal(M.embed(one), TR.widen(W["emb.4"][7]))
    two = one.copy()
    two[0] = 11
    assert np.array_equal(M.embed(two), TR.widen(W["emb.4"][7]) + TR.widen(W["text_emb"][11]))  # sum, not mean
    init = allneg.copy()
    init[0] = s.init_text
    init[16] = s.init_audio
    assert np.array_equal(M.embed(init), TR.widen(W["text_emb"][s.init_text]) + TR.widen(W["emb.15"][s.init_audio]))


def test_invalid_ids_rejected():
    s, W, M = tiny_model(depformer=False)
    st = M.new_stream()
    ok = np.zeros(s.n_streams, np.int32)
    for bad_k, bad_v in ((0, -2), (3, -2), (0, s.text_in), (9, s.audio_in), (16, -3)):
        ids = ok.copy()
        ids[bad_k] = bad_v
        with pytest.raises(ValueError):
            st.step(ids)
    assert st.pos == 0  # state unchanged on error
    st.step(ok)
    assert st.pos == 1


def test_delay_assembly_integer_cases():
    # P1 section 7: delays [0,0,1,1,1,1,1,1,1,0,1,1,1,1,1,1,1]; initial IDs text 32000 / audio 2048.
    s, W, M = tiny_model(depformer=False)
    st = M.new_stream()
    d = np.array(s.delays)
    ids0 = np.arange(s.n_streams, dtype=np.int32) + 10
    ids1 = np.arange(s.n_streams, dtype=np.int32) + 30
    in0 = st.delay_assemble(ids0)
    init = np.array([s.init_text] + [s.init_audio] * 16)
    assert np.array_equal(in0, np.where(d == 0, ids0, init))
    s2 = M.new_stream()
    s2.step(ids0)
    in1 = s2.delay_assemble(ids1)
    assert np.array_equal(in1, np.where(d == 0, ids1, ids0))
    # after a position set, delayed streams read initial IDs again
    s3 = M.new_stream()
    s3.set_position(500)
    assert np.array_equal(s3.delay_assemble(ids1), np.where(d == 0, ids1, init))


# --------------------------------------------------------------------------
# block structure with structured weights (one layer)
# --------------------------------------------------------------------------

def _zero_blocks(W, s):
    for l in range(s.n_layers):
        for n in ("in_proj", "out_proj", "linear_in", "linear_out"):
            W[f"layers.{l}.{n}"][...] = 0


def test_zero_sublayers_are_identity():
    # y = x + a, output = y + f: with all projections zero the residual stream is the
    # embedding sum and h = RMSNorm_out(x) (P1 section 3 block equations).
    s, W, M = tiny_model(depformer=False, mutate=_zero_blocks)
    st = M.new_stream()
    ids = I.make_ids(s, 3)[:, 0]
    for t in range(3):
        inp = ids[t].copy()
        if t == 0:
            inp = np.where(np.array(s.delays) == 0, ids[0], [s.init_text] + [s.init_audio] * 16).astype(np.int32)
        else:
            inp = np.where(np.array(s.delays) == 0, ids[t], ids[t - 1]).astype(np.int32)
        x = M.embed(inp)
        hid, res, _, _ = st.step(ids[t])
        assert np.array_equal(res, x)
        assert np.allclose(hid, O.rmsnorm(x, W["out_norm"], s.eps), rtol=1e-15, atol=0)


def test_swiglu_first_half_is_gated():
    # P1 section 3: SiLU on the first half g (rows 0..F-1), multiplied by z (rows F..2F-1).
    s = I.tiny_shape(n_layers=1)
    cg, cz = 2.0, 0.5

    def mut(W, s):
        _zero_blocks(W, s)
        wi = W["layers.0.linear_in"]
        wi[0, 0] = bf16(cg)        # g_0 = cg * v_0
        wi[s.ffn, 0] = bf16(cz)    # z_0 = cz * v_0
        W["layers.0.linear_out"][3, 0] = bf16(1.0)  # f_3 = s_0

    s, W, M = tiny_model(s, depformer=False, mutate=mut)
    st = M.new_stream()
    ids = I.make_ids(s, 1)[0, 0]
    inp = np.where(np.array(s.delays) == 0, ids, [s.init_text] + [s.init_audio] * 16).astype(np.int32)
    y = M.embed(inp)
    v0 = O.rmsnorm(y, W["layers.0.norm2"], s.eps)[0]
    _, res, _, _ = st.step(ids)
    g, z = cg * v0, cz * v0
    expect = y.copy()
    expect[3] += (g / (1.0 + math.exp(-g))) * z
    swapped = (z / (1.0 + math.exp(-z))) * g
    assert abs(res[3] - expect[3]) < 1e-12
    assert abs((res[3] - y[3]) - swapped) > 1e-3


def test_value_rows_and_window_uniform_attention():
    # Q rows zero -> all scores equal -> attention is the plain mean of V over the window
    # 0 <= t - s < ctx (P1 section 3 mask); V = rows 2D..3D-1 of the fused projection.
    ctx = 4
    s = I.tiny_shape(n_layers=1, ctx=ctx)
    cv = 0.5

    def mut(W, s):
        _zero_blocks(W, s)
        W["layers.0.in_proj"][2 * s.D + 0, 1] = bf16(cv)   # v_0 = cv * u_1
        W["layers.0.in_proj"][s.D + 7, 2] = bf16(1.0)      # K rows nonzero: irrelevant when q = 0
        W["layers.0.out_proj"][9, 0] = bf16(1.0)           # a_9 = o_0

    s, W, M = tiny_model(s, depformer=False, mutate=mut)
    st = M.new_stream()
    T = 10
    ids = I.make_ids(s, T)[:, 0]
    us = []
    for t in range(T):
        src = [t - d for d in s.delays]
        inp = np.array([ids[j, k] if j >= 0 else (s.init_text if k == 0 else s.init_audio)
                        for k, j in enumerate(src)], np.int32)
        x = M.embed(inp)
        us.append(O.rmsnorm(x, W["layers.0.norm1"], s.eps)[1])
        _, res, _, _ = st.step(ids[t])
        lo = max(0, t - ctx + 1)
        expect = np.mean([cv * u for u in us[lo:t + 1]])
        assert abs(res[9] - x[9] - expect) < 1e-12, t
        if t >= ctx:
            wrong = np.mean([cv * u for u in us[lo - 1:t + 1]])  # one key too many
            assert abs(res[9] - x[9] - wrong) > 1e-6


def test_text_head_reads_final_norm():
    # P1 section 3: h = final RMSNorm(x); logits = h W_text^T (untied, no softcap).
    s = I.tiny_shape(n_layers=1)

    def mut(W, s):
        _zero_blocks(W, s)
        W["text_linear"][...] = 0
        for i in range(s.text_out):
            W["text_linear"][i, i % s.D] = bf16(1.0 if i < s.D else -1.0)

    s, W, M = tiny_model(s, depformer=False, mutate=mut)
    st = M.new_stream()
    ids = I.make_ids(s, 1)[0, 0]
    hid, res, lg, am = st.step(ids)
    expect = np.array([hid[i % s.D] * (1.0 if i < s.D else -1.0) for i in range(s.text_out)])
    assert np.array_equal(lg, expect)
    assert am == int(np.argmax(expect))


# --------------------------------------------------------------------------
# incremental decode == full recompute; C == independent NumPy statement
# --------------------------------------------------------------------------

@pytest.mark.parametrize("ctx,T", [(16, 12), (4, 10)])
def test_incremental_equals_full_sequence(ctx, T):
    s, W, M = tiny_model(I.tiny_shape(ctx=ctx), depformer=False)
    ids = I.make_ids(s, T, seed=77)[:, 0]
    st = M.new_stream()
    inc_h, inc_l, inc_a = [], [], []
    for t in range(T):
        h, _, lg, a = st.step(ids[t])
        inc_h.append(h)
        inc_l.append(lg)
        inc_a.append(a)
    fh, fl, fa = M.full_sequence(ids)
    assert np.allclose(np.array(inc_h), fh, rtol=1e-12, atol=1e-12)
    assert np.allclose(np.array(inc_l), fl, rtol=1e-12, atol=1e-12)
    assert list(fa) == inc_a
    # independent NumPy statement (explicit T x T mask)
    nh, nl = TR.temporal_sequence(s.asdict(), W, ids)
    assert np.allclose(fh, nh, rtol=1e-11, atol=1e-11)
    assert np.allclose(fl, nl, rtol=1e-11, atol=1e-11)


def test_window_matters_after_ctx():
    # with ctx=4 the outputs at t >= 4 differ from an unbounded context (mask is active)
    s4, W, M4 = tiny_model(I.tiny_shape(ctx=4), depformer=False)
    s16 = I.tiny_shape(ctx=16)
    M16 = O.Oracle(s16.asdict(), [W[n] for n, _, _ in I.tensor_specs(s16, False)], depformer=False)
    ids = I.make_ids(s4, 8, seed=5)[:, 0]
    h4, _, _ = M4.full_sequence(ids)
    h16, _, _ = M16.full_sequence(ids)
    assert np.array_equal(h4[:4], h16[:4])
    assert np.max(np.abs(h4[4:] - h16[4:])) > 1e-6


def test_first_frame_attention_is_value():
    # at pos 0 the only key is the frame itself: softmax = 1, o = v
    s = I.tiny_shape(n_layers=1)

    def mut(W, s):
        W["layers.0.linear_in"][...] = 0
        W["layers.0.linear_out"][...] = 0

    s, W, M = tiny_model(s, depformer=False, mutate=mut)
    ids = I.make_ids(s, 1)[0, 0]
    inp = np.where(np.array(s.delays) == 0, ids, [s.init_text] + [s.init_audio] * 16).astype(np.int32)
    x = M.embed(inp)
    u = O.rmsnorm(x, W["layers.0.norm1"], s.eps)
    v = O.matvec(W["layers.0.in_proj"][2 * s.D:], u)
    expect = x + O.matvec(W["layers.0.out_proj"], v)
    _, res, _, _ = M.new_stream().step(ids)
    assert np.allclose(res, expect, rtol=1e-13, atol=1e-13)


def _rne_bf16(x):
    """float64 -> bf16 bits, round to nearest even (finite values)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


@pytest.mark.parametrize("H,dh", [(2, 128), (4, 64)])
def test_loaded_history_equals_computed_history(H, dh):
    """A stream that decodes positions 0..19 and a stream that loads the bf16-rounded K/V of
    those positions, computed from the oracle's own steps (embedding sum -> RMSNorm ->
    fused QKV -> RoPE of the keys at their positions), continue within bf16-rounding
    distance of each other.  All delays are 0 so that a position's input does not depend on
    the previous frame's IDs.  The same history loaded in the transposed layout
    [position][head][dh] instead of [head][position][dh] misses by far more, so a layout
    error in the load would fail here."""
    s = I.tiny_shape(n_layers=1, H=H, dh=dh, ctx=32, delays=[0] * 17)
    s, W, M = tiny_model(s, depformer=False)
    T0, T1 = 20, 4
    D = s.D
    ids = I.make_ids(s, T0 + T1, seed=9)[:, 0]
    a = M.new_stream()
    ha = [a.step(ids[t])[0] for t in range(T0 + T1)]
    K = np.zeros((H, T0, dh))
    V = np.zeros((H, T0, dh))
    for p in range(T0):
        u = O.rmsnorm(M.embed(ids[p]), W["layers.0.norm1"], s.eps)
        qkv = O.matvec(W["layers.0.in_proj"], u)
        for h in range(H):
            K[h, p] = O.rope(qkv[D + h * dh:D + (h + 1) * dh], p, s.rope_theta)
            V[h, p] = qkv[2 * D + h * dh:2 * D + (h + 1) * dh]
    Kb, Vb = _rne_bf16(K), _rne_bf16(V)

    def run(k, v):
        st = M.new_stream()
        st.load_kv(0, 0, k, v)
        st.set_position(T0)
        return [st.step(ids[t])[0] for t in range(T0, T0 + T1)]

    def err(hs):
        return max(float(np.max(np.abs(h - ha[T0 + i])) / np.max(np.abs(ha[T0 + i]))) for i, h in enumerate(hs))

    e_load = err(run(Kb, Vb))
    assert 0.0 < e_load <= 1e-3, e_load          # bf16 rounding of K and V only
    e_transposed = err(run(np.ascontiguousarray(Kb.transpose(1, 0, 2)).reshape(H, T0, dh),
                           np.ascontiguousarray(Vb.transpose(1, 0, 2)).reshape(H, T0, dh)))
    assert e_transposed > 100 * e_load, (e_transposed, e_load)


def test_key_outside_the_window_changes_nothing():
    s, W, M = tiny_model(I.tiny_shape(ctx=8), depformer=False)
    ids = I.make_ids(s, 3, seed=9)[:, 0]
    k_hist = [I.make_kv_history(s, 20, seed=3, layer=l, stream=0) for l in range(s.n_layers)]
    # changing a key outside the window (position 5 < 23-8+1) changes nothing; inside does
    c = M.new_stream()
    d = M.new_stream()
    for st, bump in ((c, 5), (d, 19)):
        for l in range(s.n_layers):
            k, v = k_hist[l]
            k2 = k.copy()
            if l == 0:
                k2[:, bump, :] = bf16(np.full(s.dh, 4.0, np.float32))
            st.load_kv(l, 0, k2, v)
        st.set_position(20)
    ref = M.new_stream()
    for l in range(s.n_layers):
        ref.load_kv(l, 0, *k_hist[l])
    ref.set_position(20)
    outs = {}
    for name, st in (("c", c), ("d", d), ("ref", ref)):
        for t in range(3):
            h = st.step(ids[t])[0]
        outs[name] = h
    assert np.array_equal(outs["c"], outs["ref"])
    assert not np.array_equal(outs["d"], outs["ref"])


# --------------------------------------------------------------------------
# depformer: P1 section 4
# --------------------------------------------------------------------------

def test_depformer_matches_numpy_and_supplied_codes():
    s, W, M = tiny_model()
    rng = np.random.default_rng(3)
    hidden = rng.standard_normal(s.D)
    sup = I.make_supplied_codes(s, 1)[0, 0]
    lg, codes = M.depformer_step(hidden, 17, sup)
    nl, nc = TR.depformer(s.asdict(), W, hidden, 17, sup)
    assert np.allclose(lg, nl, rtol=1e-11, atol=1e-11)
    assert np.array_equal(codes, nc)
    assert np.array_equal(codes[8:], sup[8:])       # supplied codes replace the sampled ones
    for q in range(8):
        assert codes[q] == int(np.argmax(lg[q]))     # greedy where not supplied
    # fresh depth context each call: the same call gives the same result
    lg2, codes2 = M.depformer_step(hidden, 17, sup)
    assert np.array_equal(lg, lg2) and np.array_equal(codes, codes2)


def test_depformer_context_8_vs_16():
    s8, W, M8 = tiny_model(I.tiny_shape(dep_ctx=8))
    s16 = I.tiny_shape(dep_ctx=16)
    M16 = O.Oracle(s16.asdict(), [W[n] for n, _, _ in I.tensor_specs(s16)])
    rng = np.random.default_rng(4)
    hidden = rng.standard_normal(s8.D)
    sup = rng.integers(0, s8.dep_card, s8.dep_steps).astype(np.int32)  # all supplied: same inputs
    l8, _ = M8.depformer_step(hidden, 5, sup)
    l16, _ = M16.depformer_step(hidden, 5, sup)
    assert np.array_equal(l8[:8], l16[:8])
    assert np.max(np.abs(l8[8:] - l16[8:])) > 1e-9


def test_depformer_no_final_norm_and_input_embedding():
    # all depth blocks zero -> z_q = W_in,q h + E(prev); logits_q = W_head,q z_q, no norm
    s = I.tiny_shape()

    def mut(W, s):
        for j in range(s.dep_layers):
            W[f"depformer.{j}.in_proj"][...] = 0
            W[f"depformer.{j}.out_proj"][...] = 0
            for q in range(s.dep_steps):
                W[f"depformer.{j}.gating.{q}.linear_in"][...] = 0
                W[f"depformer.{j}.gating.{q}.linear_out"][...] = 0

    s, W, M = tiny_model(s, mutate=mut)
    rng = np.random.default_rng(6)
    hidden = rng.standard_normal(s.D)
    sup = np.full(s.dep_steps, -1, np.int32)
    sup[3] = 9
    lg, codes = M.depformer_step(hidden, 12, sup)
    prev = 12
    for q in range(s.dep_steps):
        emb = W["depformer_text_emb"] if q == 0 else W[f"depformer_emb.{q - 1}"]
        z = O.matvec(W[f"depformer_in.{q}"], hidden) + TR.widen(emb[prev])
        assert np.allclose(lg[q], O.matvec(W[f"linears.{q}"], z), rtol=1e-13, atol=1e-13), q
        prev = int(codes[q])
    assert codes[3] == 9


def test_depformer_weight_slices_are_per_position():
    # only slice q*=5 of the packed depth attention projections is nonzero: positions
    # before 5 cannot see it (P1 section 4 table: slice [3072,1024] at one q)
    s = I.tiny_shape()
    qs = 5

    def zero_attn(W, s):
        for j in range(s.dep_layers):
            W[f"depformer.{j}.in_proj"][...] = 0
            W[f"depformer.{j}.out_proj"][...] = 0

    s, Wz, Mz = tiny_model(s, mutate=zero_attn)
    Wq = {k: v.copy() for k, v in Wz.items()}
    ref = I.make_weights(s)
    Dd = s.dep_D
    for j in range(s.dep_layers):
        Wq[f"depformer.{j}.in_proj"][qs * 3 * Dd:(qs + 1) * 3 * Dd] = ref[f"depformer.{j}.in_proj"][qs * 3 * Dd:(qs + 1) * 3 * Dd]
        Wq[f"depformer.{j}.out_proj"][qs * Dd:(qs + 1) * Dd] = ref[f"depformer.{j}.out_proj"][qs * Dd:(qs + 1) * Dd]
    Mq = O.Oracle(s.asdict(), [Wq[n] for n, _, _ in I.tensor_specs(s)])
    rng = np.random.default_rng(8)
    hidden = rng.standard_normal(s.D)
    sup = rng.integers(0, s.dep_card, s.dep_steps).astype(np.int32)
    lz, _ = Mz.depformer_step(hidden, 1, sup)
    lq, _ = Mq.depformer_step(hidden, 1, sup)
    assert np.array_equal(lz[:qs], lq[:qs])
    assert np.max(np.abs(lz[qs] - lq[qs])) > 1e-9
