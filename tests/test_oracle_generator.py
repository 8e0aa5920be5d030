"""Pins of the oracle's generator step ("PersonaPlex native LM audit", section 7 "One exact
generator step", and section 6 "Generator delayed-code cache").

- The ring logic against a trace worked by hand from the seven steps
  (tests/golden/generator_trace.json): what the model is handed at each call (input column,
  provided text, provided depth targets) and the aligned output.  A wrong output column,
  a placement without the stream delay, provided flags that are never cleared, a provided
  slot overwritten by a selection, or a missing initial token each change this trace.
- The direct-input temporal forward the generator uses equals the frame step with its own
  delay assembly when both are handed the same frames.
"""
import json
import os

import numpy as np

from full_duplex_speech_moshi_gb300 import inputs as I
from oracle import oracle as O
from oracle.generator import Generator, GeneratorRing

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_ring_follows_the_hand_worked_trace():
    g = json.load(open(os.path.join(GOLDEN, "generator_trace.json")))
    ring = GeneratorRing(g["delays"], g["init_ids"])
    for c in g["calls"]:
        seen = []

        def model(inp, text_p, supplied, s=ring.s):
            seen.append(dict(inputs=list(inp), text_provided=text_p, supplied=list(supplied)))
            return 100 + s, [200 + 10 * s + q for q in range(16)]

        out = ring.step(c["provided"], model)
        assert out == c["output"], (c["call"], out, c["output"])
        if c["model"] is None:
            assert seen == [], c["call"]
        else:
            assert seen == [c["model"]], (c["call"], seen, c["model"])
    assert ring.s == len(g["calls"])


def test_user_codes_come_out_aligned_with_the_frame_they_were_given_in():
    # user codebooks handed in at call c reappear, all eight together, in the output of
    # call c + 1 (codebook 0 has no delay, codebooks 1-7 one frame)
    ring = GeneratorRing(I.DELAYS_17, [32000] + [2048] * 16)
    outs = []
    for c in range(12):
        prov = [-1] * 9 + [1000 + 8 * c + j for j in range(8)]
        outs.append(ring.step(prov, lambda inp, tp, sup, s=ring.s: (5, [7] * 16)))
    for c in range(1, 11):
        assert outs[c + 1][9:] == [1000 + 8 * c + j for j in range(8)], c


def test_direct_forward_equals_frame_step_with_delay_assembly():
    s = I.tiny_shape(n_layers=1)
    W = I.make_weights(s, depformer=False)
    specs = I.tensor_specs(s, False)
    M = O.Oracle(s.asdict(), [W[n] for n, _, _ in specs], depformer=False)
    ids = I.make_ids(s, 6, seed=77)[:, 0]
    a = M.new_stream()
    b = M.new_stream()
    init = np.array([s.init_text] + [s.init_audio] * (s.n_streams - 1), np.int32)
    d = np.array(s.delays[:s.n_streams])
    for t in range(6):
        ha, _, la, ta = a.step(ids[t])
        prev = ids[t - 1] if t > 0 else init
        inp = np.where(d == 0, ids[t], prev).astype(np.int32)
        hb, _, lb, tb = b.forward(inp)
        assert np.array_equal(ha, hb) and np.array_equal(la, lb) and ta == tb, t
    assert a.pos == b.pos == 6


def test_generator_over_the_oracle_model():
    # a tiny model driven by the generator: the first two calls return nothing, later
    # outputs carry the provided user codes aligned, the text / agent codes the model
    # selected, and every selection is a valid token of its table
    s = I.tiny_shape()
    W = I.make_weights(s)
    specs = I.tensor_specs(s)
    M = O.Oracle(s.asdict(), [W[n] for n, _, _ in specs])
    gen = Generator(M, s.asdict())
    rng = np.random.default_rng(5)
    user = rng.integers(0, s.dep_card, size=(10, 8))
    selected = []
    for c in range(10):
        out, last = gen.step([-1] * 9 + user[c].tolist())
        if c >= 1:
            h, lg, am, dl, codes = last
            assert 0 <= am < s.text_out and all(0 <= int(x) < s.dep_audio_in for x in codes)
            selected.append([am] + [int(x) for x in codes])   # index c - 1
        if c < 2:
            assert out is None
        else:
            assert out[9:] == user[c - 1].tolist(), c
            assert out[0] == selected[c - 2][0] and out[1] == selected[c - 2][1], c
            assert out[2:9] == selected[c - 1][2:9], c
