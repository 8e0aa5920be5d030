"""Pins of the oracle's pinned-ring mode ("PersonaPlex native LM audit", section 6 "Three
distinct caches": the pinned RingKVCache labels slot positions with a delta <= 0 rule, so
a full ring hides one key; the same mapping applies to the depth cache and to Mimi's
transformer caches).  The mode is a compatibility option; the declared mask stays the
default (reading c7)."""
import json
import os

import numpy as np

from full_duplex_speech_moshi_gb300 import inputs as I
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pinned_ring.json")


def test_labels_and_visible_keys_match_page_examples():
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        labels = O.ring_labels(c["capacity"], c["end_offset"])
        if "labels" in c:
            assert labels == c["labels"]
        if "slot0_label" in c:
            assert labels[0] == c["slot0_label"]
        vis = O.visible_positions(c["query"], c["capacity"], True)
        if "visible" in c:
            assert vis == c["visible"]
        if "visible_count" in c:
            assert len(vis) == c["visible_count"]
        # the declared mask sees capacity keys (or every key before the ring fills)
        assert len(O.visible_positions(c["query"], c["capacity"], False)) == min(c["query"] + 1, c["capacity"])


def test_pinned_window_is_contiguous_and_latest():
    for cap in (4, 7, 16):
        for pos in range(0, 4 * cap):
            vis = O.visible_positions(pos, cap, True)
            n = pos + 1 if pos + 1 < cap else cap - 1
            assert vis == list(range(pos - n + 1, pos + 1)), (cap, pos, vis)


def _model(pinned, ctx, dep_ctx):
    s = I.tiny_shape(ctx=ctx, dep_ctx=dep_ctx, pinned_ring=pinned)
    W = I.make_weights(I.tiny_shape(), depformer=True)  # the same weights for every window
    specs = I.tensor_specs(s, True)
    return s, O.Oracle(s.asdict(), [W[n] for n, _, _ in specs], depformer=True)


def test_pinned_frames_equal_declared_frames_one_key_shorter():
    """A full ring hides exactly its oldest key, so the pinned mode at capacity C attends
    like the declared mask at C - 1, before and after the ring wraps."""
    C = 6
    s, pinned = _model(1, C, 8)
    _, shorter = _model(0, C - 1, 8)
    _, declared = _model(0, C, 8)
    a, b, d = pinned.new_stream(), shorter.new_stream(), declared.new_stream()
    ids = I.make_ids(s, 3 * C, seed=61)[:, 0]
    differs = False
    for t in range(3 * C):
        ha = a.step(ids[t])[0]
        hb = b.step(ids[t])[0]
        hd = d.step(ids[t])[0]
        assert np.array_equal(ha, hb), t
        if t + 1 >= C:
            differs |= not np.allclose(ha, hd, rtol=0, atol=1e-12)
        else:
            assert np.array_equal(ha, hd), t
    assert differs


def test_pinned_full_sequence_equals_incremental():
    C = 5
    s, m = _model(1, C, 8)
    T = 3 * C
    ids = I.make_ids(s, T, seed=62)[:, 0]
    hid, lg, am = m.full_sequence(ids)
    st = m.new_stream()
    for t in range(T):
        h, _, l, a = st.step(ids[t])
        assert np.allclose(h, hid[t], rtol=1e-10, atol=1e-11), t
        assert a == am[t]


def test_pinned_depth_cache_equals_one_key_shorter_window():
    s, pinned = _model(1, 16, 16)
    _, shorter = _model(0, 16, 15)
    rng = np.random.default_rng(5)
    h = rng.normal(0, 1, s.D)
    sup = np.full(s.dep_steps, -1, np.int32)
    la, ca = pinned.depformer_step(h, 7, sup)
    lb, cb = shorter.depformer_step(h, 7, sup)
    assert np.array_equal(ca, cb) and np.array_equal(la, lb)
    # only the last position (q = 15, the ring full) differs from the declared 16-key window
    _, declared = _model(0, 16, 16)
    ld, _ = declared.depformer_step(h, 7, cb)
    lp, _ = pinned.depformer_step(h, 7, cb)
    assert s.dep_steps == 16
    assert np.array_equal(lp[:15], ld[:15]) and not np.allclose(lp[15], ld[15], rtol=0, atol=1e-12)
