"""Stream snapshots through the C ABI: a restored stream continues bit-identically to the
stream that was snapshotted (before and after the KV ring wraps, into the same context
after a reset and into a second context with the same configuration), and foreign or
corrupt buffers are rejected."""
import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I
from full_duplex_speech_moshi_gb300 import pm

from harness import Pair, small_shape

pytestmark = pytest.mark.gpu


def _run(pair, ids):
    out = []
    for t in range(ids.shape[0]):
        out.append(pair.gpu_frame(ids[t:t + 1]))
    return out


def _same(a, b):
    for (ha, la, ta), (hb, lb, tb) in zip(a, b):
        assert np.array_equal(ha, hb) and np.array_equal(la, lb) and np.array_equal(ta, tb)


@pytest.mark.parametrize("prefix", [20, 45])  # ring of 32: before and after the wrap
def test_restore_continues_bit_identically(prefix):
    s = small_shape()
    a = Pair(s, B_max=1, depformer=False)
    b = Pair(s, B_max=1, depformer=False, weights=a.W)
    torch = a.torch
    try:
        ids = I.make_ids(s, prefix + 6, seed=81)[:, 0]
        _run(a, ids[:prefix])
        snap = torch.empty(a.ctx.snapshot_bytes(), dtype=torch.uint8, device="cuda")
        a.ctx.snapshot(0, snap)
        cont = _run(a, ids[prefix:])
        assert a.ctx.get_positions()[0] == prefix + 6
        # the same context after a reset
        a.ctx.reset()
        a.ctx.restore(0, snap)
        assert a.ctx.get_positions()[0] == prefix
        _same(cont, _run(a, ids[prefix:]))
        # a second context with the same configuration and weights
        b.ctx.restore(0, snap)
        _same(cont, _run(b, ids[prefix:]))
    finally:
        a.close()
        b.close()


def test_restore_rejects_foreign_and_corrupt_buffers():
    s = small_shape()
    a = Pair(s, B_max=1, depformer=False)
    c = Pair(small_shape(ctx=48), B_max=1, depformer=False, weights=a.W)
    torch = a.torch
    try:
        ids = I.make_ids(s, 4, seed=82)[:, 0]
        _run(a, ids)
        snap = torch.empty(a.ctx.snapshot_bytes(), dtype=torch.uint8, device="cuda")
        a.ctx.snapshot(0, snap)
        with pytest.raises(pm.PMError) as e:
            c.ctx.restore(0, snap)           # another ring length
        assert e.value.status == pm.PM_ERR_ARG
        bad = snap.clone()
        bad[:4] = 0                          # not a snapshot
        with pytest.raises(pm.PMError) as e:
            a.ctx.restore(0, bad)
        assert e.value.status == pm.PM_ERR_ARG
        assert a.ctx.get_positions()[0] == 4  # state unchanged
    finally:
        a.close()
        c.close()


def test_restore_rejects_invalid_ids_in_the_snapshot():
    """A snapshot whose header is intact but whose delay ring or selections hold an ID
    outside the embedding tables is refused on the host before any copy into the context,
    so no kernel ever sees the bad value as a table row."""
    s = small_shape()
    a = Pair(s, B_max=1, depformer=False)
    torch = a.torch
    try:
        ids = I.make_ids(s, 6, seed=83)[:, 0]
        _run(a, ids)
        snap = torch.empty(a.ctx.snapshot_bytes(), dtype=torch.uint8, device="cuda")
        a.ctx.snapshot(0, snap)
        # header words: the delay ring [4 slots][32 streams] at byte 128, selections at 640
        ring_word = lambda q, k: 128 // 4 + (q & 3) * pm.PM_MAX_STREAMS + k
        rows = lambda k: s.text_in if k == 0 else s.audio_in
        cases = [(ring_word(5, 2), 2), (ring_word(4, 0), 0), (ring_word(3, 12), 12), (640 // 4 + 0, 0),
                 (640 // 4 + 3, 3)]
        for w, k in cases:
            for value in (rows(k), rows(k) + 5, -5, 1 << 30):
                bad = snap.clone()
                bad.view(torch.int32)[w] = value
                a.ctx.reset()
                with pytest.raises(pm.PMError) as e:
                    a.ctx.restore(0, bad)
                assert e.value.status == pm.PM_ERR_ARG, (w, value)
                assert a.ctx.get_positions()[0] == 0, (w, value)  # nothing restored
        # the intact snapshot still restores and continues bit-identically
        a.ctx.reset()
        a.ctx.restore(0, snap)
        more = I.make_ids(s, 3, seed=84)[:, 0]
        cont = _run(a, more)
        b = Pair(s, B_max=1, depformer=False, weights=a.W)
        try:
            _same(cont, _run(b, np.concatenate([ids, more]))[6:])
        finally:
            b.close()
    finally:
        a.close()
