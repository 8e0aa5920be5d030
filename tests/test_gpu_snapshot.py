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
