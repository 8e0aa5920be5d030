"""Prefill (pm_prefill) through the C ABI against the float64 oracle stepping the same
frames one by one: T frames of one stream as batched passes of up to 64 rows (tensor-core
projections, causal attention within the pass), then ordinary decode frames that read the
KV rows the prefill left in the ring.  Shapes as the other parity tests (a 32-frame ring,
so a 64-row pass reuses every slot twice)."""
import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I
from full_duplex_speech_moshi_gb300 import pm

from harness import Pair, hidden_err, logits_rel_l2, small_shape, HIDDEN_TOL, LOGITS_TOL, GAP_MIN, top2_gap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pair():
    p = Pair(small_shape(), B_max=2, depformer=False)
    yield p
    p.close()


def _prefill(pair, stream, ids):
    pair.ctx.prefill(stream, ids.shape[0], np.ascontiguousarray(ids, np.int32), pair.logits, pair.hidden, pair.token)
    pair.torch.cuda.synchronize()
    return (pair.hidden[0].double().cpu().numpy(), pair.logits[0].double().cpu().numpy(),
            int(pair.token[0].cpu().numpy()))


def _check(g, r, where):
    gh, gl, gt = g
    rh, rl, rt = r
    assert hidden_err(gh, rh) <= HIDDEN_TOL, (where, hidden_err(gh, rh))
    assert logits_rel_l2(gl, rl) <= LOGITS_TOL, (where, logits_rel_l2(gl, rl))
    if top2_gap(rl) > GAP_MIN:
        assert gt == rt, (where, gt, rt)


def test_prefill_from_reset_then_decode(pair):
    s = pair.shape
    pair.ctx.reset()
    st = pair.orc.new_stream()
    T = 70
    ids = I.make_ids(s, T + 5, seed=91)[:, 0]
    g = _prefill(pair, 0, ids[:T])
    r = None
    for t in range(T):
        r = st.step(ids[t])
    _check(g, (r[0], r[2], r[3]), "prefill")
    assert pair.ctx.get_positions()[0] == T
    for t in range(T, T + 5):
        gh, gl, gt = pair.gpu_frame(ids[t:t + 1])
        rh, _, rl, rt = st.step(ids[t])
        _check((gh[0], gl[0], int(gt[0])), (rh, rl, rt), f"decode t={t}")


def test_prefill_after_wrapped_decode(pair):
    s = pair.shape
    pair.ctx.reset()
    st = pair.orc.new_stream()
    ids = I.make_ids(s, 40 + 20 + 3, seed=92)[:, 0]
    for t in range(40):                     # the 32-slot ring wraps
        pair.gpu_frame(ids[t:t + 1])
        st.step(ids[t])
    g = _prefill(pair, 0, ids[40:60])
    r = None
    for t in range(40, 60):
        r = st.step(ids[t])
    _check(g, (r[0], r[2], r[3]), "prefill after decode")
    for t in range(60, 63):
        gh, gl, gt = pair.gpu_frame(ids[t:t + 1])
        rh, _, rl, rt = st.step(ids[t])
        _check((gh[0], gl[0], int(gt[0])), (rh, rl, rt), f"decode t={t}")


def test_prefill_window_of_several_chunks():
    """A 600-position ring and 700 frames: passes of 64 rows from 0 to 640, the last one 60
    rows; from position 256 on a pass attends over more than one 256-key chunk (three at
    the end, past the ring's wrap), so its rows are merged from chunk partials."""
    p = Pair(small_shape(ctx=600), B_max=1, depformer=False)
    try:
        s = p.shape
        st = p.orc.new_stream()
        T = 700
        ids = I.make_ids(s, T + 3, seed=93)[:, 0]
        g = _prefill(p, 0, ids[:T])
        r = None
        for t in range(T):
            r = st.step(ids[t])
        _check(g, (r[0], r[2], r[3]), "prefill of 700 frames")
        assert p.ctx.get_positions()[0] == T
        for t in range(T, T + 3):
            gh, gl, gt = p.gpu_frame(ids[t:t + 1])
            rh, _, rl, rt = st.step(ids[t])
            _check((gh[0], gl[0], int(gt[0])), (rh, rl, rt), f"decode t={t}")
    finally:
        p.close()


def test_prefill_of_one_stream_leaves_the_others(pair):
    s = pair.shape
    pair.ctx.reset()
    st = pair.orc.new_stream()
    ids = I.make_ids(s, 12, seed=93)[:, 0]
    g = _prefill(pair, 1, ids)
    r = None
    for t in range(12):
        r = st.step(ids[t])
    _check(g, (r[0], r[2], r[3]), "stream 1")
    assert pair.ctx.get_positions()[:2] == [0, 12]


def test_prefill_rejects_invalid_ids(pair):
    s = pair.shape
    pair.ctx.reset()
    ids = I.make_ids(s, 5, seed=94)[:, 0].copy()
    ids[3, 0] = pm.PM_ID_FEEDBACK
    with pytest.raises(pm.PMError) as e:
        pair.ctx.prefill(0, 5, ids)
    assert e.value.status == pm.PM_ERR_INVALID_ID
    ids[3, 0] = s.text_in
    with pytest.raises(pm.PMError) as e:
        pair.ctx.prefill(0, 5, ids)
    assert e.value.status == pm.PM_ERR_INVALID_ID
    assert pair.ctx.get_positions()[0] == 0
    # the same IDs in device memory: checked on the device, the pass is a no-op
    dev = pair.torch.from_numpy(ids).cuda()
    pair.ctx.prefill(0, 5, dev)
    assert pair.ctx.device_status() == pm.PM_ERR_INVALID_ID
    assert pair.ctx.get_positions()[0] == 0
