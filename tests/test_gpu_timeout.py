"""Bounded device waits that run out, made to happen without any GPU fault: the poll
budget of the waits is lowered to zero through the C ABI (pm_set_wait_budget), so every
such wait of the next frame gives up at once.  The frame must be abandoned --
pm_device_status reports PM_ERR_TIMEOUT, the stream's position does not move -- and once
the budget is restored the same position is decoded again and matches the float64 oracle
frame after frame.  Covered for the batch-1 kernel chain and for the persistent frame
program (whose phase counters must be cleared for the next launch even though the
timed-out CTAs never reached the final phase)."""
import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I

from harness import Pair, small_shape

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("program", [False, True], ids=["kernel_chain", "frame_program"])
def test_wait_timeout_abandons_the_frame_and_recovers(program):
    from full_duplex_speech_moshi_gb300 import pm
    s = small_shape(ffn=3072, ctx=48)   # D and ffn multiples of 1024: the frame program applies
    p = Pair(s, B_max=1, depformer=False, flags=pm.PM_FLAG_FRAME_PROGRAM if program else 0)
    try:
        ids = I.make_ids(s, 14, seed=41)[:, 0]
        for t in range(4):
            p.check_frame(p.gpu_frame(ids[t:t + 1]), p.oracle_frame(ids[t:t + 1]), f"t={t}")
        for attempt in range(2):        # twice in a row: the second must also time out cleanly
            p.ctx.set_wait_budget(0)
            p.token.fill_(-7)
            p.ctx.frame_step(1, np.ascontiguousarray(ids[4:5]), p.logits, p.hidden, p.token)
            assert p.ctx.device_status() == pm.PM_ERR_TIMEOUT, attempt
            assert p.ctx.get_positions()[0] == 4, attempt
            assert int(p.token[0]) == -7, attempt      # no selection was made
        p.ctx.set_wait_budget()
        assert p.ctx.device_status() == pm.PM_OK
        # the abandoned position is decoded again, then the stream carries on
        for t in range(4, 14):
            p.check_frame(p.gpu_frame(ids[t:t + 1]), p.oracle_frame(ids[t:t + 1]), f"after timeout t={t}")
        assert p.ctx.device_status() == pm.PM_OK
        assert p.ctx.get_positions()[0] == 14
    finally:
        p.close()


def test_wait_timeout_in_the_persistent_depformer():
    """The batch-1 depformer launch with a zero poll budget: PM_ERR_TIMEOUT, no feedback
    codes recorded; with the budget restored the next call matches the oracle."""
    from full_duplex_speech_moshi_gb300 import pm
    from harness import logits_rel_l2
    s = small_shape()
    p = Pair(s, B_max=1)
    try:
        ids = I.make_ids(s, 2, seed=43)[:, 0]
        st = p.streams[0]
        rh, _, _, rt = st.step(ids[0])
        p.gpu_frame(ids[0:1])
        sup = np.full((1, s.dep_steps), -1, np.int32)
        p.ctx.set_wait_budget(0)
        p.dcodes.fill_(-7)
        p.ctx.depformer_step(1, hidden=p.hidden, text_tok=np.array([int(rt)], np.int32), supplied=sup,
                             logits=p.dlogits, codes=p.dcodes)
        assert p.ctx.device_status() == pm.PM_ERR_TIMEOUT
        p.ctx.set_wait_budget()
        ol, oc = p.orc.depformer_step(rh, int(rt), oc_sup := oc_supplied(s))
        p.ctx.depformer_step(1, hidden=p.hidden, text_tok=np.array([int(rt)], np.int32), supplied=oc_sup[None],
                             logits=p.dlogits, codes=p.dcodes)
        assert p.ctx.device_status() == pm.PM_OK
        gl = p.dlogits[0].double().cpu().numpy()
        for q in range(s.dep_steps):
            assert logits_rel_l2(gl[q], ol[q]) <= 1e-2, q
        assert np.array_equal(p.dcodes[0].cpu().numpy(), oc)
    finally:
        p.close()


def oc_supplied(s):
    """Seeded supplied codes at every position (so the comparison needs no lockstep)."""
    return np.random.default_rng(44).integers(0, s.dep_card, s.dep_steps).astype(np.int32)

