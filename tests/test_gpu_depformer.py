"""The batch-1 depformer as one persistent launch (the default) against the float64 oracle
("PersonaPlex native LM audit", section 4) and against the chain of one kernel per
projection (PM_FLAG_DEPFORMER_CHAIN), on the same weights and inputs.

- logits of all sixteen positions within the parity tolerance of the oracle, greedy codes
  equal wherever the oracle's top-2 gap exceeds 1e-2, supplied codes passed through;
- lockstep (the oracle's codes supplied at every position) so that every position's logits
  are compared;
- the persistent launch and the chain agree to 1e-3 (different summation orders);
- a call replayed on the same inputs reproduces every bit (fixed reduction orders);
- an invalid supplied code in device memory leaves the feedback state untouched.
"""
import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I

from harness import GAP_MIN, Pair, logits_rel_l2, small_shape, top2_gap

pytestmark = pytest.mark.gpu


def _dep(pair, text, sup, hidden=None):
    pair.ctx.depformer_step(1, hidden=pair.hidden if hidden is None else hidden, text_tok=np.array([text], np.int32),
                            supplied=np.ascontiguousarray(sup[None], np.int32), logits=pair.dlogits,
                            codes=pair.dcodes)
    pair.torch.cuda.synchronize()
    return pair.dlogits[0].double().cpu().numpy(), pair.dcodes[0].cpu().numpy()


@pytest.mark.parametrize("dep_ctx", [8, 16])
def test_persistent_depformer_matches_oracle_and_chain(dep_ctx):
    from full_duplex_speech_moshi_gb300 import pm
    s = small_shape(dep_ctx=dep_ctx)
    a = Pair(s, B_max=1)
    b = Pair(s, B_max=1, weights=a.W, flags=pm.PM_FLAG_DEPFORMER_CHAIN)
    try:
        ids = I.make_ids(s, 4, seed=71)[:, 0]
        sup = I.make_supplied_codes(s, 4, seed=72)[:, 0]
        st = a.orc.new_stream()
        differs = False
        for t in range(4):
            a.gpu_frame(ids[t:t + 1])
            b.gpu_frame(ids[t:t + 1])
            rh, _, rl, rt = st.step(ids[t])
            text = int(rt)
            gl, gc = _dep(a, text, sup[t])
            ol, oc = a.orc.depformer_step(rh, text, sup[t])
            for q in range(s.dep_steps):
                assert logits_rel_l2(gl[q], ol[q]) <= 1e-2, (t, q)
                if gc[q] != oc[q]:
                    assert sup[t, q] < 0 and top2_gap(ol[q]) <= GAP_MIN, (t, q, gc[q], oc[q])
                    break
            else:
                assert np.array_equal(gc[sup[t] >= 0], sup[t][sup[t] >= 0])
            # lockstep: the oracle's codes supplied everywhere
            gl2, gc2 = _dep(a, text, oc.astype(np.int32))
            ol2, _ = a.orc.depformer_step(rh, text, oc.astype(np.int32))
            for q in range(s.dep_steps):
                assert logits_rel_l2(gl2[q], ol2[q]) <= 1e-2, (t, q)
            assert np.array_equal(gc2, oc)
            # the chain on the same inputs, and a replay of the persistent launch
            bl, bc = _dep(b, text, oc.astype(np.int32), hidden=b.hidden)
            for q in range(s.dep_steps):
                assert logits_rel_l2(gl2[q], bl[q]) <= 1e-3, (t, q)
            differs = differs or not np.array_equal(gl2, bl)
            gl3, gc3 = _dep(a, text, oc.astype(np.int32))
            assert np.array_equal(gl3, gl2) and np.array_equal(gc3, gc2), t
        assert differs  # the default context did not run the chain
    finally:
        a.close()
        b.close()


def test_persistent_depformer_invalid_supplied_code_is_a_no_op():
    from full_duplex_speech_moshi_gb300 import pm
    s = small_shape()
    p = Pair(s, B_max=1)
    torch = p.torch
    try:
        ids = I.make_ids(s, 1, seed=73)[:, 0]
        p.gpu_frame(ids[0:1])
        sup = torch.full((1, s.dep_steps), -1, dtype=torch.int32, device="cuda")
        p.ctx.depformer_step(1, None, None, sup, p.dlogits, p.dcodes)
        assert p.ctx.device_status() == pm.PM_OK
        before = p.dcodes.clone()
        p.dcodes.fill_(-7)
        sup[0, 5] = s.dep_audio_in          # one past the depth table
        p.ctx.depformer_step(1, None, None, sup, p.dlogits, p.dcodes)
        assert p.ctx.device_status() == pm.PM_ERR_INVALID_ID
        assert int(p.dcodes.min()) == -7 and int(p.dcodes.max()) == -7  # nothing written
        sup[0, 5] = -1
        p.ctx.depformer_step(1, None, None, sup, p.dlogits, p.dcodes)
        assert p.ctx.device_status() == pm.PM_OK
        assert torch.equal(p.dcodes, before)
    finally:
        p.close()
