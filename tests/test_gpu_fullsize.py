"""GPU parity at the full model shapes of the decode-step workloads.

  config 0  one temporal block, B=1, 16 frames from an empty cache
  config 1  32-block stack, B=1, primed frames then greedy text fed back on the device
  config 2  32-block stack, B=1, 3000 cached positions (seeded K/V), decode past 3000
            so the ring wraps and keys keep absolute RoPE positions
  config 3  32-block stack, B=16, per-stream cache lengths uniform 64..3000 (seeded K/V)
  config 4  config 1 plus the depformer (dep_ctx 8, greedy q0-7, supplied q8-15)

The quick tests run a few frames of each; the `slow` tests run the workloads at their
stated lengths in lockstep with the oracle (about 0.4 s per full frame on 16 host cores):
config 1 for 256 primed + 512 greedy-feedback frames, config 2 for 256 frames past
position 3000, config 3 for 16 frames of all 16 streams, config 4 for 64 frames of
temporal stack + depformer with every selection fed back.  Lockstep: where the two sides
select different tokens (allowed only where the oracle's top-2 logit gap is at most
1e-2), the oracle's token is fed to both sides and the run continues.  Every frame is
compared element by element at the stated tolerances; the worst errors of each run are
reported (PM_PARITY_LOG).  Long histories are seeded K/V written identically to both
sides, a stand-in whose attention cost and semantics match a computed history.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I

from harness import GAP_MIN, HIDDEN_TOL, LOGITS_TOL, Pair, Worst, hidden_err, logits_rel_l2, record_parity, top2_gap

pytestmark = pytest.mark.gpu

_POOL = ThreadPoolExecutor(min(32, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def full():
    p = Pair(I.FULL, B_max=16, depformer=True)
    yield p
    p.close()


def _gpu_history(pair, b, L, seed):
    """Seeded K/V for positions 0..L-1 of stream b in every layer, into the GPU ring."""
    torch = pair.torch
    s = pair.shape
    for l in range(s.n_layers):
        k, v = I.make_kv_history(s, L, seed=seed, layer=l, stream=b, pool=_POOL)
        # positions L-ctx..L-1 are the ones a ring of ctx slots still holds
        p0 = max(0, L - s.ctx)
        idx = torch.from_numpy(np.arange(p0, L) % s.ctx).cuda()
        kt = torch.from_numpy(np.ascontiguousarray(k[:, p0:L, :]).view(np.int16)).cuda().view(torch.bfloat16)
        vt = torch.from_numpy(np.ascontiguousarray(v[:, p0:L, :]).view(np.int16)).cuda().view(torch.bfloat16)
        pair.kv[l, 0, b].index_copy_(1, idx, kt)
        pair.kv[l, 1, b].index_copy_(1, idx, vt)


def _oracle_history(pair, b, L, seed):
    """The same seeded history in a fresh oracle stream at position L."""
    s = pair.shape
    st = pair.orc.new_stream()
    for l in range(s.n_layers):
        k, v = I.make_kv_history(s, L, seed=seed, layer=l, stream=b, pool=_POOL)
        st.load_kv(l, 0, k, v)
    st.set_position(L)
    return st


def test_config0_one_block():
    p = Pair(I.ModelShape(n_layers=1), B_max=1, depformer=False)
    try:
        ids = I.make_ids(p.shape, 16, seed=2000)[:, 0]
        for t in range(16):
            p.check_frame(p.gpu_frame(ids[t:t + 1]), p.oracle_frame(ids[t:t + 1]), f"t={t}")
    finally:
        p.close()


def test_config1_full_stack_greedy_feedback(full):
    s = full.shape
    full.ctx.reset()
    st = full.orc.new_stream()
    ids = I.make_ids(s, 14, seed=2001)[:, 0]
    prev = None
    for t in range(14):
        g_ids = ids[t:t + 1].copy()
        r_ids = ids[t].copy()
        if t >= 6:  # 6 primed frames with seeded text, then greedy feedback
            g_ids[0, 0] = -3
            r_ids[0] = prev
        gh, gl, gt = full.gpu_frame(g_ids)
        rh, _, rl, rt = st.step(r_ids)
        assert hidden_err(gh[0], rh) <= 2e-2, t
        assert logits_rel_l2(gl[0], rl) <= 1e-2, t
        if int(gt[0]) != rt:
            assert top2_gap(rl) <= GAP_MIN, (t, int(gt[0]), rt)
            break
        prev = rt


def test_config1_frame_program(full):
    """The 32-block stack through the persistent single-launch frame program."""
    from full_duplex_speech_moshi_gb300 import pm
    p = Pair(I.FULL, B_max=1, depformer=False, flags=pm.PM_FLAG_FRAME_PROGRAM, weights=full.W)
    try:
        ids = I.make_ids(p.shape, 8, seed=2005)[:, 0]
        for t in range(8):
            p.check_frame(p.gpu_frame(ids[t:t + 1]), p.oracle_frame(ids[t:t + 1]), f"t={t}")
    finally:
        p.close()


def test_config2_long_context_wrap(full):
    s = full.shape
    full.ctx.reset()
    _gpu_history(full, 0, s.ctx, seed=31)
    st = _oracle_history(full, 0, s.ctx, seed=31)
    full.ctx.set_positions([s.ctx])
    ids = I.make_ids(s, 3, seed=2002)[:, 0]
    for t in range(3):  # positions 3000, 3001, 3002: slots 0, 1, 2 overwrite the oldest keys
        h, _, lg, a = st.step(ids[t])
        full.check_frame(full.gpu_frame(ids[t:t + 1]), (h[None], lg[None], np.array([a])), f"t={t}")
    assert full.ctx.get_positions()[0] == s.ctx + 3


def test_prefill_pass_on_a_full_ring(full):
    """The startup-prompt path at full size: 3000 cached positions (seeded K/V), then one
    64-frame prefill pass whose rows reuse 64 slots of the full ring, then decode frames
    reading what it left; against the oracle stepping the same frames."""
    s = full.shape
    full.ctx.reset()
    _gpu_history(full, 0, s.ctx, seed=33)
    st = _oracle_history(full, 0, s.ctx, seed=33)
    full.ctx.set_positions([s.ctx])
    T = 64
    ids = I.make_ids(s, T + 2, seed=2005)[:, 0]
    full.ctx.prefill(0, T, np.ascontiguousarray(ids[:T]), full.logits, full.hidden, full.token)
    full.torch.cuda.synchronize()
    g = (full.hidden[:1].double().cpu().numpy(), full.logits[:1].double().cpu().numpy(), full.token[:1].cpu().numpy())
    for t in range(T):
        h, _, lg, a = st.step(ids[t])
    full.check_frame(g, (h[None], lg[None], np.array([a])), "prefill")
    assert full.ctx.get_positions()[0] == s.ctx + T
    for t in range(T, T + 2):
        h, _, lg, a = st.step(ids[t])
        full.check_frame(full.gpu_frame(ids[t:t + 1]), (h[None], lg[None], np.array([a])), f"t={t}")


def test_config3_batched_ragged(full):
    s = full.shape
    B = 16
    T = 2
    full.ctx.reset()
    L = I.make_cache_lengths(B, 64, s.ctx, seed=3000)
    for b in range(B):
        _gpu_history(full, b, int(L[b]), seed=32)
    full.ctx.set_positions(list(L))
    ids = I.make_ids(s, T, B=B, seed=2003)
    g = [full.gpu_frame(ids[t], B=B) for t in range(T)]
    assert full.ctx.get_positions()[:B] == list(L + T)
    for b in range(B):  # the oracle runs stream by stream (streams are independent)
        st = _oracle_history(full, b, int(L[b]), seed=32)
        for t in range(T):
            h, _, lg, a = st.step(ids[t, b])
            gb = (g[t][0][b:b + 1], g[t][1][b:b + 1], g[t][2][b:b + 1])
            full.check_frame(gb, (h[None], lg[None], np.array([a])), f"b={b} L={L[b]} t={t}")
        del st


def test_config4_depformer(full):
    s = full.shape
    full.ctx.reset()
    st = full.orc.new_stream()
    ids = I.make_ids(s, 3, seed=2004)[:, 0]
    sup = I.make_supplied_codes(s, 3, seed=4000)[:, 0]
    for t in range(3):
        gh, _, gt = full.gpu_frame(ids[t:t + 1])
        rh, _, rl, rt = st.step(ids[t])
        text = int(rt)
        ol, oc = full.orc.depformer_step(rh, text, sup[t])
        # greedy positions 0-7 chosen on the device, 8-15 supplied
        full.ctx.depformer_step(1, hidden=full.hidden, text_tok=np.array([text], np.int32),
                                supplied=np.ascontiguousarray(sup[t:t + 1]), logits=full.dlogits,
                                codes=full.dcodes)
        full.torch.cuda.synchronize()
        gl = full.dlogits[0].double().cpu().numpy()
        gc = full.dcodes[0].cpu().numpy()
        for q in range(s.dep_steps):
            assert logits_rel_l2(gl[q], ol[q]) <= 1e-2, (t, q)
            if gc[q] != oc[q]:
                assert sup[t, q] < 0 and top2_gap(ol[q]) <= GAP_MIN, (t, q, gc[q], oc[q])
                break
        else:
            assert np.array_equal(gc[8:], sup[t, 8:])


def _check(w, gh, gl, rh, rl, where):
    he, le = hidden_err(gh, rh), logits_rel_l2(gl, rl)
    w.add(he, le)
    assert he <= HIDDEN_TOL, f"{where}: hidden err {he:.3e}"
    assert le <= LOGITS_TOL, f"{where}: logits rel L2 {le:.3e}"


def _token(w, gt, rt, rl, where):
    if int(gt) != int(rt):
        assert top2_gap(rl) <= GAP_MIN, f"{where}: token {int(gt)} vs oracle {int(rt)}"
        w.forced += 1


@pytest.mark.slow
def test_config1_stated_length_lockstep(full):
    """256 primed frames, then 512 frames whose text input is the previous frame's greedy
    token (on the GPU through the device-side feedback ID wherever its token equals the
    oracle's), every frame against the oracle."""
    s = full.shape
    P, F = 256, 512
    full.ctx.reset()
    st = full.orc.new_stream()
    ids = I.make_ids(s, P + F, seed=2011)[:, 0]
    w = Worst()
    prev_r = prev_g = None
    for t in range(P + F):
        g_ids = ids[t:t + 1].copy()
        r_ids = ids[t].copy()
        if t >= P:
            r_ids[0] = prev_r
            g_ids[0, 0] = -3 if prev_g == prev_r else prev_r
        gh, gl, gt = full.gpu_frame(g_ids)
        rh, _, rl, rt = st.step(r_ids)
        _check(w, gh[0], gl[0], rh, rl, f"t={t}")
        _token(w, gt[0], rt, rl, f"t={t}")
        prev_r, prev_g = int(rt), int(gt[0])
    assert full.ctx.get_positions()[0] == P + F
    record_parity("config1_256_primed_512_feedback", **w.asdict())
    del st


@pytest.mark.slow
def test_config2_stated_length_past_the_wrap(full):
    """3000 cached positions (seeded K/V), then 256 frames at positions 3000..3255: every
    frame overwrites the ring's oldest slot and attends over exactly 3000 keys."""
    s = full.shape
    N = 256
    full.ctx.reset()
    _gpu_history(full, 0, s.ctx, seed=31)
    st = _oracle_history(full, 0, s.ctx, seed=31)
    full.ctx.set_positions([s.ctx])
    ids = I.make_ids(s, N, seed=2012)[:, 0]
    w = Worst()
    for t in range(N):
        gh, gl, gt = full.gpu_frame(ids[t:t + 1])
        rh, _, rl, rt = st.step(ids[t])
        _check(w, gh[0], gl[0], rh, rl, f"pos={s.ctx + t}")
        _token(w, gt[0], rt, rl, f"pos={s.ctx + t}")
    assert full.ctx.get_positions()[0] == s.ctx + N
    record_parity("config2_256_past_3000", **w.asdict())
    del st


@pytest.mark.slow
def test_config3_batched_sixteen_frames(full):
    """All 16 streams (cache lengths uniform 64..3000) for 16 frames on the batched path
    (PM_CONFIG3_FRAMES sets another length: the workload states 128, about 13 minutes of
    oracle time on 16 cores)."""
    s = full.shape
    B, T = 16, int(os.environ.get("PM_CONFIG3_FRAMES", "16"))
    full.ctx.reset()
    L = I.make_cache_lengths(B, 64, s.ctx, seed=3000)
    for b in range(B):
        _gpu_history(full, b, int(L[b]), seed=34)
    full.ctx.set_positions(list(L))
    ids = I.make_ids(s, T, B=B, seed=2013)
    g = [full.gpu_frame(ids[t], B=B) for t in range(T)]
    assert full.ctx.get_positions()[:B] == list(L + T)
    w = Worst()
    for b in range(B):
        st = _oracle_history(full, b, int(L[b]), seed=34)
        for t in range(T):
            h, _, lg, a = st.step(ids[t, b])
            _check(w, g[t][0][b], g[t][1][b], h, lg, f"b={b} L={L[b]} t={t}")
            _token(w, g[t][2][b], a, lg, f"b={b} L={L[b]} t={t}")
        del st
    record_parity(f"config3_B16_ragged_{T}_frames", **w.asdict())


def _depformer_lockstep(full, w, t, h_ref, text, sup_row):
    """One depformer call on both sides; where a greedy code differs at a near tie, the
    GPU call is repeated with the oracle's codes supplied up to that position.  Returns
    the oracle's codes (identical to the GPU's final codes)."""
    s = full.shape
    ol, oc = full.orc.depformer_step(h_ref, text, sup_row)
    sup_g = sup_row.copy()
    while True:
        full.ctx.depformer_step(1, hidden=full.hidden, text_tok=np.array([text], np.int32),
                                supplied=np.ascontiguousarray(sup_g[None]), logits=full.dlogits, codes=full.dcodes)
        full.torch.cuda.synchronize()
        gl = full.dlogits[0].double().cpu().numpy()
        gc = full.dcodes[0].cpu().numpy()
        diff = [q for q in range(s.dep_steps) if gc[q] != oc[q]]
        if not diff:
            break
        q = diff[0]
        assert sup_row[q] < 0 and top2_gap(ol[q]) <= GAP_MIN, (t, q, int(gc[q]), int(oc[q]))
        w.forced += 1
        sup_g[:q + 1] = oc[:q + 1]
    for q in range(s.dep_steps):
        le = logits_rel_l2(gl[q], ol[q])
        w.logits = max(w.logits, le)
        assert le <= LOGITS_TOL, (t, q, le)
    assert np.array_equal(gc[sup_row >= 0], sup_row[sup_row >= 0])
    return oc


@pytest.mark.slow
def test_config4_stated_length_generator_loop(full):
    """64 frames of temporal stack + depformer from reset.  Frame 0 takes seeded IDs; from
    then on every stream is fed back, as the generator does: the text stream takes the
    previous greedy text token, audio stream k the previous frame's depth code k-1 (q0-7
    greedy, q8-15 supplied from seeded codes).  On the GPU the feedback stays on the
    device (ID -3) wherever its selections equal the oracle's.  PM_CONFIG4_FRAMES sets
    another length (the workload states 1000 frames, about 8 minutes of oracle time)."""
    s = full.shape
    N = int(os.environ.get("PM_CONFIG4_FRAMES", "64"))
    full.ctx.reset()
    st = full.orc.new_stream()
    ids0 = I.make_ids(s, 1, seed=2014)[0, 0]
    sup = I.make_supplied_codes(s, N, seed=4000)[:, 0]
    w = Worst()
    prev_r = prev_g = None
    for t in range(N):
        if t == 0:
            r_ids = ids0.copy()
            g_ids = ids0[None].copy()
        else:
            r_ids = prev_r.copy()
            g_ids = np.where(prev_g == prev_r, -3, prev_r)[None].astype(np.int32)
        gh, gl, gt = full.gpu_frame(g_ids)
        rh, _, rl, rt = st.step(r_ids)
        _check(w, gh[0], gl[0], rh, rl, f"t={t}")
        _token(w, gt[0], rt, rl, f"t={t}")
        text = int(rt)
        oc = _depformer_lockstep(full, w, t, rh, text, sup[t])
        # the GPU's own selections this frame: its text token and the codes it produced
        # (the oracle's text token was supplied to its depformer)
        prev_r = np.concatenate([[text], oc]).astype(np.int32)
        prev_g = np.concatenate([[int(gt[0])], full.dcodes[0].cpu().numpy()]).astype(np.int32)
    record_parity(f"config4_{N}_frames_generator_loop", **w.asdict())
    del st

