"""GPU parity at the full model shapes of the decode-step workloads.

  config 0  one temporal block, B=1, 16 frames from an empty cache
  config 1  32-block stack, B=1, primed frames then greedy text fed back on the device
  config 2  32-block stack, B=1, 3000 cached positions (seeded K/V), decode past 3000
            so the ring wraps and keys keep absolute RoPE positions
  config 3  32-block stack, B=16, per-stream cache lengths uniform 64..3000 (seeded K/V)
  config 4  config 1 plus the depformer (dep_ctx 8, greedy q0-7, supplied q8-15)

The oracle runs sampled frames of each (it needs about 0.3 s per full frame on 16
cores); long histories are seeded K/V written identically to both sides, a stand-in
whose attention cost and semantics match a computed history.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I

from harness import GAP_MIN, Pair, hidden_err, logits_rel_l2, top2_gap

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
