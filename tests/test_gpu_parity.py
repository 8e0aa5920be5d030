"""GPU parity at small shapes: the CUDA path through the C ABI against the float64 oracle
on the same seeded bf16 inputs, frame by frame.

Shapes are small enough for the oracle to finish in seconds yet span several GEMV tiles
per CTA with ragged unit ranges, the K = 2816 / 768 GEMV variants, and a 32-frame ring
that wraps.
"""
import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I

from harness import GAP_MIN, Pair, hidden_err, logits_rel_l2, small_shape, top2_gap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pair():
    p = Pair(small_shape(), B_max=4)
    yield p
    p.close()


def test_decode_parity_with_ring_wrap(pair):
    s = pair.shape
    pair.ctx.reset()
    pair.streams[0] = pair.orc.new_stream()
    T = 2 * s.ctx + 5
    ids = I.make_ids(s, T, seed=11)[:, 0]
    worst = 0.0
    for t in range(T):
        g = pair.gpu_frame(ids[t:t + 1])
        r = pair.oracle_frame(ids[t:t + 1])
        worst = max(worst, pair.check_frame(g, r, f"t={t}"))
    assert pair.ctx.get_positions()[0] == T
    print(f"worst hidden err {worst:.3e}")


def test_greedy_text_feedback_on_device(pair):
    """Text ID -3 makes the frame read the previous frame's greedy token on the device.
    The oracle feeds back its own token; both run until a near-tie (top-2 gap below 1e-2)
    is resolved differently, which may happen only at a near-tie."""
    s = pair.shape
    pair.ctx.reset()
    st = pair.orc.new_stream()
    T = 20
    ids = I.make_ids(s, T, seed=12)[:, 0]
    prev = None
    for t in range(T):
        gids = ids[t:t + 1].copy()
        rids = ids[t].copy()
        if t > 0:
            gids[0, 0] = -3
            rids[0] = prev
        gh, gl, gt = pair.gpu_frame(gids)
        rh, _, rl, rt = st.step(rids)
        assert hidden_err(gh[0], rh) <= 2e-2, t
        assert logits_rel_l2(gl[0], rl) <= 1e-2, t
        if int(gt[0]) != rt:
            assert top2_gap(rl) <= GAP_MIN, (t, int(gt[0]), rt)
            break
        prev = rt


def test_depformer_parity(pair):
    s = pair.shape
    pair.ctx.reset()
    st = pair.orc.new_stream()
    ids = I.make_ids(s, 3, seed=13)[:, 0]
    sup = I.make_supplied_codes(s, 3, seed=14)[:, 0]
    for t in range(3):
        gh, _, gt = pair.gpu_frame(ids[t:t + 1])
        rh, _, rl, rt = st.step(ids[t])
        text = int(rt)
        # (a) greedy run, compare along the chain until a near-tie diverges it
        pair.ctx.depformer_step(1, hidden=pair.hidden, text_tok=np.array([text], np.int32),
                                supplied=np.ascontiguousarray(sup[t:t + 1]), logits=pair.dlogits,
                                codes=pair.dcodes)
        pair.torch.cuda.synchronize()
        gl = pair.dlogits[0].double().cpu().numpy()
        gc = pair.dcodes[0].cpu().numpy()
        ol, oc = pair.orc.depformer_step(rh, text, sup[t])
        for q in range(s.dep_steps):
            assert logits_rel_l2(gl[q], ol[q]) <= 1e-2, (t, q)
            if gc[q] != oc[q]:
                assert sup[t, q] < 0 and top2_gap(ol[q]) <= GAP_MIN, (t, q, gc[q], oc[q])
                break
        # (b) lockstep: the oracle's codes supplied at every position -> every logit comparable
        pair.ctx.depformer_step(1, hidden=pair.hidden, text_tok=np.array([text], np.int32),
                                supplied=oc.astype(np.int32)[None].copy(), logits=pair.dlogits,
                                codes=pair.dcodes)
        pair.torch.cuda.synchronize()
        ol2, oc2 = pair.orc.depformer_step(rh, text, oc.astype(np.int32))
        gl2 = pair.dlogits[0].double().cpu().numpy()
        for q in range(s.dep_steps):
            assert logits_rel_l2(gl2[q], ol2[q]) <= 1e-2, (t, q)
        assert np.array_equal(pair.dcodes[0].cpu().numpy(), oc)


def test_batched_ragged_history(pair):
    """B = 4 streams with per-stream positions and seeded K/V history written directly into
    the cache (lengths below, at and past the 32-frame window)."""
    s = pair.shape
    torch = pair.torch
    B = 4
    L = np.array([5, 31, 32, 45], np.int32)
    pair.ctx.reset()
    streams = [pair.orc.new_stream() for _ in range(B)]
    kv = pair.kv  # [layers, 2, B_max, H, ctx, dh] bf16
    for b in range(B):
        for l in range(s.n_layers):
            k, v = I.make_kv_history(s, int(L[b]), seed=21, layer=l, stream=b)
            streams[b].load_kv(l, 0, k, v)
            # ring slot of position p is p mod ctx; later positions overwrite earlier ones
            for p0 in range(int(L[b])):
                slot = p0 % s.ctx
                kv[l, 0, b, :, slot, :] = torch.from_numpy(k[:, p0, :].astype(np.int16)).view(torch.bfloat16).cuda()
                kv[l, 1, b, :, slot, :] = torch.from_numpy(v[:, p0, :].astype(np.int16)).view(torch.bfloat16).cuda()
        streams[b].set_position(int(L[b]))
    pair.ctx.set_positions(list(L))
    ids = I.make_ids(s, 4, B=B, seed=22)
    for t in range(4):
        g = pair.gpu_frame(ids[t], B=B)
        outs = [streams[b].step(ids[t, b]) for b in range(B)]
        r = (np.stack([o[0] for o in outs]), np.stack([o[2] for o in outs]), np.array([o[3] for o in outs]))
        pair.check_frame(g, r, f"t={t}")
    assert pair.ctx.get_positions()[:B] == list(L + 4)


@pytest.mark.parametrize("B,flags", [(12, 0), (20, 0), (12, 8)])
def test_batched_paths_by_batch_size(B, flags):
    """B = 12: the batched GEMV with two 8-column MMA groups (B <= 16); B = 20: the
    tensor-core path (N = 32); B = 12 with PM_FLAG_BATCHED_TCGEN05 (8): the tensor-core
    path for a batch the GEMV would take.  Streams start at staggered positions with
    seeded K/V history and run past the ring's wrap."""
    s = small_shape()
    p = Pair(s, B_max=B, depformer=False, flags=flags)
    try:
        torch = p.torch
        L = 1 + (np.arange(B, dtype=np.int32) * 7) % (s.ctx + 9)
        for b in range(B):
            for l in range(s.n_layers):
                k, v = I.make_kv_history(s, int(L[b]), seed=31, layer=l, stream=b)
                p.streams[b].load_kv(l, 0, k, v)
                for p0 in range(int(L[b])):
                    slot = p0 % s.ctx
                    p.kv[l, 0, b, :, slot, :] = torch.from_numpy(k[:, p0, :].astype(np.int16)).view(torch.bfloat16).cuda()
                    p.kv[l, 1, b, :, slot, :] = torch.from_numpy(v[:, p0, :].astype(np.int16)).view(torch.bfloat16).cuda()
            p.streams[b].set_position(int(L[b]))
        p.ctx.set_positions(list(L))
        ids = I.make_ids(s, 3, B=B, seed=32)
        for t in range(3):
            p.check_frame(p.gpu_frame(ids[t], B=B), p.oracle_frame(ids[t]), f"B={B} t={t}")
        assert p.ctx.get_positions()[:B] == list(L + 3)
    finally:
        p.close()


def test_invalid_ids_leave_state_unchanged(pair):
    from full_duplex_speech_moshi_gb300 import pm
    s = pair.shape
    pair.ctx.reset()
    st = pair.orc.new_stream()
    ids = I.make_ids(s, 3, seed=15)[:, 0]
    pair.check_frame(pair.gpu_frame(ids[0:1]), _orc(st, ids[0]))
    # host memory: rejected before any launch
    for bad in (-2, s.text_in, -4):
        b = ids[1:2].copy()
        b[0, 0] = bad
        with pytest.raises(pm.PMError) as e:
            pair.ctx.frame_step(1, b, pair.logits, pair.hidden, pair.token)
        assert e.value.status == pm.PM_ERR_INVALID_ID
    b = ids[1:2].copy()
    b[0, 5] = s.audio_in
    with pytest.raises(pm.PMError):
        pair.ctx.frame_step(1, b, pair.logits, pair.hidden, pair.token)
    assert pair.ctx.get_positions()[0] == 1
    # device memory: the frame becomes a no-op, reported by pm_device_status
    bd = pair.torch.from_numpy(ids[1:2].copy()).cuda()
    bd[0, 3] = -2
    pair.ctx.frame_step(1, bd, pair.logits, pair.hidden, pair.token)
    assert pair.ctx.device_status() == pm.PM_ERR_INVALID_ID
    assert pair.ctx.device_status() == pm.PM_OK  # cleared
    assert pair.ctx.get_positions()[0] == 1
    # the stream continues exactly as if the bad frame had never been sent
    for t in (1, 2):
        pair.check_frame(pair.gpu_frame(ids[t:t + 1]), _orc(st, ids[t]), f"t={t}")


def _orc(st, ids):
    h, _, lg, a = st.step(ids)
    return h[None], lg[None], np.array([a])


def test_reset_replays_bit_identically(pair):
    s = pair.shape
    ids = I.make_ids(s, 6, seed=16)[:, 0]
    runs = []
    for _ in range(2):
        pair.ctx.reset()
        outs = [pair.gpu_frame(ids[t:t + 1]) for t in range(6)]
        runs.append(outs)
    for a, b in zip(*runs):
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])


def test_single_block_tiny_shapes():
    """The smallest supported shapes (K = 256 / 512 GEMV variants, one CTA per unit)."""
    p = Pair(I.tiny_shape(), B_max=1)
    try:
        ids = I.make_ids(p.shape, 20, seed=17)[:, 0]
        for t in range(20):
            p.check_frame(p.gpu_frame(ids[t:t + 1]), p.oracle_frame(ids[t:t + 1]), f"t={t}")
        # depformer on the next frame's hidden state: the oracle runs greedy, and its
        # codes are supplied to the GPU so that every position's logits are comparable
        rh, _, _, rt = p.streams[0].step(ids[0])
        p.gpu_frame(ids[0:1])
        oc_l, oc = p.orc.depformer_step(rh, int(rt), np.full(p.shape.dep_steps, -1, np.int32))
        p.ctx.depformer_step(1, hidden=p.hidden, text_tok=np.array([int(rt)], np.int32),
                             supplied=oc.astype(np.int32)[None].copy(), logits=p.dlogits, codes=p.dcodes)
        p.torch.cuda.synchronize()
        gl = p.dlogits[0].double().cpu().numpy()
        for q in range(p.shape.dep_steps):
            assert logits_rel_l2(gl[q], oc_l[q]) <= 1e-2, q
    finally:
        p.close()


def test_frame_program_small_shapes():
    """The persistent single-launch frame program (D, ffn multiples of 1024) against the
    oracle: ring wrap, device-side greedy feedback, invalid device IDs as a no-op."""
    from full_duplex_speech_moshi_gb300 import pm
    s = small_shape(ffn=3072, ctx=96)
    p = Pair(s, B_max=1, depformer=False, flags=pm.PM_FLAG_FRAME_PROGRAM)
    try:
        T = 2 * s.ctx + 7
        ids = I.make_ids(s, T, seed=31)[:, 0]
        for t in range(T):
            p.check_frame(p.gpu_frame(ids[t:t + 1]), p.oracle_frame(ids[t:t + 1]), f"t={t}")
        assert p.ctx.get_positions()[0] == T
        # an invalid ID in device memory leaves the state unchanged
        bd = p.torch.from_numpy(ids[0:1].copy()).cuda()
        bd[0, 2] = -2
        p.ctx.frame_step(1, bd, p.logits, p.hidden, p.token)
        assert p.ctx.device_status() == pm.PM_ERR_INVALID_ID
        assert p.ctx.get_positions()[0] == T
        # greedy feedback on the device continues the same stream
        st = p.streams[0]
        more = I.make_ids(s, 6, seed=32)[:, 0]
        prev = None
        for t in range(6):
            gids = more[t:t + 1].copy()
            rids = more[t].copy()
            if t > 0:
                gids[0, 0] = -3
                rids[0] = prev
            gh, gl, gt = p.gpu_frame(gids)
            rh, _, rl, rt = st.step(rids)
            assert hidden_err(gh[0], rh) <= 2e-2 and logits_rel_l2(gl[0], rl) <= 1e-2, t
            if int(gt[0]) != rt:
                assert top2_gap(rl) <= GAP_MIN
                break
            prev = rt
    finally:
        p.close()


def test_frame_program_matches_kernel_chain():
    """Both batch-1 implementations (one persistent launch, one kernel per step) on the
    same inputs agree to the parity tolerances at every frame."""
    from full_duplex_speech_moshi_gb300 import pm
    s = small_shape(ffn=3072, ctx=48)
    a = Pair(s, B_max=1, depformer=False, flags=pm.PM_FLAG_FRAME_PROGRAM)
    try:
        b_kv = pm.alloc_kv_cache(a.cfg)
        b = pm.Context(s.asdict(), a.Wd, b_kv, B_max=1, depformer=False,
                       stream=a.torch.cuda.current_stream().cuda_stream)
        ids = I.make_ids(s, 60, seed=33)[:, 0]
        lg = a.torch.zeros_like(a.logits)
        hd = a.torch.zeros_like(a.hidden)
        for t in range(60):
            ga = a.gpu_frame(ids[t:t + 1])
            b.frame_step(1, np.ascontiguousarray(ids[t:t + 1]), lg, hd, None)
            a.torch.cuda.synchronize()
            assert hidden_err(ga[0][0], hd[0].double().cpu().numpy()) <= 1e-3, t
            assert logits_rel_l2(ga[1][0], lg[0].double().cpu().numpy()) <= 1e-3, t
        b.close()
    finally:
        a.close()


def test_pinned_ring_mode_parity():
    """PM_FLAG_PINNED_RING: the attention windows of the pinned ring cache (a full ring
    hides its oldest key; "PersonaPlex native LM audit", section 6), temporal (B = 1 GEMV
    path and B = 2 tensor-core path, through two ring wraps) and depth, against the
    oracle's pinned-ring mode."""
    s = small_shape(pinned_ring=1)
    p = Pair(s, B_max=2)
    try:
        for B in (1, 2):
            p.ctx.reset()
            streams = [p.orc.new_stream() for _ in range(B)]
            T = 2 * s.ctx + 3
            ids = I.make_ids(s, T, B=B, seed=71 + B)
            for t in range(T):
                g = p.gpu_frame(ids[t], B=B)
                outs = [streams[b].step(ids[t, b]) for b in range(B)]
                r = (np.stack([o[0] for o in outs]), np.stack([o[2] for o in outs]), np.array([o[3] for o in outs]))
                p.check_frame(g, r, f"B={B} t={t}")
        # depth: the oracle's codes supplied everywhere, so every position's logits compare
        p.ctx.reset()
        st = p.orc.new_stream()
        ids = I.make_ids(s, 2, seed=75)[:, 0]
        for t in range(2):
            gh, _, _ = p.gpu_frame(ids[t:t + 1])
            rh, _, _, rt = st.step(ids[t])
            sup = np.full(s.dep_steps, -1, np.int32)
            ol, oc = p.orc.depformer_step(rh, int(rt), sup)
            p.ctx.depformer_step(1, hidden=p.hidden, text_tok=np.array([int(rt)], np.int32),
                                 supplied=oc.astype(np.int32)[None].copy(), logits=p.dlogits, codes=p.dcodes)
            p.torch.cuda.synchronize()
            gl = p.dlogits[0].double().cpu().numpy()
            for q in range(s.dep_steps):
                assert logits_rel_l2(gl[q], ol[q]) <= 1e-2, (t, q)
    finally:
        p.close()


@pytest.mark.parametrize("B", [2, 8, 16])
def test_batched_replays_bit_identical(B):
    """The batched paths (batched GEMV on warp MMAs, head-per-cluster or balanced-split
    attention) merge partial sums in a fixed order: replaying the same frames from the same
    state reproduces every bit.  A missing ordering between a slot's reads and the bulk copy
    that refills it shows up here as replays that differ."""
    s = small_shape()
    p = Pair(s, B_max=B, depformer=False)
    try:
        pos = [int(v) for v in (np.arange(B) * 5 % 40 + 3)]
        ids = I.make_ids(s, 3, B=B, seed=51)
        runs = []
        for _ in range(3):
            # same state every time: the ring is cleared too (streams past the 32-slot
            # wrap would otherwise read the slots the previous replay wrote)
            p.kv.zero_()
            p.ctx.reset()
            p.ctx.set_positions(pos)
            runs.append([p.gpu_frame(ids[t], B=B) for t in range(3)])
        for other in runs[1:]:
            for a, b in zip(runs[0], other):
                assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    finally:
        p.close()
