"""The streaming Mimi decoder (include/pm_mimi.h) against the oracle's non-streaming
float64 decode of the same code frames (oracle/mimi.py; "PersonaPlex native LM audit",
chapter "Exact Mimi codec construction", and its rule that streaming emits exactly the
non-streaming causal result frame by frame).

Tolerance: per 80 ms frame, relative L2 of the PCM <= 1e-4.  The GPU computes in fp32
with the oracle's bf16 weights widened exactly; each output is a chain of about 30
dependent reductions (front projections, 8 blocks x 4 projections, 13 SEANet
convolutions) of at most 3,584 terms, and an fp32 sum of K terms carries a relative error
of order sqrt(K) * 2^-24 ~ 4e-6; thirty such stages bound the drift near 1e-4.
ELU (expm1f), GELU (erff) and the softmax's exp2f are within a few ulp.

Cases: the small shape (two blocks, a 6-position window outrun every three frames, two
SEANet stages) at B = 1 and at B = 3 with a stream reset midway; host and device codes
bit-identical; an invalid device code (the call is a no-op, zeros out, reported by
pm_mimi_status) and an invalid host code (refused before launch); a replay after reset
bit-identical; the full shape at B = 1 and B = 8 (ragged: B = 5 calls on the B_max = 8
context); the full shape for 130 frames, past the 250-position window (slow).
"""
import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I

from harness import record_parity

pytestmark = pytest.mark.gpu

TOL = 1e-4


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


class MimiPair:
    def __init__(self, shape, B_max, seed=5000):
        import torch
        from full_duplex_speech_moshi_gb300 import pm
        from oracle import mimi as M
        self.torch, self.pm, self.M = torch, pm, M
        self.shape = shape
        self.W = I.make_mimi_weights(shape, base_seed=seed)
        self.Wd = pm.upload_weights(self.W)
        self.dec = pm.MimiDecoder(shape, self.Wd, B_max=B_max)
        self.fs = pm.mimi_frame_samples(shape)
        self.orc = M.MimiDecoderOracle(M.MimiShape(**shape), self.W)

    def oracle(self, codes):
        """codes [T][n_q] from reset -> PCM [T][frame_samples] (float64)."""
        return self.orc.decode(np.asarray(codes)).reshape(len(codes), self.fs)

    def step(self, codes_b, device_codes=False):
        """One call on B = len(codes_b) streams; returns PCM [B][fs] float64."""
        torch = self.torch
        B = len(codes_b)
        pcm = torch.full((B, self.fs), float("nan"), dtype=torch.float32, device="cuda")
        c = np.ascontiguousarray(codes_b, dtype=np.int32)
        if device_codes:
            c = torch.from_numpy(c).cuda()
        self.dec.decode(B, c, pcm)
        torch.cuda.synchronize()
        return pcm.double().cpu().numpy()

    def close(self):
        self.dec.close()


def _stream(pair, codes, name):
    """Decode codes [T][B][n_q] frame by frame; compare each stream with the oracle."""
    T, B, _ = codes.shape
    got = np.stack([pair.step(codes[t]) for t in range(T)])  # [T][B][fs]
    worst = 0.0
    for b in range(B):
        ref = pair.oracle(codes[:, b])
        for t in range(T):
            e = _rel_l2(got[t, b], ref[t])
            worst = max(worst, e)
            assert e <= TOL, (name, b, t, e)
    record_parity(name, frames=T * B, worst_pcm_rel_l2=worst)
    return got


def test_small_shape_streaming_B1():
    p = MimiPair(I.MIMI_SMALL, B_max=1)
    try:
        codes = I.make_mimi_codes(I.MIMI_SMALL, 12, 1, seed=1)
        _stream(p, codes, "mimi_small_B1_12_frames")
        assert p.dec.frames()[0] == 12
    finally:
        p.close()


def test_small_shape_three_streams_with_a_reset():
    p = MimiPair(I.MIMI_SMALL, B_max=3)
    try:
        codes = I.make_mimi_codes(I.MIMI_SMALL, 10, 3, seed=2)
        got = [p.step(codes[t]) for t in range(4)]
        p.dec.reset([0, 1, 0])
        got += [p.step(codes[t]) for t in range(4, 10)]
        got = np.stack(got)
        worst = 0.0
        for b in range(3):
            c = codes[:, b] if b != 1 else codes[4:, 1]
            ref = p.oracle(c)
            g = got[:, b] if b != 1 else got[4:, 1]
            for t in range(len(c)):
                e = _rel_l2(g[t], ref[t])
                worst = max(worst, e)
                assert e <= TOL, (b, t, e)
        assert p.dec.frames() == [10, 6, 10]
        record_parity("mimi_small_B3_reset", frames=26, worst_pcm_rel_l2=worst)
    finally:
        p.close()


def test_host_and_device_codes_agree_and_replay_is_identical():
    p = MimiPair(I.MIMI_SMALL, B_max=2)
    try:
        codes = I.make_mimi_codes(I.MIMI_SMALL, 6, 2, seed=3)
        a = np.stack([p.step(codes[t]) for t in range(6)])
        p.dec.reset()
        b = np.stack([p.step(codes[t], device_codes=True) for t in range(6)])
        assert np.array_equal(a, b)
        assert p.dec.status() == p.pm.PM_OK
    finally:
        p.close()


def test_invalid_codes():
    p = MimiPair(I.MIMI_SMALL, B_max=2)
    pm = p.pm
    try:
        codes = I.make_mimi_codes(I.MIMI_SMALL, 5, 2, seed=4)
        out = [p.step(codes[t]) for t in range(2)]
        # device code out of range: the call is a no-op and its PCM is zeros
        bad = codes[2].copy()
        bad[1, 3] = I.MIMI_SMALL["card"]
        z = p.step(bad, device_codes=True)
        assert np.all(z == 0.0)
        assert p.dec.status() == pm.PM_ERR_INVALID_ID
        assert p.dec.status() == pm.PM_OK  # reading clears it
        assert p.dec.frames() == [2, 2]
        # host code out of range: refused before launch
        bad[1, 3] = -1
        with pytest.raises(pm.PMError) as ei:
            p.step(bad)
        assert ei.value.status == pm.PM_ERR_INVALID_ID
        assert p.dec.frames() == [2, 2]
        # the streams continue as if neither call had been made
        out += [p.step(codes[t]) for t in range(2, 5)]
        out = np.stack(out)
        for b in range(2):
            ref = p.oracle(codes[:, b])
            for t in range(5):
                assert _rel_l2(out[t, b], ref[t]) <= TOL, (b, t)
    finally:
        p.close()


def test_pcm_into_pinned_host_memory():
    p = MimiPair(I.MIMI_SMALL, B_max=1)
    torch = p.torch
    try:
        codes = I.make_mimi_codes(I.MIMI_SMALL, 3, 1, seed=5)
        dev = np.stack([p.step(codes[t]) for t in range(3)])
        p.dec.reset()
        host = torch.empty((1, p.fs), dtype=torch.float32).pin_memory()
        for t in range(3):
            p.dec.decode(1, codes[t], host)
            torch.cuda.synchronize()
            assert np.array_equal(host.double().numpy(), dev[t])
    finally:
        p.close()


@pytest.fixture(scope="module")
def full8():
    p = MimiPair(I.MIMI_FULL, B_max=8)
    yield p
    p.close()


def test_full_shape_B1(full8):
    full8.dec.reset()
    codes = I.make_mimi_codes(I.MIMI_FULL, 8, 1, seed=6)
    _stream(full8, codes, "mimi_full_B1_8_frames")


def test_full_shape_B8_and_a_ragged_call(full8):
    full8.dec.reset()
    codes = I.make_mimi_codes(I.MIMI_FULL, 4, 8, seed=7)
    got = np.stack([full8.step(codes[t]) for t in range(4)])
    # a B = 5 call on the B_max = 8 context advances only streams 0..4
    extra = I.make_mimi_codes(I.MIMI_FULL, 1, 5, seed=8)[0]
    five = full8.step(extra)
    assert full8.dec.frames() == [5] * 5 + [4] * 3
    worst = 0.0
    for b in range(8):
        ref = full8.oracle(codes[:, b])
        for t in range(4):
            e = _rel_l2(got[t, b], ref[t])
            worst = max(worst, e)
            assert e <= TOL, (b, t, e)
        if b < 5:
            ref5 = full8.oracle(np.concatenate([codes[:, b], extra[b:b + 1]]))
            e = _rel_l2(five[b], ref5[4])
            worst = max(worst, e)
            assert e <= TOL, (b, e)
    record_parity("mimi_full_B8_4_frames_plus_B5", frames=37, worst_pcm_rel_l2=worst)


@pytest.mark.slow
def test_full_shape_past_the_window():
    """130 frames = 260 positions: the last frames attend over a window that has slid."""
    p = MimiPair(I.MIMI_FULL, B_max=1)
    try:
        codes = I.make_mimi_codes(I.MIMI_FULL, 130, 1, seed=9)
        _stream(p, codes, "mimi_full_B1_130_frames")
    finally:
        p.close()
