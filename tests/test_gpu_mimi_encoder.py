"""The streaming Mimi encoder (pm_mimi_encode) against the oracle's non-streaming float64
encode of the same PCM (oracle/mimi.py MimiEncoderOracle; "PersonaPlex native LM audit",
chapter "Exact Mimi codec construction": the ENCODE order, the SEANet encoder stages, the
replicate-padded downsampler and the split quantizer).

Latent: per frame relative L2 <= 1e-4 (fp32 arithmetic on the oracle's bf16 weights; about
30 dependent reductions of at most 4,096 terms: the same bound as the decoder's).

Codes: both sides pick the nearest entry per level, the GPU on its fp32 residual, the
oracle on its float64 one.  Where the oracle's gap between the best and second-best squared
distance exceeds 1e-4 of the best distance, the codes must be equal.  Below that margin
(a near tie: the two residuals differ by the latent's rounding) the GPU's code must be
within the margin of the best, and the oracle continues its residual chain from the GPU's
code (lockstep), so later levels stay comparable.
"""
import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I

from harness import record_parity

pytestmark = pytest.mark.gpu

TOL = 1e-4
GAP_REL = 1e-4


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


class EncPair:
    def __init__(self, shape, B_max, seed=7000):
        import torch
        from full_duplex_speech_moshi_gb300 import pm
        from oracle import mimi as M
        self.torch, self.pm, self.M = torch, pm, M
        self.shape = shape
        self.W = I.make_mimi_encoder_weights(shape, base_seed=seed)
        self.Wd = pm.upload_weights(self.W)
        self.enc = pm.MimiEncoder(shape, self.Wd, B_max=B_max)
        self.fs = pm.mimi_frame_samples(shape)
        self.n_q = dict(I.MIMI_FULL, **shape)["n_q"]
        self.orc = M.MimiEncoderOracle(M.MimiShape(**shape), self.W)

    def step(self, pcm_b, device_pcm=False):
        """One call on B = len(pcm_b) streams -> (codes [B][n_q], latent [B][dim])."""
        torch = self.torch
        B = len(pcm_b)
        codes = torch.full((B, self.n_q), -7, dtype=torch.int32, device="cuda")
        lat = torch.full((B, self.orc.s.dim), float("nan"), dtype=torch.float32, device="cuda")
        x = np.ascontiguousarray(pcm_b, dtype=np.float32)
        if device_pcm:
            x = torch.from_numpy(x).cuda()
        self.enc.encode(B, x, codes, lat)
        torch.cuda.synchronize()
        return codes.cpu().numpy(), lat.double().cpu().numpy()

    def check_stream(self, pcm, codes, lats, w, skip_codes=()):
        """pcm [F * fs] from reset, the GPU's codes [F][n_q] and latents [F][dim]; the codes
        of frames in skip_codes are not compared."""
        ref = self.orc.latent(pcm.astype(np.float64))
        cbs = [self.orc.W[f"q.codebook.{j}"] for j in range(self.n_q)]
        for f in range(len(codes)):
            e = _rel_l2(lats[f], ref[f])
            w["latent"] = max(w["latent"], e)
            assert e <= TOL, (f, e)
            if f in skip_codes:
                continue
            forced = [-1] * self.n_q
            oc, gaps = self.orc.quantize(ref[f])
            for j in range(self.n_q):
                # redo the level with the codes so far forced (lockstep), on the oracle's residual
                oc, gaps = self.orc.quantize(ref[f], forced)
                v = (self.orc.W["q.sem.in"] if j == 0 else self.orc.W["q.ac.in"]) @ ref[f]
                if j > 0:
                    for jj in range(1, j):
                        v = v - cbs[jj][oc[jj]]
                d = ((cbs[j] - v[None, :]) ** 2).sum(1)
                best = d.min()
                if gaps[j] > GAP_REL * best:
                    assert codes[f][j] == oc[j], (f, j, codes[f][j], oc[j], gaps[j])
                else:
                    assert d[codes[f][j]] <= best * (1 + GAP_REL), (f, j)
                    w["forced"] += int(codes[f][j] != oc[j])
                forced[j] = int(codes[f][j])
            w["frames"] += 1

    def close(self):
        self.enc.close()


def _worst():
    return {"latent": 0.0, "forced": 0, "frames": 0}


def _run(pair, pcm, name):
    """pcm [B][F * fs]: stream frame by frame, check every stream against the oracle."""
    B, N = pcm.shape
    F = N // pair.fs
    got = [pair.step(pcm[:, f * pair.fs:(f + 1) * pair.fs]) for f in range(F)]
    codes = np.stack([g[0] for g in got], axis=1)   # [B][F][n_q]
    lats = np.stack([g[1] for g in got], axis=1)
    w = _worst()
    for b in range(B):
        pair.check_stream(pcm[b], codes[b], lats[b], w)
    record_parity(name, frames=w["frames"], worst_latent_rel_l2=w["latent"], near_tie_codes_taken_from_gpu=w["forced"])
    return codes, lats


def test_small_shape_streaming_B1():
    p = EncPair(I.MIMI_SMALL, B_max=1)
    try:
        pcm = I.make_mimi_pcm(12 * p.fs, 1, seed=1)
        _run(p, pcm, "mimi_enc_small_B1_12_frames")
        assert p.enc.frames()[0] == 12
    finally:
        p.close()


def test_small_shape_three_streams_with_a_reset():
    p = EncPair(I.MIMI_SMALL, B_max=3)
    try:
        pcm = I.make_mimi_pcm(10 * p.fs, 3, seed=2)
        got = [p.step(pcm[:, f * p.fs:(f + 1) * p.fs]) for f in range(4)]
        p.enc.reset([0, 1, 0])
        got += [p.step(pcm[:, f * p.fs:(f + 1) * p.fs]) for f in range(4, 10)]
        codes = np.stack([g[0] for g in got], axis=1)
        lats = np.stack([g[1] for g in got], axis=1)
        w = _worst()
        for b in range(3):
            f0 = 4 if b == 1 else 0
            p.check_stream(pcm[b, f0 * p.fs:], codes[b, f0:], lats[b, f0:], w)
        assert p.enc.frames() == [10, 6, 10]
        record_parity("mimi_enc_small_B3_reset", frames=w["frames"], worst_latent_rel_l2=w["latent"],
                      near_tie_codes_taken_from_gpu=w["forced"])
    finally:
        p.close()


def test_host_and_device_pcm_agree_and_outputs_to_pinned_memory():
    p = EncPair(I.MIMI_SMALL, B_max=2)
    torch = p.torch
    try:
        pcm = I.make_mimi_pcm(5 * p.fs, 2, seed=3)
        a = [p.step(pcm[:, f * p.fs:(f + 1) * p.fs]) for f in range(5)]
        p.enc.reset()
        b = [p.step(pcm[:, f * p.fs:(f + 1) * p.fs], device_pcm=True) for f in range(5)]
        for x, y in zip(a, b):
            assert np.array_equal(x[0], y[0]) and np.array_equal(x[1], y[1])
        p.enc.reset()
        hc = torch.empty((2, p.n_q), dtype=torch.int32).pin_memory()
        for f in range(5):
            p.enc.encode(2, pcm[:, f * p.fs:(f + 1) * p.fs], hc)
            torch.cuda.synchronize()
            assert np.array_equal(hc.numpy(), a[f][0])
        # the wrong direction on a context is refused before anything runs
        assert p.enc.L.pm_mimi_decode(p.enc.h, 1, hc.data_ptr(), hc.data_ptr()) == p.pm.PM_ERR_STATE
    finally:
        p.close()


def test_a_quantiser_wait_that_runs_out():
    """With a poll budget of 0 the quantiser's copy waits give up at once: that call's codes
    are undefined and pm_mimi_status reports PM_ERR_TIMEOUT; the streaming state advances as
    usual, so with the budget restored the next frames match the oracle again."""
    p = EncPair(I.MIMI_SMALL, B_max=1)
    pm = p.pm
    try:
        pcm = I.make_mimi_pcm(6 * p.fs, 1, seed=13)
        frame = lambda f: pcm[:, f * p.fs:(f + 1) * p.fs]
        got = [p.step(frame(0)), p.step(frame(1))]
        assert p.enc.status() == pm.PM_OK
        p.enc.set_wait_budget(0)
        got.append(p.step(frame(2)))
        assert p.enc.status() == pm.PM_ERR_TIMEOUT
        assert p.enc.status() == pm.PM_OK  # reading clears it
        p.enc.set_wait_budget()
        got += [p.step(frame(f)) for f in range(3, 6)]
        assert p.enc.status() == pm.PM_OK and p.enc.frames()[0] == 6
        w = _worst()
        p.check_stream(pcm[0], np.stack([g[0][0] for g in got]), np.stack([g[1][0] for g in got]), w,
                       skip_codes=(2,))
    finally:
        p.close()


@pytest.fixture(scope="module")
def full8():
    p = EncPair(I.MIMI_FULL, B_max=8)
    yield p
    p.close()


def test_full_shape_B1(full8):
    full8.enc.reset()
    _run(full8, I.make_mimi_pcm(8 * full8.fs, 1, seed=4), "mimi_enc_full_B1_8_frames")


def test_full_shape_B8(full8):
    full8.enc.reset()
    _run(full8, I.make_mimi_pcm(4 * full8.fs, 8, seed=5), "mimi_enc_full_B8_4_frames")


@pytest.mark.slow
def test_full_shape_past_the_window():
    """130 frames = 260 positions of the encoder transformer: past its 250-position window."""
    p = EncPair(I.MIMI_FULL, B_max=1)
    try:
        _run(p, I.make_mimi_pcm(130 * p.fs, 1, seed=6), "mimi_enc_full_B1_130_frames")
    finally:
        p.close()
