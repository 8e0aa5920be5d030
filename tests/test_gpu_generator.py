"""pm_generator_step (the generator's token ring and provided ring, "PersonaPlex native LM
audit" section 7 "One exact generator step") against the oracle's restatement of the
seven steps (oracle/generator.py), bit-exact on every integer output.

The session follows the startup order of the audit's section 9: voice-prompt frames, six
silence frames, system text one token per frame, six silence frames -- every stream
provided (seeded stand-ins for the agent's voice / silence codes and the user's sine
codes, text pad ID 3 outside the system text) -- then live frames in which only the user's
codebooks are provided and the model selects text and agent codes.

Lockstep: a greedy selection may differ between the two sides only where the oracle's
top-2 logit gap is at most 1e-2.  The oracle runs one call ahead; wherever its selection
at such a near tie would be a target of the GPU's next call, that value is handed to the
GPU as a forced (provided) code, which the step places with the stream's delay -- so both
sides continue from the same ring.  Every other selection must match exactly, and the
model outputs (text logits, hidden state, depth logits) must match at the parity
tolerances.
"""
import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I

from harness import GAP_MIN, Pair, Worst, hidden_err, logits_rel_l2, record_parity, small_shape, top2_gap

pytestmark = pytest.mark.gpu


def _session(s, n_live, seed):
    """Provided codes per call [n][17] (-1: not provided): the startup prefix, then live
    calls with the user's codebooks only."""
    rng = np.random.default_rng(seed)
    sine = rng.integers(0, s.dep_card, 8)
    silence = rng.integers(0, s.dep_card, 8)
    voice = rng.integers(0, s.dep_card, (4, 8))
    system = rng.integers(4, s.text_out, 5)
    rows = []
    for v in voice:
        rows.append([3] + list(v) + list(sine))
    rows += [[3] + list(silence) + list(sine)] * 6
    for t in system:
        rows.append([int(t)] + list(silence) + list(sine))
    rows += [[3] + list(silence) + list(sine)] * 6
    n_prefix = len(rows)
    for _ in range(n_live):
        rows.append([-1] * 9 + list(rng.integers(0, s.dep_card, 8)))
    return np.array(rows, np.int32), n_prefix


class _Lockstep:
    """One stream: the oracle generator one call ahead of the GPU."""

    def __init__(self, pair, calls):
        from oracle.generator import Generator
        self.gen = Generator(pair.orc, pair.shape.asdict())
        self.calls = calls
        self.steps = []

    def oracle(self, c):
        while len(self.steps) <= c and len(self.steps) < len(self.calls):
            self.steps.append(self.gen.step(self.calls[len(self.steps)].tolist()))
        return self.steps[c] if c < len(self.steps) else (None, None)

    def forced(self, c, w):
        """The GPU's provided codes for call c: the session's, plus the oracle's near-tie
        selections that call c places (delay 0: this call's targets; delay 1: the next)."""
        row = self.calls[c].copy()
        _, last = self.oracle(c)
        if last is not None:
            h, lg, am, dl, codes = last
            if row[0] < 0 and top2_gap(lg) <= GAP_MIN:
                row[0] = am
                w.forced += 1
            if row[1] < 0 and top2_gap(dl[0]) <= GAP_MIN:
                row[1] = codes[0]
                w.forced += 1
        _, nxt = self.oracle(c + 1)
        if nxt is not None:
            _, _, _, dl, codes = nxt
            for q in range(1, 8):
                if row[q + 1] < 0 and top2_gap(dl[q]) <= GAP_MIN:
                    row[q + 1] = codes[q]
                    w.forced += 1
        return row


def _check_call(w, c, b, ls, out, valid, tl, hid, dl):
    o_out, last = ls.oracle(c)
    if o_out is None:
        assert valid[b] == 0 and np.all(out[b] == -1), (c, b)
    else:
        assert valid[b] == 1, (c, b)
        assert out[b].tolist() == o_out, (c, b, out[b].tolist(), o_out)
    if last is not None:
        h, lg, am, odl, codes = last
        he, le = hidden_err(hid[b], h), logits_rel_l2(tl[b], lg)
        w.add(he, le)
        assert he <= 2e-2 and le <= 1e-2, (c, b, he, le)
        for q in range(odl.shape[0]):
            lq = logits_rel_l2(dl[b, q], odl[q])
            w.logits = max(w.logits, lq)
            assert lq <= 1e-2, (c, b, q, lq)


def _run_calls(pair, B, lss, c_of_row, w):
    torch = pair.torch
    s = pair.shape
    prov = np.stack([ls.forced(c_of_row[b], w) for b, ls in enumerate(lss)]).astype(np.int32)
    out = torch.full((B, s.n_streams), -9, dtype=torch.int32, device="cuda")
    valid = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    dl = torch.zeros((B, s.dep_steps, s.dep_card), dtype=torch.float32, device="cuda")
    pair.ctx.generator_step(B, prov, out, valid, pair.logits, pair.hidden, dl)
    torch.cuda.synchronize()
    res = (out.cpu().numpy(), valid.cpu().numpy(), pair.logits[:B].double().cpu().numpy(),
           pair.hidden[:B].double().cpu().numpy(), dl.double().cpu().numpy())
    for b, ls in enumerate(lss):
        _check_call(w, c_of_row[b], b, ls, *res)
    return res


def test_generator_session_matches_oracle():
    s = small_shape()
    p = Pair(s, B_max=1)
    try:
        calls, n_prefix = _session(s, 24, seed=61)
        ls = _Lockstep(p, calls)
        w = Worst()
        for c in range(len(calls)):
            out, valid, _, _, _ = _run_calls(p, 1, [ls], [c], w)
            if n_prefix + 2 <= c:
                # live calls: the user's codebooks of the previous call come out aligned
                assert out[0, 9:].tolist() == calls[c - 1, 9:].tolist(), c
        assert len(calls) >= 32
        # the temporal position advanced once per model step (every call but the first)
        assert p.ctx.get_positions()[0] == len(calls) - 1
        record_parity("generator_session_B1", **w.asdict())
    finally:
        p.close()


def test_generator_batch_with_a_stream_reset_midway():
    """Two streams on the batched path; stream 1 is reset after five calls, so it meets
    the generator's first call (no model step) while stream 0 runs: its frame is undone
    and both streams stay equal to their own oracle generators."""
    s = small_shape()
    p = Pair(s, B_max=2)
    try:
        calls0, _ = _session(s, 16, seed=62)
        calls1, _ = _session(s, 16, seed=63)
        ls = [_Lockstep(p, calls0), _Lockstep(p, calls1)]
        w = Worst()
        c1 = 0
        for c in range(len(calls0) - 6):
            if c == 5:
                p.ctx.reset([0, 1])
                ls[1] = _Lockstep(p, calls1)
                c1 = 0
            _run_calls(p, 2, ls, [c, c1], w)
            c1 += 1
        pos = p.ctx.get_positions()
        assert pos[0] == len(calls0) - 6 - 1 and pos[1] == c1 - 1, pos
        record_parity("generator_B2_with_reset", **w.asdict())
    finally:
        p.close()


def test_generator_state_travels_in_a_snapshot():
    """Snapshot mid-session, restore into a fresh context: the continuation is
    bit-identical (the token ring, provided ring and offset are part of the snapshot)."""
    s = small_shape()
    a = Pair(s, B_max=1)
    b = Pair(s, B_max=1, weights=a.W)
    torch = a.torch
    try:
        calls, _ = _session(s, 12, seed=64)
        out = torch.zeros((1, s.n_streams), dtype=torch.int32, device="cuda")
        for c in range(20):
            a.ctx.generator_step(1, calls[c:c + 1], out)
        snap = torch.empty(a.ctx.snapshot_bytes(), dtype=torch.uint8, device="cuda")
        a.ctx.snapshot(0, snap)
        b.ctx.restore(0, snap)
        oa = torch.zeros_like(out)
        ob = torch.zeros_like(out)
        for c in range(20, len(calls)):
            a.ctx.generator_step(1, calls[c:c + 1], oa, None, a.logits)
            b.ctx.generator_step(1, calls[c:c + 1], ob, None, b.logits)
            torch.cuda.synchronize()
            assert torch.equal(oa, ob) and torch.equal(a.logits, b.logits), c
    finally:
        a.close()
        b.close()
