"""pm_text_head_noalloc, the entry point for callers that cannot allocate device memory
(code running during CUDA stream capture, real-time threads that must not block on the
allocator, hosts that own all device memory): its scratch is a static device array in
the library instead of context workspaces.

It is checked two ways on the same residual stream: against the text head of
pm_frame_step, and against the float64 oracle's final RMSNorm -> text head -> argmax.  The
model has one block whose projections are all zero, so the frame's residual stream before
the final norm is exactly the embedding sum of the frame's delayed inputs; that sum,
formed here, is the no-allocation call's input.  Two calls in a row must each reproduce
both within the parity tolerances, a call with only the token output must give the same
token, and the call's status output must report PM_OK.

This file is collected last on purpose: a failure here leaves every other test run.
"""
import numpy as np
import pytest

from full_duplex_speech_moshi_gb300 import inputs as I

from harness import GAP_MIN, Pair, hidden_err, logits_rel_l2, small_shape, top2_gap

pytestmark = pytest.mark.gpu


def test_noalloc_text_head_matches_frame_step_and_oracle():
    from full_duplex_speech_moshi_gb300 import pm
    from oracle import oracle as O
    s = small_shape(n_layers=1)
    W = I.make_weights(s, depformer=False)
    for n in ("in_proj", "out_proj", "linear_in", "linear_out"):
        W[f"layers.0.{n}"][...] = 0
    p = Pair(s, B_max=2, depformer=False, weights=W)
    torch = p.torch
    try:
        B = 2
        ids = I.make_ids(s, 1, B=B, seed=91)[0]
        gh, gl, gt = p.gpu_frame(ids, B=B)        # existing entry point
        # residual = embedding sum of the first frame's inputs (delayed streams: initial IDs)
        inp = np.where(np.array(s.delays)[None, :] == 0, ids,
                       np.array([s.init_text] + [s.init_audio] * (s.n_streams - 1))[None, :])
        x = torch.zeros((B, s.D), dtype=torch.float32, device="cuda")
        for b in range(B):
            for k in range(s.n_streams):
                if inp[b, k] >= 0:
                    table = p.Wd["text_emb"] if k == 0 else p.Wd[f"emb.{k - 1}"]
                    x[b] += table[int(inp[b, k])].float()
        # the oracle's head on the same residual (float64)
        xr = x.double().cpu().numpy()
        oh = [O.rmsnorm(xr[b], W["out_norm"], s.eps) for b in range(B)]
        ol = [O.matvec(W["text_linear"], oh[b]) for b in range(B)]
        ot = [O.argmax(ol[b]) for b in range(B)]

        hid = torch.empty((B, s.D), dtype=torch.float32, device="cuda")
        lg = torch.empty((B, s.text_out), dtype=torch.float32, device="cuda")
        tok = torch.empty((B,), dtype=torch.int32, device="cuda")
        status = torch.empty((1,), dtype=torch.int32, device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        for call in range(2):
            hid.fill_(float("nan"))
            lg.fill_(float("nan"))
            tok.fill_(-7)
            status.fill_(-7)
            st = pm.pm_text_head_noalloc(B, s.D, s.text_out, x, p.Wd["out_norm"], p.Wd["text_linear"], s.eps,
                                         hid, lg, tok, status, stream)
            assert st == pm.PM_OK, st
            torch.cuda.synchronize()
            assert int(status[0]) == pm.PM_OK
            nh = hid.double().cpu().numpy()
            nl = lg.double().cpu().numpy()
            nt = tok.cpu().numpy()
            for b in range(B):
                assert hidden_err(nh[b], gh[b]) <= 2e-2, (call, b)
                assert logits_rel_l2(nl[b], gl[b]) <= 1e-2, (call, b)
                assert hidden_err(nh[b], oh[b]) <= 2e-2, (call, b, "oracle")
                assert logits_rel_l2(nl[b], ol[b]) <= 1e-2, (call, b, "oracle")
                if top2_gap(gl[b]) > GAP_MIN:
                    assert int(nt[b]) == int(gt[b]), (call, b)
                if top2_gap(ol[b]) > GAP_MIN:
                    assert int(nt[b]) == ot[b], (call, b, "oracle")
        # only the token requested (no hidden, no logits, no status)
        tok.fill_(-7)
        assert pm.pm_text_head_noalloc(B, s.D, s.text_out, x, p.Wd["out_norm"], p.Wd["text_linear"], s.eps,
                                       None, None, tok, None, stream) == pm.PM_OK
        torch.cuda.synchronize()
        assert np.array_equal(tok.cpu().numpy(), nt)
        # sizes beyond the static scratch and misaligned or host outputs are refused
        # without launching anything
        assert pm.pm_text_head_noalloc(65, s.D, s.text_out, x, p.Wd["out_norm"], p.Wd["text_linear"], s.eps,
                                       hid, lg, tok, status, stream) == pm.PM_ERR_UNSUPPORTED
        flat = torch.empty((B * s.D + 1,), dtype=torch.float32, device="cuda")
        assert pm.pm_text_head_noalloc(B, s.D, s.text_out, x, p.Wd["out_norm"], p.Wd["text_linear"], s.eps,
                                       flat[1:], lg, tok, status, stream) == pm.PM_ERR_ARG
        host_tok = np.zeros(B, np.int32)
        assert pm.pm_text_head_noalloc(B, s.D, s.text_out, x, p.Wd["out_norm"], p.Wd["text_linear"], s.eps,
                                       hid, lg, host_tok, status, stream) == pm.PM_ERR_ARG
    finally:
        p.close()
