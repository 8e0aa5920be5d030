"""The generator step (LMGen) of "PersonaPlex native LM audit", section 7 "One exact
generator step", restated in the section's order over the float64 oracle.

TEST INFRASTRUCTURE ONLY: used by the tests; never by the library.

State (section 6 "Generator delayed-code cache"): an integer token ring of C = 4 columns per
stream and a boolean "provided" ring of the same shape, plus the generator offset s, which
is separate from the temporal attention position.  Unwritten slots hold -2, the
ungenerated-cache sentinel.  Per call, with d[k] the delay of stream k and max_delay their
maximum (1):

  1. codes handed in for stream k (the user's codebooks, or forced agent text/codes) are
     placed at column (s + d[k]) mod C and marked provided;
  2. the initial calls insert the native initial tokens: stream k gets its initial ID at
     column s mod C while s <= d[k] (marked provided); at s = 0 nothing else happens: the
     offset advances and the call returns no output;
  3. the temporal input is column (s - 1) mod C, the targets are column s mod C;
  4. the temporal model runs on that input; the text token is selected unless the text
     target is provided, in which case the provided token conditions the depth model;
  5. depth positions q = 0..15 (stream k = q + 1) select a code, replaced by the target
     where the target is provided; the chosen code is the next position's input;
  6. selected text / codes are written only into unprovided target slots; the input
     column's provided flags are cleared;
  7. once the initial delay padding is over (s > max_delay), the aligned output of stream
     k is column (s - max_delay + d[k]) mod C; then s advances.

Readings where the section is silent: "initial calls insert native initial tokens" is
taken for every stream whose delay is at least the call's offset (so the first call fills
the whole first column and the second call the delayed streams' second column); those
slots count as provided, so the depth model is handed the initial audio ID at delayed
positions on the first model step (the depth tables have a row for it).  The first output
is returned at s = max_delay + 1, the first call whose delay-0 output column was selected by
the model.  A provided value of -1 in the caller's array means "nothing provided for this
stream" (the no-input ID is not supplied through the ring).
"""
from __future__ import annotations

from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np

C_RING = 4
SENTINEL = -2


class GeneratorRing:
    """The integer part of the generator: rings, offset and the seven steps, with the model
    behind a callable `model(inputs, text_provided, supplied) -> (text, codes)` where
    `inputs` are the 17 temporal inputs, `text_provided` is the provided text token or
    None, and `supplied` holds per depth position the provided code or -1."""

    def __init__(self, delays: Sequence[int], init_ids: Sequence[int]):
        self.d = [int(x) for x in delays]
        self.S = len(self.d)
        self.max_delay = max(self.d)
        self.init = [int(x) for x in init_ids]
        self.ring = [[SENTINEL] * C_RING for _ in range(self.S)]
        self.prov = [[False] * C_RING for _ in range(self.S)]
        self.s = 0

    def step(self, provided: Optional[Sequence[int]], model: Callable) -> Optional[List[int]]:
        C, S, s = C_RING, self.S, self.s
        # 1. place provided codes at (s + d[k]) mod C
        if provided is not None:
            for k in range(S):
                if int(provided[k]) >= 0:
                    col = (s + self.d[k]) % C
                    self.ring[k][col] = int(provided[k])
                    self.prov[k][col] = True
        # 2. initial tokens while s <= d[k]; the call at s = 0 runs no model
        for k in range(S):
            if s <= self.d[k]:
                self.ring[k][s % C] = self.init[k]
                self.prov[k][s % C] = True
        if s == 0:
            self.s = 1
            return None
        # 3. input column and target column
        inp = [self.ring[k][(s - 1) % C] for k in range(S)]
        tgt = s % C
        # 4-5. temporal model, text selection, depth positions with provided targets
        text_p = self.ring[0][tgt] if self.prov[0][tgt] else None
        supplied = [self.ring[k][tgt] if self.prov[k][tgt] else -1 for k in range(1, S)]
        text, codes = model(inp, text_p, supplied)
        # 6. write selections into unprovided target slots; clear the input's flags
        if not self.prov[0][tgt]:
            self.ring[0][tgt] = int(text)
        for k in range(1, S):
            if not self.prov[k][tgt]:
                self.ring[k][tgt] = int(codes[k - 1])
        for k in range(S):
            self.prov[k][(s - 1) % C] = False
        # 7. aligned output once the initial delay padding is over
        out = None
        if s > self.max_delay:
            out = [self.ring[k][(s - self.max_delay + self.d[k]) % C] for k in range(S)]
        self.s = s + 1
        return out


class Generator:
    """GeneratorRing over the float64 oracle: greedy text and depth codes."""

    def __init__(self, model, shape: dict):
        self.m = model
        self.stream = model.new_stream()
        init = [int(shape["init_text"])] + [int(shape["init_audio"])] * (int(shape["n_streams"]) - 1)
        self.ring = GeneratorRing(shape["delays"][:shape["n_streams"]], init)
        self.last = None   # (hidden, logits, text, depth logits, codes) of the last model step

    def _model(self, inp, text_p, supplied):
        h, _, lg, am = self.stream.forward(np.asarray(inp, np.int32))
        text = am if text_p is None else int(text_p)
        dl, codes = self.m.depformer_step(h, text, np.asarray(supplied, np.int32))
        self.last = (h, lg, int(am), dl, codes)
        return text, [int(c) for c in codes]

    def step(self, provided: Optional[Sequence[int]] = None) -> Tuple[Optional[List[int]], Optional[tuple]]:
        self.last = None
        out = self.ring.step(provided, self._model)
        return out, self.last
