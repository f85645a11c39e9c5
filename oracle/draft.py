"""Plain CPU oracle for the draft-side sampler (one draft step).

TEST INFRASTRUCTURE ONLY: this module defines what a draft step must return
so that tests can check the CUDA library against it.  Only tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the library and works in float64 throughout.

Pages:

[AReno] inclusionAI/AReno PR #550, "feat(engine): MTP training loss and
    speculative decoding for bailing_v3", "What does this PR do?", Phase 2:
    the MTP layer drafts tokens EAGLE-style, one position at a time, with the
    sampler settings of the target, and the verify needs each draft token
    together with the distribution q it was drawn from.
[AReaL] areal-project/AReaL PR #1659: EAGLE top-k draft tokens are passed
    through to the verify.

READING (the pages fix no draft-side sampler, only that it exists): q_j is
the sampler-equivalent distribution of the draft logits, built exactly as the
verify builds its target p (temperature, top-k, top-p, each renormalised,
with the same total order and the same parameter and invalid-input rules);
x_j ~ q_j is drawn by the verify's two-level exponential race with its own
Philox streams, 3 for the entries and 4 for the blocks, at counter position
j, so that a draft step never reuses a random number of the verify; the
reported logprob is the verify's logprob of an emitted token under q_j.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import philox
from .verify import (F_BAD_PARAM, F_MARGIN_DRAW, F_MARGIN_TOPP, F_NAN, exponential_race, params_valid,
                     target_distribution, token_logprob)

DRAFT_STREAMS = (philox.STREAM_DRAFT_RACE, philox.STREAM_DRAFT_BLOCK)


@dataclass
class DraftRow:
    q: np.ndarray        # float64 [V]; zero outside the kept set, all zero for an invalid row
    x: int               # the drawn token (-1 for an invalid row)
    logprob: float
    flags: int
    draw_margin: bool = False
    topp_margin: bool = False


def draft_row(l: np.ndarray, T: float, K: int, P: float, seed: int, row: int, pos: int) -> DraftRow:
    """One draft step for one row: q = the sampler-equivalent distribution of
    the draft logits l, x ~ q by the exponential race on the draft streams."""
    V = l.shape[0]
    # invalid input, as the verify reads it: a NaN or +inf logit, or no finite one
    if np.any(np.isnan(l)) or np.any(l == np.inf) or np.max(l) == -np.inf:
        return DraftRow(np.zeros(V), -1, 0.0, F_NAN)
    flags = 0
    if not params_valid(T, P):
        flags |= F_BAD_PARAM
        T = 0.0
    if not (0 < K < V):
        K = 0
    if P >= 1.0 or not (P > 0.0):
        P = 1.0
    t = target_distribution(l, T, K, P)
    if t.topp_margin:
        flags |= F_MARGIN_TOPP
    x, margin = exponential_race(t.p, seed, row, pos, t.p, streams=DRAFT_STREAMS)
    if margin:
        flags |= F_MARGIN_DRAW
    return DraftRow(t.p.copy(), int(x), token_logprob(l, t, int(x), T), flags, bool(margin),
                    bool(t.topp_margin))


def draft_sample(logits: np.ndarray, temperature: np.ndarray, top_k: np.ndarray, top_p: np.ndarray,
                 seed: int, pos: int, rows=None, row_base: int = 0) -> dict:
    """A draft step over `rows` (default all) of logits [B, V]; row r draws
    as stream row row_base + r (mod 2^32), as in the verify."""
    B = logits.shape[0]
    rows = list(range(B)) if rows is None else list(rows)
    out = {"q": [], "tokens": [], "logprobs": [], "flags": [], "draw_margin": [], "topp_margin": [],
           "rows": np.asarray(rows, dtype=np.int64)}
    for r in rows:
        res = draft_row(np.asarray(logits[r], dtype=np.float64), float(temperature[r]), int(top_k[r]),
                        float(top_p[r]), seed, (int(row_base) + int(r)) % (1 << 32), int(pos))
        out["q"].append(res.q)
        out["tokens"].append(res.x)
        out["logprobs"].append(res.logprob)
        out["flags"].append(res.flags)
        out["draw_margin"].append(res.draw_margin)
        out["topp_margin"].append(res.topp_margin)
    for key in ("q", "tokens", "logprobs", "flags", "draw_margin", "topp_margin"):
        out[key] = np.asarray(out[key])
    return out
