"""Helpers for the GPU parity tests: run the library through its C ABI on
synthetic inputs and compare with the oracle row by row.

Comparison rules (tolerances from the verify method's spec bar):
* the input-validation flags (NaN, bad token, bad parameter) must match
  exactly; an invalid row must come back as tokens -1, accept_len 0,
  logprobs 0 and alpha 0;
* tokens and accept_len must match exactly and logprobs within 1e-5.  A
  decision the oracle flags within its 1e-6 margin (an accept test, a top-p
  boundary, a draw) may go either way, and so may everything after it in
  the row: a row that differs is accepted only when its first difference
  comes at or after such a decision.  Those rows count as exempt and every
  test caps them (flagged rows that agree are ordinary matches);
* alpha_j depends on no decision, only on p_j: it must agree within 1e-5 at
  every position whose top-p boundary is certain;
* the device's own margin flags must agree with the oracle's on all but a
  capped number of rows (both compute the same quantities, in float32 and
  float64);
* positions after the drawn token hold token -1 and logprob 0.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import verify as ov

HARD = ov.F_NAN | ov.F_BAD_TOKEN | ov.F_BAD_PARAM
MARGINS = ov.F_MARGIN_ACCEPT | ov.F_MARGIN_DRAW | ov.F_MARGIN_TOPP
LP_TOL = 1e-5
ALPHA_TOL = 1e-5


def to_device(inp, device="cuda"):
    """Tensors for spec_verify from a synth.VerifyInputs-like object."""
    from speculative_decoding_verify_07_gb300 import binding as sv
    dt = torch.bfloat16 if inp.dtype == "bf16" else torch.float32
    logits = torch.from_numpy(np.ascontiguousarray(inp.logits, dtype=np.float32)).to(dt).to(device)
    q = torch.from_numpy(np.ascontiguousarray(inp.q, dtype=np.float32)).to(device)
    x = torch.from_numpy(np.ascontiguousarray(inp.drafts, dtype=np.int32)).to(device)
    params = sv.make_params(inp.temperature, inp.top_k, inp.top_p, device)
    return logits, q, x, params


def host_outputs(out):
    return {
        "tokens": out.tokens.cpu().numpy(),
        "accept_len": out.accept_len.cpu().numpy(),
        "logprobs": out.logprobs.cpu().numpy(),
        "alpha": out.alpha.cpu().numpy(),
        "flags": out.flags.cpu().numpy().astype(np.int64) & 0xFFFFFFFF,
    }


def run_gpu(inp, device="cuda", seed=None, row_base=0):
    from speculative_decoding_verify_07_gb300 import binding as sv
    logits, q, x, params = to_device(inp, device)
    out = sv.spec_verify(logits, q, x, params, inp.seed if seed is None else seed, row_base=row_base)
    torch.cuda.synchronize()
    return host_outputs(out)


def run_oracle(inp, rows=None, seed=None, row_base=0):
    return ov.verify(inp.logits, inp.q, inp.drafts, inp.temperature, inp.top_k, inp.top_p,
                     inp.seed if seed is None else seed, rows=rows, row_base=row_base)


def default_exempt_cap(n_rows: int) -> int:
    return max(2, math.ceil(0.01 * n_rows))


def _first_difference(orc, i, gpu, r, k1):
    """First position where the GPU row differs from the oracle row (token,
    or logprob beyond LP_TOL); k1 when they agree everywhere."""
    ot, gt = orc["tokens"][i], gpu["tokens"][r]
    lo, lg = orc["logprobs"][i], gpu["logprobs"][r].astype(np.float64)
    for j in range(k1):
        if ot[j] != gt[j] or abs(lo[j] - lg[j]) > LP_TOL:
            return j
    return k1


def compare(gpu, orc, context="", max_exempt=None, max_margin_disagree=None):
    """Compare GPU outputs (all rows) with oracle outputs (rows in orc['rows']).

    A row that differs is accepted only when the oracle flags a decision at
    or before the first differing position (an accept test, a top-p
    boundary, or the draw at the chain's end); such rows are counted as
    exempt and capped (default: 1% of the rows, at least 2).  Flagged rows
    that agree are ordinary matches.  Returns a summary dict (rows, exempt,
    flagged, margin_disagree); raises AssertionError listing the first
    problems.
    """
    problems = []
    exempt_rows = 0
    flagged_rows = 0
    margin_disagree = 0
    k1 = gpu["tokens"].shape[1]
    k = k1 - 1
    for i, r in enumerate(orc["rows"]):
        of = int(orc["flags"][i])
        gf = int(gpu["flags"][r])
        g_tok, g_lp = gpu["tokens"][r], gpu["logprobs"][r].astype(np.float64)
        g_acc = int(gpu["accept_len"][r])
        g_al = gpu["alpha"][r].astype(np.float64) if k > 0 else np.zeros(0)
        if (of & HARD) != (gf & HARD):
            problems.append(f"row {r}: flags oracle {of:#x} gpu {gf:#x}")
            continue
        if of & ov.F_NAN:
            if g_acc != 0 or np.any(g_tok != -1) or np.any(g_lp != 0) or np.any(g_al != 0):
                problems.append(f"row {r}: invalid row not cleared: {g_acc} {g_tok.tolist()}")
            continue
        if (of & MARGINS) != (gf & MARGINS):
            margin_disagree += 1
        a = int(orc["a"][i])
        tm = orc["topp_margin"][i]
        ma = orc["margin_accept"][i]
        flagged = [j for j in range(min(a, k - 1) + 1) if j < k and (ma[j] or tm[j])]
        if bool(orc["draw_margin"][i]) or tm[a]:
            flagged.append(a)
        if flagged:
            flagged_rows += 1
        # alpha_j depends only on p_j: it must agree wherever the top-p
        # boundary at j is certain
        if k > 0:
            sure = ~tm[:k]
            al_o = orc["alpha"][i]
            if not np.all(np.abs(al_o[sure] - g_al[sure]) <= ALPHA_TOL):
                problems.append(f"row {r}: alpha oracle {al_o.tolist()} gpu {g_al.tolist()}")
        f = _first_difference(orc, i, gpu, r, k1)
        same = f == k1 and int(orc["accept_len"][i]) == g_acc
        if same:
            if (of & ov.F_RESIDUAL_EMPTY) != (gf & ov.F_RESIDUAL_EMPTY):
                problems.append(f"row {r}: residual-empty flag oracle {of:#x} gpu {gf:#x}")
            continue
        if flagged and min(flagged) <= f:
            exempt_rows += 1
            continue
        problems.append(f"row {r}: accept_len oracle {int(orc['accept_len'][i])} gpu {g_acc}, tokens oracle "
                        f"{orc['tokens'][i].tolist()} gpu {g_tok.tolist()}, logprobs oracle "
                        f"{orc['logprobs'][i].tolist()} gpu {g_lp.tolist()} (first difference at {f}, "
                        f"flagged decisions {flagged}) flags {of:#x}/{gf:#x}")
    n = len(orc["rows"])
    cap = default_exempt_cap(n) if max_exempt is None else max_exempt
    mcap = max(1, math.ceil(0.01 * n)) if max_margin_disagree is None else max_margin_disagree
    summary = {"rows": n, "exempt": exempt_rows, "flagged": flagged_rows, "problems": len(problems),
               "margin_disagree": margin_disagree}
    assert not problems, f"{context}: {len(problems)} mismatches, e.g.\n" + "\n".join(problems[:12])
    assert exempt_rows <= cap, f"{context}: {exempt_rows} differing flagged rows of {n} (cap {cap})"
    assert margin_disagree <= mcap, f"{context}: margin flags disagree on {margin_disagree} rows of {n}"
    return summary
