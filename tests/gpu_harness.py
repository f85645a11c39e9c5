"""Helpers for the GPU parity tests: run the library through its C ABI on
synthetic inputs and compare with the oracle row by row.

Comparison rules (tolerances from the verify method's spec bar):
* tokens and accept_len must match exactly, except in rows where the oracle
  flags an accept or draw decision within its 1e-6 margin;
* the input-validation flags (NaN, bad token, bad parameter) must match
  exactly; margin flags are diagnostics and are not compared;
* logprobs of emitted tokens and alpha must agree within 1e-5 absolute;
* positions after the drawn token hold token -1 and logprob 0.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import verify as ov

HARD = ov.F_NAN | ov.F_BAD_TOKEN | ov.F_BAD_PARAM
EXEMPT = ov.F_MARGIN_ACCEPT | ov.F_MARGIN_DRAW
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


def run_gpu(inp, device="cuda", seed=None):
    from speculative_decoding_verify_07_gb300 import binding as sv
    logits, q, x, params = to_device(inp, device)
    out = sv.spec_verify(logits, q, x, params, inp.seed if seed is None else seed)
    torch.cuda.synchronize()
    return {
        "tokens": out.tokens.cpu().numpy(),
        "accept_len": out.accept_len.cpu().numpy(),
        "logprobs": out.logprobs.cpu().numpy(),
        "alpha": out.alpha.cpu().numpy(),
        "flags": out.flags.cpu().numpy().astype(np.int64) & 0xFFFFFFFF,
    }


def run_oracle(inp, rows=None, seed=None):
    return ov.verify(inp.logits, inp.q, inp.drafts, inp.temperature, inp.top_k, inp.top_p,
                     inp.seed if seed is None else seed, rows=rows)


def compare(gpu, orc, context=""):
    """Compare GPU outputs (all rows) with oracle outputs (rows in orc['rows']).

    Returns a summary dict; raises AssertionError listing the first problems.
    """
    problems = []
    exempt_rows = 0
    for i, r in enumerate(orc["rows"]):
        of = int(orc["flags"][i])
        gf = int(gpu["flags"][r])
        if (of & HARD) != (gf & HARD):
            problems.append(f"row {r}: flags oracle {of:#x} gpu {gf:#x}")
            continue
        if of & EXEMPT:
            exempt_rows += 1
            a = int(gpu["accept_len"][r])
            k1 = gpu["tokens"].shape[1]
            if not (1 <= a <= k1):
                problems.append(f"row {r}: exempt row has accept_len {a}")
            continue
        oa, ga = int(orc["accept_len"][i]), int(gpu["accept_len"][r])
        if oa != ga or not np.array_equal(orc["tokens"][i], gpu["tokens"][r]):
            problems.append(f"row {r}: accept_len {oa}/{ga} tokens oracle {orc['tokens'][i].tolist()} "
                            f"gpu {gpu['tokens'][r].tolist()} flags {of:#x}/{gf:#x}")
            continue
        if (of & ov.F_RESIDUAL_EMPTY) != (gf & ov.F_RESIDUAL_EMPTY):
            problems.append(f"row {r}: residual-empty flag oracle {of:#x} gpu {gf:#x}")
        lp_o = orc["logprobs"][i]
        lp_g = gpu["logprobs"][r].astype(np.float64)
        if not np.all(np.abs(lp_o - lp_g) <= LP_TOL):
            problems.append(f"row {r}: logprobs oracle {lp_o.tolist()} gpu {lp_g.tolist()}")
        if gpu["alpha"].shape[1] > 0:
            al_o = orc["alpha"][i]
            al_g = gpu["alpha"][r].astype(np.float64)
            if not np.all(np.abs(al_o - al_g) <= ALPHA_TOL):
                problems.append(f"row {r}: alpha oracle {al_o.tolist()} gpu {al_g.tolist()}")
    summary = {"rows": len(orc["rows"]), "exempt": exempt_rows, "problems": len(problems)}
    assert not problems, f"{context}: {len(problems)} mismatches, e.g.\n" + "\n".join(problems[:12])
    return summary
