"""The oracle over many rows of a large synthetic workload, in a pool of
worker processes (spawned, so that no worker inherits a CUDA context).

Each worker rebuilds the workload from its seed with `synth` and runs the
oracle on its share of the rows; the results are gathered in row order.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

_INP = None


def _init(name, kwargs):
    global _INP
    from speculative_decoding_verify_07_gb300 import synth
    _INP = synth.make_verify(name, **kwargs)


def _rows(args):
    rows, seed, row_base = args
    from oracle import verify as ov
    inp = _INP
    return ov.verify(inp.logits, inp.q, inp.drafts, inp.temperature, inp.top_k, inp.top_p,
                     inp.seed if seed is None else seed, rows=rows, row_base=row_base)


def oracle_rows(name, rows, kwargs=None, seed=None, row_base=0, workers=None):
    """Oracle outputs for `rows` of workload `name` (synth.make_verify(name, **kwargs))."""
    kwargs = kwargs or {}
    rows = list(rows)
    if workers is None:
        workers = max(1, min(len(os.sched_getaffinity(0)), 8, len(rows)))
    chunks = [rows[i::workers] for i in range(workers)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers, initializer=_init, initargs=(name, kwargs)) as pool:
        parts = pool.map(_rows, [(c, seed, row_base) for c in chunks if c])
    # interleave back into row order
    out = {}
    keys = [k for k in parts[0] if k != "rows"]
    pos = {}
    for p in parts:
        for i, r in enumerate(p["rows"]):
            pos[int(r)] = (p, i)
    for key in keys:
        out[key] = np.stack([pos[r][0][key][pos[r][1]] for r in rows])
    out["rows"] = np.asarray(rows, dtype=np.int64)
    return out
