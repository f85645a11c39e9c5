"""Plain CPU oracle for the state commit that follows verify.

TEST INFRASTRUCTURE ONLY (see oracle/verify.py for who may import it).

[AReno] inclusionAI/AReno PR #550, "feat(engine): MTP training loss and
speculative decoding for bailing_v3", "What does this PR do?" Phase 2: the
recurrent and conv caches of the linear-attention layers are stacked across
layers and the verify forward writes one state per fed token into a shared
verify-state buffer; after acceptance the accepted position's state is
committed into the cache ("commit in 4 kernels", table "Per-step
optimizations").  The GPU check table ("How was it tested?") requires the
recurrent, conv and KV state after full and partial commits to match
sequential decode, which for a pure gather means byte equality.

Row r commits verify state a_r = accept_len[r] - 1 (the state after the fed
tokens x_0..x_{a-1}, READING) into cache slot cache_slot[r] of every layer:

    cache_rec[l, slot_r]  = verify_rec[l, r, a_r]     for all layers l
    cache_conv[l, slot_r] = verify_conv[l, r, a_r]

accept_len[r] == 0 (an invalid row) skips the row.  accept_len outside
[0, S] or a slot outside [0, slots) flags the row (F_BAD_IDX) and skips it.
"""
from __future__ import annotations

import numpy as np

F_BAD_IDX = 128


def commit(verify_rec: np.ndarray, verify_conv: np.ndarray, accept_len: np.ndarray,
           cache_slot, cache_rec: np.ndarray, cache_conv: np.ndarray):
    """Return (new cache_rec, new cache_conv, flags[B]); inputs are not modified.

    verify_rec  [L, B, S, ...]   verify_conv [L, B, S, ...]
    cache_rec   [L, slots, ...]  cache_conv  [L, slots, ...]
    cache_slot  [B] or None (slot r for row r)
    """
    L, B, S = verify_rec.shape[:3]
    slots = cache_rec.shape[1]
    slot = np.arange(B) if cache_slot is None else np.asarray(cache_slot)
    acc = np.asarray(accept_len).astype(np.int64)
    flags = np.zeros(B, dtype=np.uint32)
    bad = (acc < 0) | (acc > S) | (slot < 0) | (slot >= slots)
    flags[bad] |= F_BAD_IDX
    live = (~bad) & (acc > 0)
    rows = np.nonzero(live)[0]
    src = acc[rows] - 1
    new_rec = cache_rec.copy()
    new_conv = cache_conv.copy()
    # NumPy fancy indexing: for every layer, gather the chosen state of each
    # live row and scatter it to the row's slot.
    new_rec[:, slot[rows]] = verify_rec[:, rows, src]
    new_conv[:, slot[rows]] = verify_conv[:, rows, src]
    return new_rec, new_conv, flags
