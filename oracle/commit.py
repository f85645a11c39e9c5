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


def commit_swap(verify_rec: np.ndarray, verify_conv: np.ndarray, accept_len: np.ndarray,
                slot_of_row: np.ndarray, scratch_slot: np.ndarray, cache_rec: np.ndarray,
                cache_conv: np.ndarray):
    """Zero-copy commit with a scratch slot per row.

    [InfiniLM] InfiniTensor/InfiniLM PR #588, "feat: add mtp draft models for
    speculative decoding", section 2 item 5: the verify forward reads the
    row's committed state and writes into a scratch state slot; when every
    draft is accepted the slot numbers are swapped in O(1); after a partial
    accept the state at the accepted position is brought into the committed
    slot (there by replay; here the per-position states are stacked, so it
    is a gather).  READING: of the S = k + 1 states of a row, the first S - 1
    live in the stacked verify buffer and the last one (after every fed
    token) in cache slot scratch_slot[r], where the verify forward wrote it.

    verify_rec  [L, B, S-1, ...]   verify_conv [L, B, S-1, ...]
    cache_rec   [L, slots, ...]    cache_conv  [L, slots, ...]
    slot_of_row [B], scratch_slot [B]: each row's committed and scratch slot.

    Row r with accept_len a:
      a == S      : slot_of_row[r] and scratch_slot[r] trade places (no copy);
      1 <= a < S  : cache[l, slot_of_row[r]] = verify[l, r, a - 1] for all l;
      a == 0      : nothing (an invalid row);
    a outside [0, S], a slot outside [0, slots), or slot_of_row[r] ==
    scratch_slot[r] flags the row (F_BAD_IDX) and leaves it alone.
    Returns (cache_rec, cache_conv, slot_of_row, scratch_slot, flags), new
    arrays; the inputs are not modified.
    """
    L, B, Sm1 = verify_rec.shape[:3]
    S = Sm1 + 1
    slots = cache_rec.shape[1]
    acc = np.asarray(accept_len).astype(np.int64)
    sl = np.asarray(slot_of_row).astype(np.int64).copy()
    sc = np.asarray(scratch_slot).astype(np.int64).copy()
    flags = np.zeros(B, dtype=np.uint32)
    new_rec = cache_rec.copy()
    new_conv = cache_conv.copy()
    for r in range(B):
        a = int(acc[r])
        bad = (a < 0 or a > S or not (0 <= sl[r] < slots) or not (0 <= sc[r] < slots)
               or sl[r] == sc[r])
        if bad:
            flags[r] |= F_BAD_IDX
            continue
        if a == 0:
            continue
        if a == S:
            sl[r], sc[r] = sc[r], sl[r]
        else:
            new_rec[:, sl[r]] = verify_rec[:, r, a - 1]
            new_conv[:, sl[r]] = verify_conv[:, r, a - 1]
    return new_rec, new_conv, sl.astype(np.int32), sc.astype(np.int32), flags
