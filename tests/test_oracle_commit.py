"""Pin for the commit oracle: explicit per-element loops over layers and rows."""
import numpy as np

from oracle import commit as oc
from speculative_decoding_verify_07_gb300 import synth


def test_commit_matches_explicit_loops():
    vrec, vconv, acc, slot, crec, cconv = synth.make_commit_small()
    acc = acc.copy()
    acc[1] = 0          # skipped row
    new_rec, new_conv, flags = oc.commit(vrec, vconv, acc, slot, crec, cconv)
    L, B, S = vrec.shape[:3]
    exp_rec, exp_conv = crec.copy(), cconv.copy()
    for l in range(L):
        for r in range(B):
            if acc[r] == 0:
                continue
            exp_rec[l, slot[r]] = vrec[l, r, acc[r] - 1]
            exp_conv[l, slot[r]] = vconv[l, r, acc[r] - 1]
    assert np.array_equal(new_rec.view(np.uint32), exp_rec.view(np.uint32))
    assert np.array_equal(new_conv, exp_conv)
    assert not flags.any()
    # untouched slots keep their contents
    untouched = sorted(set(range(crec.shape[1])) - set(slot[acc > 0]))
    assert np.array_equal(new_rec[:, untouched], crec[:, untouched])


def test_commit_flags_bad_indices_and_skips():
    vrec, vconv, acc, slot, crec, cconv = synth.make_commit_small()
    acc = acc.copy()
    slot = slot.copy()
    acc[0] = 4          # > S
    acc[2] = -1
    slot[3] = 99        # out of range
    acc[3] = 1
    new_rec, new_conv, flags = oc.commit(vrec, vconv, acc, slot, crec, cconv)
    assert flags[0] == oc.F_BAD_IDX and flags[2] == oc.F_BAD_IDX and flags[3] == oc.F_BAD_IDX
    for r in (0, 2):
        if 0 <= slot[r] < crec.shape[1]:
            assert np.array_equal(new_rec[:, slot[r]], crec[:, slot[r]])


def test_commit_identity_slots():
    vrec, vconv, acc, _, crec, cconv = synth.make_commit_small(slots=5)
    acc = np.maximum(acc, 1)
    new_rec, _, _ = oc.commit(vrec, vconv, acc, None, crec, cconv)
    for r in range(5):
        assert np.array_equal(new_rec[:, r], vrec[:, r, acc[r] - 1])
