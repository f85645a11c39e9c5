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


def _swap_case(seed=3, L=2, B=6, S=3, slots=14):
    rng = np.random.default_rng(seed)
    vrec = rng.standard_normal((L, B, S - 1, 2, 3, 4)).astype(np.float32)
    vconv = rng.integers(0, 1 << 16, size=(L, B, S - 1, 2, 5), dtype=np.uint16)
    crec = rng.standard_normal((L, slots, 2, 3, 4)).astype(np.float32)
    cconv = rng.integers(0, 1 << 16, size=(L, slots, 2, 5), dtype=np.uint16)
    perm = rng.permutation(slots)
    return vrec, vconv, crec, cconv, perm[:B].astype(np.int32), perm[B:2 * B].astype(np.int32)


def test_commit_swap_matches_explicit_loops():
    vrec, vconv, crec, cconv, sl, sc = _swap_case()
    acc = np.array([3, 1, 2, 0, 3, 2], np.int32)
    nr, nc, nsl, nsc, fl = oc.commit_swap(vrec, vconv, acc, sl, sc, crec, cconv)
    er, ec, esl, esc = crec.copy(), cconv.copy(), sl.copy(), sc.copy()
    for r in range(6):
        if acc[r] == 3:
            esl[r], esc[r] = sc[r], sl[r]
        elif acc[r] > 0:
            for l in range(vrec.shape[0]):
                er[l, sl[r]] = vrec[l, r, acc[r] - 1]
                ec[l, sl[r]] = vconv[l, r, acc[r] - 1]
    assert np.array_equal(nr.view(np.uint32), er.view(np.uint32)) and np.array_equal(nc, ec)
    assert np.array_equal(nsl, esl) and np.array_equal(nsc, esc) and not fl.any()
    # full accepts move no state: the cache is untouched in their slots
    for r in (0, 4):
        assert np.array_equal(nr[:, sl[r]], crec[:, sl[r]]) and np.array_equal(nr[:, sc[r]], crec[:, sc[r]])


def test_commit_swap_commits_what_the_copying_commit_does():
    # Place the last state of each row in its scratch slot and stack the
    # others: after either commit, the row's committed slot holds the same
    # bytes (the state after its accepted tokens).
    vrec, vconv, crec, cconv, sl, sc = _swap_case(seed=9)
    L, B, Sm1 = vrec.shape[:3]
    S = Sm1 + 1
    rng = np.random.default_rng(1)
    last_rec = rng.standard_normal((L, B) + vrec.shape[3:]).astype(np.float32)
    last_conv = rng.integers(0, 1 << 16, size=(L, B) + vconv.shape[3:], dtype=np.uint16)
    crec2, cconv2 = crec.copy(), cconv.copy()
    crec2[:, sc] = last_rec
    cconv2[:, sc] = last_conv
    full_rec = np.concatenate([vrec, last_rec[:, :, None]], axis=2)
    full_conv = np.concatenate([vconv, last_conv[:, :, None]], axis=2)
    acc = rng.integers(1, S + 1, size=B).astype(np.int32)
    sr, scv, nsl, _, _ = oc.commit_swap(vrec, vconv, acc, sl, sc, crec2, cconv2)
    pr, pc, _ = oc.commit(full_rec, full_conv, acc, sl, crec, cconv)
    for r in range(B):
        assert np.array_equal(sr[:, nsl[r]].view(np.uint32), pr[:, sl[r]].view(np.uint32))
        assert np.array_equal(scv[:, nsl[r]], pc[:, sl[r]])


def test_commit_swap_flags_bad_rows():
    vrec, vconv, crec, cconv, sl, sc = _swap_case()
    acc = np.array([4, -1, 1, 2, 3, 1], np.int32)
    sl = sl.copy()
    sc = sc.copy()
    sl[2] = 99
    sc[3] = sl[3]
    sc[5] = -2
    nr, _, nsl, nsc, fl = oc.commit_swap(vrec, vconv, acc, sl, sc, crec, cconv)
    assert list(fl) == [oc.F_BAD_IDX] * 4 + [0, oc.F_BAD_IDX]
    assert nsl[4] == sc[4] and nsc[4] == sl[4]          # the good full accept swapped
    assert np.array_equal(nsl[:4], sl[:4])
