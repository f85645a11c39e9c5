"""GPU parity of spec_commit against the oracle (byte equality)."""
import numpy as np
import pytest
import torch

from oracle import commit as oc
from speculative_decoding_verify_07_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _run(vrec, vconv, acc, slot, crec, cconv, flags=True):
    from speculative_decoding_verify_07_gb300 import binding as sv
    d = lambda a: None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()
    t_vrec, t_crec = d(vrec), d(crec)
    t_vconv = None if vconv is None else d(vconv.view(np.int16))
    t_cconv = None if cconv is None else d(cconv.view(np.int16))
    t_flags = torch.zeros(len(acc), dtype=torch.int32, device="cuda") if flags else None
    sv.spec_commit(t_vrec, t_vconv, d(acc.astype(np.int32)),
                   None if slot is None else d(slot.astype(np.int32)), t_crec, t_cconv, t_flags)
    torch.cuda.synchronize()
    out_rec = None if t_crec is None else t_crec.cpu().numpy()
    out_conv = None if t_cconv is None else t_cconv.cpu().numpy().view(np.uint16)
    return out_rec, out_conv, (None if t_flags is None else t_flags.cpu().numpy())


@pytest.mark.parametrize("shape", [dict(), dict(H=3, Dk=5, Dv=7, C=9, W=3), dict(L=1, B=1, S=1, slots=1)])
def test_commit_small_matches_oracle(shape):
    vrec, vconv, acc, slot, crec, cconv = synth.make_commit_small(**shape)
    acc = acc.copy()
    acc[0] = 0   # a skipped row
    er, ec, ef = oc.commit(vrec, vconv, acc, slot, crec, cconv)
    gr, gc, gf = _run(vrec, vconv, acc, slot, crec, cconv)
    assert np.array_equal(gr.view(np.uint32), er.view(np.uint32))
    assert np.array_equal(gc, ec)
    assert np.array_equal(gf.astype(np.uint32), ef)


def test_commit_bad_indices_flagged_and_skipped():
    vrec, vconv, acc, slot, crec, cconv = synth.make_commit_small()
    acc = acc.copy()
    slot = slot.copy()
    acc[1] = 9
    slot[2] = 1000
    acc[2] = 1
    acc[3] = -4
    er, ec, ef = oc.commit(vrec, vconv, acc, slot, crec, cconv)
    gr, gc, gf = _run(vrec, vconv, acc, slot, crec, cconv)
    assert np.array_equal(gr.view(np.uint32), er.view(np.uint32))
    assert np.array_equal(gc, ec)
    assert np.array_equal(gf.astype(np.uint32), ef)


def test_commit_multi_chunk_blobs_with_tails():
    """Blobs of 20 KiB (recurrent) and 16 KiB + 64 B (conv): several 16 KiB chunks per blob
    with a short last chunk, plus a skipped row and out-of-range rows."""
    vrec, vconv, acc, slot, crec, cconv = synth.make_commit_small(L=3, B=6, S=3, H=2, Dk=64, Dv=40, W=4,
                                                                  C=2056, slots=8, seed=23)
    acc = acc.copy()
    slot = slot.copy()
    acc[0] = 0
    acc[1] = 3
    acc[2] = 4      # beyond S: flagged and skipped
    slot[3] = -1    # bad slot: flagged and skipped
    acc[3] = 2
    acc[4] = 1
    er, ec, ef = oc.commit(vrec, vconv, acc, slot, crec, cconv)
    gr, gc, gf = _run(vrec, vconv, acc, slot, crec, cconv)
    assert np.array_equal(gr.view(np.uint32), er.view(np.uint32))
    assert np.array_equal(gc, ec)
    assert np.array_equal(gf.astype(np.uint32), ef)


def test_commit_rec_only_conv_only_and_identity_slots():
    vrec, vconv, acc, _, crec, cconv = synth.make_commit_small(slots=5)
    er, ec, _ = oc.commit(vrec, vconv, acc, None, crec, cconv)
    gr, _, _ = _run(vrec, None, acc, None, crec, None, flags=False)
    assert np.array_equal(gr.view(np.uint32), er.view(np.uint32))
    _, gc, _ = _run(None, vconv, acc, None, None, cconv)
    assert np.array_equal(gc, ec)


def test_commit_full_size_sampled():
    """The 24-layer, 64-row workload at full size; sampled (layer, row) blobs checked."""
    from speculative_decoding_verify_07_gb300 import binding as sv
    sh = synth.CommitShape()
    acc, slot = synth.commit_indices(sh)
    g = torch.Generator(device="cuda")
    g.manual_seed(1004)
    vrec = torch.empty((sh.L, sh.B, sh.S, sh.H, sh.Dk, sh.Dv), dtype=torch.float32, device="cuda")
    vrec.view(torch.int32).random_(generator=g)
    vconv = torch.randint(-32768, 32767, (sh.L, sh.B, sh.S, sh.W, sh.C), dtype=torch.int16,
                          device="cuda", generator=g)
    crec = torch.zeros((sh.L, sh.slots, sh.H, sh.Dk, sh.Dv), dtype=torch.float32, device="cuda")
    cconv = torch.zeros((sh.L, sh.slots, sh.W, sh.C), dtype=torch.int16, device="cuda")
    acc_t = torch.from_numpy(acc).cuda()
    slot_t = torch.from_numpy(slot).cuda()
    sv.spec_commit(vrec, vconv, acc_t, slot_t, crec, cconv)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    for l, r in [(0, 0), (sh.L - 1, sh.B - 1)] + [tuple(x) for x in rng.integers(0, [sh.L, sh.B], (20, 2))]:
        s = int(acc[r]) - 1
        src = vrec[l, r, s].cpu().numpy().view(np.uint32)
        dst = crec[l, slot[r]].cpu().numpy().view(np.uint32)
        # oracle gather on the sampled blob
        exp = oc.commit(src[None, None, None], vconv[l, r, s].cpu().numpy()[None, None, None],
                        np.array([1]), None, np.zeros_like(src)[None, None],
                        np.zeros_like(vconv[l, r, s].cpu().numpy())[None, None])
        assert np.array_equal(dst, exp[0][0, 0])
        assert np.array_equal(cconv[l, slot[r]].cpu().numpy(), exp[1][0, 0])


def _swap_inputs(L=3, B=8, S=3, H=2, Dk=64, Dv=40, W=4, C=2056, slots=20, seed=31):
    rng = np.random.default_rng(seed)
    vrec = rng.standard_normal((L, B, S - 1, H, Dk, Dv)).astype(np.float32)
    vconv = rng.integers(0, 1 << 16, size=(L, B, S - 1, W, C), dtype=np.uint16)
    crec = rng.standard_normal((L, slots, H, Dk, Dv)).astype(np.float32)
    cconv = rng.integers(0, 1 << 16, size=(L, slots, W, C), dtype=np.uint16)
    perm = rng.permutation(slots)
    return vrec, vconv, crec, cconv, perm[:B].astype(np.int32), perm[B:2 * B].astype(np.int32)


def test_commit_swap_matches_oracle():
    from speculative_decoding_verify_07_gb300 import binding as sv
    vrec, vconv, crec, cconv, sl, sc = _swap_inputs()
    acc = np.array([3, 1, 2, 0, 3, 2, 4, 1], np.int32)     # full, partial, skip, bad (4 > S)
    sc = sc.copy()
    sc[7] = sl[7]                                           # equal slots: bad
    er, ec, esl, esc, ef = oc.commit_swap(vrec, vconv, acc, sl, sc, crec, cconv)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    t_crec, t_cconv = d(crec), d(cconv.view(np.int16))
    t_sl, t_sc = d(sl), d(sc)
    t_flags = torch.zeros(8, dtype=torch.int32, device="cuda")
    sv.spec_commit_swap(d(vrec), d(vconv.view(np.int16)), d(acc), t_sl, t_sc, t_crec, t_cconv, t_flags)
    torch.cuda.synchronize()
    assert np.array_equal(t_crec.cpu().numpy().view(np.uint32), er.view(np.uint32))
    assert np.array_equal(t_cconv.cpu().numpy().view(np.uint16), ec)
    assert np.array_equal(t_sl.cpu().numpy(), esl) and np.array_equal(t_sc.cpu().numpy(), esc)
    assert np.array_equal(t_flags.cpu().numpy().astype(np.uint32), ef)


def test_commit_swap_full_size_moves_only_partial_rows():
    """The 24-layer, 64-row workload with a scratch slot per row: full accepts
    trade slots, partial accepts gather; sampled blobs checked."""
    from speculative_decoding_verify_07_gb300 import binding as sv
    sh = synth.CommitShape(slots=128)
    acc, _ = synth.commit_indices(sh)
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    vrec = torch.empty((sh.L, sh.B, sh.S - 1, sh.H, sh.Dk, sh.Dv), dtype=torch.float32, device="cuda")
    vrec.view(torch.int32).random_(generator=g)
    vconv = torch.randint(-32768, 32767, (sh.L, sh.B, sh.S - 1, sh.W, sh.C), dtype=torch.int16,
                          device="cuda", generator=g)
    crec = torch.empty((sh.L, sh.slots, sh.H, sh.Dk, sh.Dv), dtype=torch.float32, device="cuda")
    crec.view(torch.int32).random_(generator=g)
    cconv = torch.randint(-32768, 32767, (sh.L, sh.slots, sh.W, sh.C), dtype=torch.int16, device="cuda",
                          generator=g)
    sl0 = np.arange(sh.B, dtype=np.int32)
    sc0 = np.arange(sh.B, 2 * sh.B, dtype=np.int32)
    t_sl, t_sc = torch.from_numpy(sl0).cuda(), torch.from_numpy(sc0).cuda()
    acc_t = torch.from_numpy(acc).cuda()
    before = crec.clone(), cconv.clone()
    sv.spec_commit_swap(vrec, vconv, acc_t, t_sl, t_sc, crec, cconv)
    torch.cuda.synchronize()
    nsl, nsc = t_sl.cpu().numpy(), t_sc.cpu().numpy()
    full = acc == sh.S
    assert np.array_equal(nsl[full], sc0[full]) and np.array_equal(nsc[full], sl0[full])
    assert np.array_equal(nsl[~full], sl0[~full])
    rng = np.random.default_rng(1)
    for l, r in [(0, 0), (sh.L - 1, sh.B - 1)] + [tuple(x) for x in rng.integers(0, [sh.L, sh.B], (20, 2))]:
        if full[r]:
            # nothing moved: the scratch slot (now committed) keeps its bytes
            assert torch.equal(crec[l, nsl[r]].view(torch.int32), before[0][l, nsl[r]].view(torch.int32))
        else:
            assert torch.equal(crec[l, nsl[r]].view(torch.int32), vrec[l, r, acc[r] - 1].view(torch.int32))
            assert torch.equal(cconv[l, nsl[r]], vconv[l, r, acc[r] - 1])
