"""GPU: spec_verify_commit gives exactly the results of spec_verify followed
by spec_commit on the same inputs -- the verify outputs, the flags (with
SPEC_F_BAD_IDX) and every byte of the caches."""
import numpy as np
import pytest
import torch

from speculative_decoding_verify_07_gb300 import synth
from tests.gpu_harness import to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _random_bits(shape, dtype, g):
    t = torch.empty(shape, dtype=torch.int32 if dtype == torch.float32 else torch.int16, device="cuda")
    t.random_(generator=g)
    return t.view(dtype)


def _states(L, B, S, H, Dk, Dv, W, C, slots, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    vrec = _random_bits((L, B, S, H, Dk, Dv), torch.float32, g) if H else None
    vconv = _random_bits((L, B, S, W, C), torch.int16, g) if W else None
    crec = _random_bits((L, slots, H, Dk, Dv), torch.float32, g) if H else None
    cconv = _random_bits((L, slots, W, C), torch.int16, g) if W else None
    return vrec, vconv, crec, cconv


def _same(a, b):
    if a is None:
        return b is None
    return torch.equal(a.view(torch.int16 if a.element_size() == 2 else torch.int32),
                       b.view(torch.int16 if b.element_size() == 2 else torch.int32))


def _both(inp, L, H, Dk, Dv, W, C, slots, slot_map, seed=5):
    from speculative_decoding_verify_07_gb300 import binding as sv
    logits, q, x, params = to_device(inp)
    B, S = logits.shape[0], logits.shape[1]
    vrec, vconv, crec, cconv = _states(L, B, S, H, Dk, Dv, W, C, slots, seed)
    slot = None if slot_map is None else torch.as_tensor(slot_map, dtype=torch.int32, device="cuda")
    # two launches
    crec1 = None if crec is None else crec.clone()
    cconv1 = None if cconv is None else cconv.clone()
    out1 = sv.spec_verify(logits, q, x, params, inp.seed)
    sv.spec_commit(vrec, vconv, out1.accept_len, slot, crec1, cconv1, flags=out1.flags)
    # one launch
    crec2 = None if crec is None else crec.clone()
    cconv2 = None if cconv is None else cconv.clone()
    out2 = sv.spec_verify_commit(logits, q, x, params, inp.seed, vrec, vconv, slot, crec2, cconv2)
    torch.cuda.synchronize()
    for name in ("tokens", "accept_len", "logprobs", "alpha", "flags"):
        assert _same(getattr(out1, name), getattr(out2, name)), name
    assert _same(crec1, crec2), "recurrent cache"
    assert _same(cconv1, cconv2), "conv cache"
    return out1, crec, crec2


def test_fused_small_with_slot_map_and_bad_slots():
    inp = synth.make_mixed(B=16, k=2, V=20000, seed_offset=3)
    slots = 20
    slot_map = np.random.default_rng(7).permutation(slots)[:16].astype(np.int32)
    slot_map[3] = -1        # bad slots: flagged and skipped
    slot_map[9] = slots + 4
    out, before, after = _both(inp, L=3, H=2, Dk=16, Dv=32, W=4, C=64, slots=slots, slot_map=slot_map)
    fl = out.flags.cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    assert fl[3] & 128 and fl[9] & 128
    # something was copied, and the bad rows' slots were not the target of any copy
    assert not torch.equal(before.view(torch.int32), after.view(torch.int32))


def test_fused_multi_piece_jobs():
    # an 80 KB recurrent blob (two jobs, ten 8 KB pieces) and a 24 KB conv blob
    inp = synth.make_mixed(B=8, k=3, V=30000, seed_offset=4)
    _both(inp, L=2, H=4, Dk=64, Dv=80, W=3, C=4096, slots=8, slot_map=None)


def test_fused_unaligned_conv_blob_takes_the_plain_copy():
    # a 30-byte conv blob: no bulk copies for this call
    inp = synth.make_mixed(B=8, k=2, V=12000, seed_offset=6)
    _both(inp, L=2, H=2, Dk=4, Dv=4, W=3, C=5, slots=10, slot_map=None)


def test_fused_with_top_p_rows():
    # rows that take the grid-wide top-p passes finalize last; their states
    # are committed after them in the same launch
    inp = synth.make_topp(B=8, V=20000, seed_offset=9)
    _both(inp, L=2, H=2, Dk=16, Dv=32, W=4, C=64, slots=8, slot_map=None)


def test_fused_conv_only_and_identity_slots():
    inp = synth.make_mixed(B=6, k=2, V=9000, seed_offset=8)
    _both(inp, L=4, H=0, Dk=0, Dv=0, W=4, C=256, slots=6, slot_map=None)


def test_fused_full_size_commit_workload():
    # the 64-row mixed verify and the 24-layer state commit of the benchmark
    inp = synth.make_mixed()
    sh = synth.CommitShape()
    _both(inp, L=sh.L, H=sh.H, Dk=sh.Dk, Dv=sh.Dv, W=sh.W, C=sh.C, slots=sh.slots, slot_map=None)
