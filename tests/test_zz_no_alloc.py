"""The allocation-free verify entry point, checked against spec_verify.

Some callers cannot allocate device memory for the verify step's scratch:
plugin or custom-op hosts that hand a kernel only its inputs and outputs,
engines whose allocator has reserved all of HBM, loops that cannot take the
synchronisation of cudaMalloc.  spec_verify_noalloc serves them from a fixed
8 MiB array inside the library.  Two calls in a row must give the results of
spec_verify with a caller-provided workspace, and a batch that needs more
scratch than the array holds must be refused without launching anything.

This file is collected last so that, if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verify_07_gb300 import synth
from tests.gpu_harness import ALPHA_TOL, LP_TOL, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_noalloc_matches_spec_verify_on_two_calls():
    from speculative_decoding_verify_07_gb300 import binding as sv
    inp = synth.make_mixed()                      # 64 rows, k=2, V=151936, bf16
    logits, q, x, params = to_device(inp)
    ref = sv.spec_verify(logits, q, x, params, inp.seed)
    torch.cuda.synchronize()
    for _ in range(2):
        out = sv.spec_verify_noalloc(logits, q, x, params, inp.seed)
        torch.cuda.synchronize()
        assert torch.equal(out.tokens, ref.tokens)
        assert torch.equal(out.accept_len, ref.accept_len)
        assert torch.equal(out.flags, ref.flags)
        assert float((out.logprobs - ref.logprobs).abs().max()) <= LP_TOL
        assert float((out.alpha - ref.alpha).abs().max()) <= ALPHA_TOL


def test_noalloc_refuses_a_batch_beyond_its_scratch():
    from speculative_decoding_verify_07_gb300 import binding as sv
    B, k, V = 4000, 16, 151936
    assert sv.workspace_size(B, k, V) > (8 << 20)
    fake = ctypes.c_void_p(4096)                 # never dereferenced: the size check comes first
    rc = sv.LIB.spec_verify_noalloc(fake, sv.SPEC_BF16, fake, fake, fake, ctypes.c_uint64(0),
                                    ctypes.c_uint32(0), B, k, V, fake, fake, fake, fake, fake, None)
    assert rc == sv.SPEC_E_WORKSPACE


def test_noalloc_refuses_a_null_pointer_before_enqueuing():
    # The argument checks come before the scratch is cleared on the stream:
    # a refused call returns its argument error and leaves the next call's
    # results as they would be without it.
    from speculative_decoding_verify_07_gb300 import binding as sv
    inp = synth.make_mixed(B=8, V=4096)
    logits, q, x, params = to_device(inp)
    ref = sv.spec_verify(logits, q, x, params, inp.seed)
    out = sv.VerifyOutputs(8, 2, "cuda")
    rc = sv.LIB.spec_verify_noalloc(None, sv.SPEC_BF16, ctypes.c_void_p(q.data_ptr()),
                                    ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(params.data_ptr()),
                                    ctypes.c_uint64(inp.seed), ctypes.c_uint32(0), 8, 2, 4096,
                                    ctypes.c_void_p(out.tokens.data_ptr()),
                                    ctypes.c_void_p(out.accept_len.data_ptr()),
                                    ctypes.c_void_p(out.logprobs.data_ptr()),
                                    ctypes.c_void_p(out.alpha.data_ptr()),
                                    ctypes.c_void_p(out.flags.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == sv.SPEC_E_NULL
    got = sv.spec_verify_noalloc(logits, q, x, params, inp.seed)
    torch.cuda.synchronize()
    assert torch.equal(got.tokens, ref.tokens) and torch.equal(got.accept_len, ref.accept_len)
