"""GB300 (sm_103a) library for the batched verify step of speculative decoding.

The CUDA library (libspecverify.so, C ABI in include/spec_verify.h) holds the
whole hot path: spec_verify (target distribution, accept chain, residual or
bonus draw, logprobs, alpha) and spec_commit (accepted-state gather).
`binding` is the thin ctypes layer over it; `synth` builds seeded synthetic
inputs; `build` compiles the library with nvcc.

    from speculative_decoding_verify_07_gb300 import binding as sv
    out = sv.spec_verify(logits, q, drafts, sv.make_params(T, K, P, dev), seed)
"""
