"""Seeded synthetic inputs for the verify and commit workloads.

This module builds inputs only.  It holds none of the verify method's
arithmetic: the draft distributions q it builds stand for a draft model's
output (a softmax of noisy logits), which the method takes as given.  Tests
and the benchmark both draw their inputs from here; neither the library nor
the oracle imports it.

Workloads (data seeded by numpy.random.default_rng(1000 + config index)):

  tiny    B=1,  k=1, V=1024,   fp32 logits ~ N(0, 2^2); draft logits = target
          + N(0, 0.5^2); q = softmax(draft); x ~ q; T=1, no filter; seed 0.
  topp    B=16, k=2, V=157184, bf16 logits ~ N(0, 3^2) with 5 distinct random
          tokens per (row, position) raised by +8; q = softmax(target +
          N(0, 0.7^2)), x ~ q; T=1, top-p 0.95.
  mixed   B=64, k=2, V=151936, bf16 logits as in `topp`; rows r%4==0 greedy,
          r%4 in {1,2} T=0.7 top-k 50 top-p 0.9, r%4==3 T=1; exact ties
          injected in 1% of (row, position): the max logit and the 50th
          largest are each copied onto another random token.
  adversarial  B=256, k=4, V=151936, fp32 logits ~ N(0, 3^2) + spikes; T=1,
          no filter.  Rows 0..127: q puts 0.99 of its mass uniformly on 8
          tokens whose target probability is below 1e-4 (the rest in
          proportion to p), x ~ q, forcing early rejection.  Rows 128..255:
          q = float32(p) exactly, x ~ q (full accept, bonus path).
  commit  L=24, B=64, S=3, H=16, Dk=Dv=128 fp32 recurrent state and W=4,
          C=4096 bf16 conv state per layer; accept_len uniform in {1,2,3};
          cache_slot = identity.

The public benchmark datasets the pages measure on are not available; these
shapes and distributions stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

CONFIG_NAMES = ("tiny", "topp", "mixed", "adversarial", "commit")


@dataclass
class VerifyInputs:
    name: str
    logits: np.ndarray        # [B, k+1, V] float32 (bf16-representable when dtype == "bf16")
    dtype: str                # "f32" or "bf16"
    q: np.ndarray             # [B, k, V] float32
    drafts: np.ndarray        # [B, k] int32
    temperature: np.ndarray   # [B] float32
    top_k: np.ndarray         # [B] int32
    top_p: np.ndarray         # [B] float32
    seed: int

    @property
    def shape(self):
        B, k1, V = self.logits.shape
        return B, k1 - 1, V


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even), kept as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    b = (b + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return b.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The upper 16 bits of bf16-representable float32 values (the bf16 encoding)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def _sample_rows(rng: np.random.Generator, probs: np.ndarray) -> np.ndarray:
    """One categorical draw per row of `probs` [..., V] by inverse CDF."""
    flat = probs.reshape(-1, probs.shape[-1])
    cdf = np.cumsum(flat, axis=1)
    u = rng.random(flat.shape[0]) * cdf[:, -1]
    idx = np.array([np.searchsorted(cdf[i], u[i], side="right") for i in range(flat.shape[0])])
    idx = np.minimum(idx, flat.shape[1] - 1)
    return idx.reshape(probs.shape[:-1]).astype(np.int32)


def _spiked_logits(rng, B, S, V, sigma=3.0, n_spikes=5, spike=8.0):
    logits = rng.normal(0.0, sigma, size=(B, S, V)).astype(np.float32)
    for b in range(B):
        for s in range(S):
            idx = rng.choice(V, size=n_spikes, replace=False)
            logits[b, s, idx] += spike
    return logits


def make_tiny(seed_offset: int = 0) -> VerifyInputs:
    rng = np.random.default_rng(1000 + 0 + seed_offset)
    B, k, V = 1, 1, 1024
    logits = rng.normal(0.0, 2.0, size=(B, k + 1, V)).astype(np.float32)
    draft = logits[:, :k].astype(np.float64) + rng.normal(0.0, 0.5, size=(B, k, V))
    q = _softmax_rows(draft).astype(np.float32)
    drafts = _sample_rows(rng, q.astype(np.float64))
    return VerifyInputs("tiny", logits, "f32", q, drafts,
                        np.ones(B, np.float32), np.zeros(B, np.int32), np.ones(B, np.float32), 0)


def _noisy_q(rng, logits, k, sigma):
    draft = logits[:, :k].astype(np.float64) + rng.normal(0.0, sigma, size=logits[:, :k].shape)
    return _softmax_rows(draft).astype(np.float32)


def make_topp(B=16, k=2, V=157184, seed_offset: int = 0) -> VerifyInputs:
    rng = np.random.default_rng(1000 + 1 + seed_offset)
    logits = round_to_bf16(_spiked_logits(rng, B, k + 1, V))
    q = _noisy_q(rng, logits, k, 0.7)
    drafts = _sample_rows(rng, q.astype(np.float64))
    return VerifyInputs("topp", logits, "bf16", q, drafts,
                        np.ones(B, np.float32), np.zeros(B, np.int32),
                        np.full(B, 0.95, np.float32), 1)


def mixed_params(B):
    T = np.ones(B, np.float32)
    K = np.zeros(B, np.int32)
    P = np.ones(B, np.float32)
    for r in range(B):
        if r % 4 == 0:
            T[r] = 0.0
        elif r % 4 in (1, 2):
            T[r], K[r], P[r] = 0.7, 50, 0.9
    return T, K, P


def make_mixed(B=64, k=2, V=151936, seed_offset: int = 0) -> VerifyInputs:
    rng = np.random.default_rng(1000 + 2 + seed_offset)
    logits = _spiked_logits(rng, B, k + 1, V)
    logits = round_to_bf16(logits)
    # Exact ties in 1% of (row, position): copy the max and the 50th largest
    # logit onto other random tokens.
    n_units = B * (k + 1)
    n_tie = max(1, n_units // 100)
    for u in rng.choice(n_units, size=n_tie, replace=False):
        b, s = divmod(int(u), k + 1)
        row = logits[b, s]
        order = np.argsort(-row, kind="stable")
        for rank in (0, 49):
            src = order[rank]
            dst = int(rng.integers(V))
            while dst == src:
                dst = int(rng.integers(V))
            row[dst] = row[src]
    q = _noisy_q(rng, logits, k, 0.7)
    drafts = _sample_rows(rng, q.astype(np.float64))
    T, K, P = mixed_params(B)
    return VerifyInputs("mixed", logits, "bf16", q, drafts, T, K, P, 2)


def make_adversarial(B=256, k=4, V=151936, seed_offset: int = 0) -> VerifyInputs:
    rng = np.random.default_rng(1000 + 3 + seed_offset)
    logits = _spiked_logits(rng, B, k + 1, V)
    p = _softmax_rows(logits[:, :k].astype(np.float64))        # T = 1, no filter
    q = np.empty((B, k, V), np.float32)
    half = B // 2
    for b in range(B):
        for j in range(k):
            if b < half:
                low = np.nonzero(p[b, j] < 1e-4)[0]
                bad = rng.choice(low, size=8, replace=False)
                qq = 0.01 * p[b, j]
                qq[bad] += 0.99 / 8
                q[b, j] = qq / qq.sum()
            else:
                q[b, j] = p[b, j].astype(np.float32)
    drafts = _sample_rows(rng, q.astype(np.float64))
    return VerifyInputs("adversarial", logits, "f32", q, drafts,
                        np.ones(B, np.float32), np.zeros(B, np.int32), np.ones(B, np.float32), 3)


MAKERS = {"tiny": make_tiny, "topp": make_topp, "mixed": make_mixed,
          "adversarial": make_adversarial}


def make_verify(name: str, **kw) -> VerifyInputs:
    return MAKERS[name](**kw)


@dataclass
class CommitShape:
    L: int = 24
    B: int = 64
    S: int = 3
    H: int = 16
    Dk: int = 128
    Dv: int = 128
    W: int = 4
    C: int = 4096
    slots: int = 64

    @property
    def rec_elems(self):            # fp32 elements per (layer, row, state)
        return self.H * self.Dk * self.Dv

    @property
    def conv_elems(self):           # bf16 elements per (layer, row, state)
        return self.W * self.C

    def bytes_moved(self, live_rows=None):
        rows = self.B if live_rows is None else live_rows
        return 2 * rows * self.L * (self.rec_elems * 4 + self.conv_elems * 2)


def commit_indices(shape: CommitShape, seed_offset: int = 0):
    """accept_len uniform in {1..S} and the identity slot map."""
    rng = np.random.default_rng(1000 + 4 + seed_offset)
    accept_len = rng.integers(1, shape.S + 1, size=shape.B).astype(np.int32)
    cache_slot = np.arange(shape.B, dtype=np.int32)
    return accept_len, cache_slot


def make_commit_small(L=3, B=5, S=3, H=2, Dk=4, Dv=8, W=4, C=24, slots=7, seed=11):
    """A small commit case with host arrays (random bits, permuted slots)."""
    rng = np.random.default_rng(seed)
    vrec = rng.standard_normal((L, B, S, H, Dk, Dv)).astype(np.float32)
    vconv = rng.integers(0, 1 << 16, size=(L, B, S, W, C), dtype=np.uint16)
    crec = rng.standard_normal((L, slots, H, Dk, Dv)).astype(np.float32)
    cconv = rng.integers(0, 1 << 16, size=(L, slots, W, C), dtype=np.uint16)
    acc = rng.integers(0, S + 1, size=B).astype(np.int32)
    slot = rng.permutation(slots)[:B].astype(np.int32)
    return vrec, vconv, acc, slot, crec, cconv
