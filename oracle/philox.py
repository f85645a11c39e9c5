"""Philox4x32-10 counter-based generator, host side.

TEST INFRASTRUCTURE ONLY: this package is the slow CPU oracle.  Only tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it; the library's product path never does.

Written from the definition in J. K. Salmon, M. A. Moraes, R. O. Dror,
D. E. Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11, section 3
(the Philox S-box and its key schedule):

* the state is four 32-bit words (X0, X1, X2, X3) and the key two words
  (K0, K1);
* one round multiplies X0 and X2 by the two Philox-4x32 multipliers, keeps the
  high and low halves of each 64-bit product, and permutes
  (X0, X1, X2, X3) -> (hi(M1*X2) ^ X1 ^ K0, lo(M1*X2), hi(M0*X0) ^ X3 ^ K1,
  lo(M0*X0));
* after each round the key is bumped by the Weyl constants (the golden ratio
  and sqrt(3)-1 in 32-bit fixed point);
* Philox4x32-10 is ten rounds.

The pages name no generator; the speculative verify method only asks for
draws "keyed by (seed, row, position)".  The counter layout and the 23-bit
uniform mapping below are this project's reading, stated in one place so the
CUDA path can implement the same stream independently.
"""
from __future__ import annotations

import numpy as np

PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = np.uint64(0xFFFFFFFF)

# Counter word 3 selects the use of a draw.
STREAM_ACCEPT = 0  # u_j for the accept test of draft j:   ctr = (0, j, row, 0), word 0
STREAM_RACE = 1    # U_v for the race inside a block:      ctr = (v >> 2, pos, row, 1), word v & 3
STREAM_BLOCK = 2   # U_b for the race among blocks:        ctr = (b >> 2, pos, row, 2), word b & 3
STREAM_DRAFT_RACE = 3    # the draft sampler's entry race:    ctr = (v >> 2, pos, row, 3), word v & 3
STREAM_DRAFT_BLOCK = 4   # the draft sampler's block race:    ctr = (b >> 2, pos, row, 4), word b & 3


def seed_key(seed: int) -> tuple[int, int]:
    """Split a 64-bit seed into the two key words (low word first)."""
    seed &= (1 << 64) - 1
    return seed & 0xFFFFFFFF, seed >> 32


def philox4x32_10(ctr: np.ndarray, key: tuple[int, int]) -> np.ndarray:
    """Apply Philox4x32-10 to an array of counters.

    ctr: integer array of shape [..., 4] (each entry < 2**32).
    key: (K0, K1).
    Returns a uint32 array of the same shape.
    """
    c = np.asarray(ctr, dtype=np.uint64)
    x0, x1, x2, x3 = (c[..., i].copy() for i in range(4))
    k0 = np.uint64(key[0] & 0xFFFFFFFF)
    k1 = np.uint64(key[1] & 0xFFFFFFFF)
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    s32 = np.uint64(32)
    for _ in range(10):
        p0 = m0 * x0            # < 2**64, exact in uint64
        p1 = m1 * x2
        hi0, lo0 = p0 >> s32, p0 & _MASK32
        hi1, lo1 = p1 >> s32, p1 & _MASK32
        x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
        k0 = (k0 + np.uint64(PHILOX_W0)) & _MASK32
        k1 = (k1 + np.uint64(PHILOX_W1)) & _MASK32
    return np.stack([x0, x1, x2, x3], axis=-1).astype(np.uint32)


def uniform_from_word(w: np.ndarray) -> np.ndarray:
    """Map 32-bit words to uniforms in (0, 1): ((w >> 9) + 1/2) * 2**-23.

    The 23 kept bits make every value exactly representable in float32 as well
    as float64, so both sides of a comparison see the same number.
    """
    w = np.asarray(w, dtype=np.uint64)
    return ((w >> np.uint64(9)).astype(np.float64) + 0.5) * 2.0 ** -23


def one_minus_uniform_from_word(w: np.ndarray) -> np.ndarray:
    """1 - U for the same words, computed exactly (no cancellation)."""
    w = np.asarray(w, dtype=np.uint64)
    return ((np.float64(2 ** 23) - (w >> np.uint64(9)).astype(np.float64)) - 0.5) * 2.0 ** -23


def accept_uniform(seed: int, row: int, j: int) -> float:
    """u_j: the accept-test uniform of draft position j in row `row`."""
    w = philox4x32_10(np.array([0, j, row, STREAM_ACCEPT]), seed_key(seed))[0]
    return float(uniform_from_word(w))


def race_words(seed: int, row: int, pos: int, v: np.ndarray, stream: int = STREAM_RACE) -> np.ndarray:
    """The race words of indices `v` (vocabulary entries, or blocks with
    stream=STREAM_BLOCK) at verify position `pos`."""
    v = np.asarray(v, dtype=np.int64)
    blocks = v >> 2
    ctr = np.stack([blocks, np.full_like(blocks, pos), np.full_like(blocks, row),
                    np.full_like(blocks, stream)], axis=-1)
    out = philox4x32_10(ctr, seed_key(seed))
    return out[np.arange(len(v)), v & 3]


def race_exponentials(seed: int, row: int, pos: int, v: np.ndarray,
                      stream: int = STREAM_RACE) -> np.ndarray:
    """E = -ln U, computed as -log1p(-(1 - U)) so U near 1 keeps full precision."""
    w = race_words(seed, row, pos, v, stream)
    return -np.log1p(-one_minus_uniform_from_word(w))
