"""Plain CPU oracle for the batched speculative verify step.

TEST INFRASTRUCTURE ONLY: this module defines what the verify step must return
so that tests can check the CUDA library against it.  Only tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
it.  It shares no code with the library: it reads logits, draft probabilities
and tokens as NumPy arrays and works in float64 throughout.

It is written step by step from these pages:

[AReno] inclusionAI/AReno PR #550, "feat(engine): MTP training loss and
    speculative decoding for bailing_v3".
    - "What does this PR do?", Phase 2: one forward verifies k+1 tokens per
      row; the sampler-equivalent target distribution (temperature, top-k,
      top-p) and exact chain rejection sampling keep the sampled distribution
      and the reported logprobs unchanged.
    - Table "On-policy accept probability of the MTP head": the closed-form
      acceptance alpha = sum_v min(p, q) and the expected accept length.
    - Table "Per-step optimizations": draws by Gumbel-max instead of
      multinomial, one-pass logprobs, no host syncs.
    - "How was it tested?": distribution preservation of rejection sampling
      (1.5% over 40k trials), exact under greedy.
[InfiniLM] InfiniTensor/InfiniLM PR #588, "feat: add mtp draft models for
    speculative decoding", section 4.1: exact bf16 ties between the top two
    candidates flip argmax between kernel paths, so ties must be defined.

Where the pages are silent the plainest reading is taken; each one is marked
READING below and listed in the design notes.

Notation: a row has k draft tokens x_0..x_{k-1} with draft distributions
q_0..q_{k-1}, and k+1 target logit vectors l_0..l_k (position j scores the
token after x_{j-1}).  p_j is the sampler-equivalent target distribution at
position j.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import philox

# Row flag bits.  The values are part of the library's interface; this file
# keeps its own copy.
F_MARGIN_ACCEPT = 1
F_MARGIN_DRAW = 2
F_MARGIN_TOPP = 4
F_NAN = 8
F_BAD_TOKEN = 16
F_BAD_PARAM = 32
F_RESIDUAL_EMPTY = 64

MARGIN = 1e-6          # decision margin, in probability units (READING)
FLT_MIN = 2.0 ** -126  # smallest normal float32


@dataclass
class PositionTarget:
    """The target distribution p_j at one verify position."""
    p: np.ndarray                 # float64 [V]; zero outside the kept set S
    greedy: bool
    kept: np.ndarray              # indices of S, in the total order
    log_z: float                  # greedy: ln sum exp(l - max); sampling: ln Z_S of exp((l-max)/T)
    topp_margin: bool = False


@dataclass
class RowResult:
    tokens: np.ndarray            # int32 [k+1]
    accept_len: int
    logprobs: np.ndarray          # float64 [k+1]
    alpha: np.ndarray             # float64 [k]
    flags: int
    # diagnostics used by the tests
    a: int = -1
    accept: list = field(default_factory=list)
    margin_accept: list = field(default_factory=list)   # per accept test taken, in chain order
    topp_margin: list = field(default_factory=list)     # per position 0..k
    draw_margin: bool = False


def total_order(l: np.ndarray) -> np.ndarray:
    """Vocabulary indices sorted by larger raw logit first, ties by smaller index.

    READING: the pages only say "sampler-equivalent"; [InfiniLM] section 4.1
    shows that exact ties are real in bf16, so they are broken by index.
    Ordering on raw logits avoids ties created by dividing by T.  A stable sort
    of -l gives exactly this order (-0.0 and +0.0 compare equal).
    """
    return np.argsort(-l, kind="stable")


def params_valid(T: float, P: float) -> bool:
    """READING: T must be 0 (greedy) or a positive normal float32; top_p in (0, 1]."""
    T_ok = (T == 0.0) or (np.isfinite(T) and T >= FLT_MIN)
    P_ok = np.isfinite(P) and (0.0 < P <= 1.0)
    return bool(T_ok and P_ok)


def target_distribution(l: np.ndarray, T: float, K: int, P: float) -> PositionTarget:
    """p_j from one logit vector [AReno "What does this PR do?", Phase 2].

    Greedy (T == 0): p is one-hot on the first entry of the total order.
    Sampling (T > 0), READING on the filter order: temperature -> top-k ->
    renormalise -> top-p -> renormalise.
      1. e_v = exp((l_v - max l) / T)   (softmax numerator of l / T)
      2. top-k: if 0 < K < V keep the first K entries of the total order.
      3. top-p: if 0 < P < 1, walk the kept entries in order and keep the
         shortest prefix whose renormalised mass reaches P (the entry that
         crosses P is kept).
      4. p = e / Z_S on the kept set S, zero elsewhere.
    """
    V = l.shape[0]
    order = total_order(l)
    m = l[order[0]]
    if T == 0.0:
        p = np.zeros(V)
        p[order[0]] = 1.0
        log_z = float(np.log(np.sum(np.exp(l - m))))
        return PositionTarget(p=p, greedy=True, kept=order[:1], log_z=log_z)

    e = np.exp((l - m) / T)
    kept = order[:K] if 0 < K < V else order
    e_kept = e[kept]
    z_k = np.sum(e_kept)
    topp_margin = False
    if 0.0 < P < 1.0:
        cum = np.cumsum(e_kept) / z_k
        i = int(np.searchsorted(cum, P, side="left"))   # first i with cum[i] >= P
        n_s = min(i + 1, len(kept))
        before = cum[n_s - 2] if n_s >= 2 else 0.0
        at = cum[n_s - 1]
        # READING: the top-p decision is uncertain when the mass before or at
        # the crossing entry lies within MARGIN of P.
        topp_margin = bool(abs(at - P) < MARGIN or abs(P - before) < MARGIN)
        kept = kept[:n_s]
    z_s = np.sum(e[kept])
    p = np.zeros(V)
    p[kept] = e[kept] / z_s
    return PositionTarget(p=p, greedy=False, kept=kept, log_z=float(np.log(z_s)),
                          topp_margin=topp_margin)


def token_logprob(l: np.ndarray, t: PositionTarget, tok: int, T: float) -> float:
    """Logprob reported for an emitted token.

    READING ("reported logprobs are unchanged", [AReno] Phase 2): the log of
    the sampler's own distribution p_j.  Under greedy decoding p_j is one-hot,
    so the raw softmax log-probability ln softmax(l)(tok) is reported instead.
    """
    m = np.max(l)
    if t.greedy:
        return float(l[tok] - m - t.log_z)
    return float((l[tok] - m) / T - t.log_z)


RACE_BLOCK = 256   # entries per block of the two-level race (READING)


def _best_two(s: np.ndarray):
    """Indices of the largest and second-largest score (first occurrence wins ties)."""
    i1 = int(np.argmax(s))
    if len(s) == 1:
        return i1, -1
    rest = s.copy()
    rest[i1] = -np.inf
    return i1, int(np.argmax(rest))


def exponential_race(r: np.ndarray, seed: int, row: int, pos: int, unc: np.ndarray,
                     streams=(philox.STREAM_RACE, philox.STREAM_BLOCK)):
    """Gumbel-max draw from the unnormalised weights r [AReno, "Per-step optimizations"].

    An exponential race: each competitor with weight w > 0 draws E = -ln U
    from the Philox stream keyed by (seed, row, position) and the largest
    score w / E wins; competitor i wins with probability w_i / sum(w)
    (equivalently argmax log w + G with Gumbel G = -ln E).  READING: the race
    runs in two levels so that only one block of entries needs a random
    number per entry.  Level 1 races the blocks of RACE_BLOCK consecutive
    indices with block weights W_b = sum of r over the block (stream 2);
    level 2 races the entries of the winning block (stream 1).  The product
    of the two winning probabilities is W_b / sum(W) * r_v / W_b = r_v /
    sum(r), so the draw is exact.  Ties go to the lower index at both levels.

    unc[v] is the magnitude whose relative error of 1e-6 bounds the error of
    r_v (p + q for a residual, p for a bonus draw); it sets the margin.
    streams: the Philox stream words of the entry and the block uniforms.
    Returns (winner, margin_flag).
    """
    support = np.nonzero(r > 0)[0]
    blocks = support // RACE_BLOCK
    ub, inv = np.unique(blocks, return_inverse=True)
    W = np.bincount(inv, weights=r[support])
    Wu = np.bincount(inv, weights=unc[support])
    Eb = philox.race_exponentials(seed, row, pos, ub, stream=streams[1])
    sb = W / Eb
    b1, b2 = _best_two(sb)
    margin = False
    if b2 >= 0 and sb[b1] - sb[b2] < MARGIN * (Wu[b1] / Eb[b1] + Wu[b2] / Eb[b2]):
        margin = True
    inb = support[blocks == ub[b1]]
    E = philox.race_exponentials(seed, row, pos, inb, stream=streams[0])
    s = r[inb] / E
    i1, i2 = _best_two(s)
    if i2 >= 0 and s[i1] - s[i2] < MARGIN * (unc[inb[i1]] / E[i1] + unc[inb[i2]] / E[i2]):
        margin = True
    return int(inb[i1]), margin


def verify_row(logits_r: np.ndarray, q_r: np.ndarray, drafts_r: np.ndarray,
               T: float, K: int, P: float, seed: int, row: int) -> RowResult:
    """The verify step for one row.

    logits_r: [k+1, V] target logits (the exact values the library reads).
    q_r:      [k, V] draft distributions, used exactly as given (no filter,
              no renormalisation).
    drafts_r: [k] draft tokens.
    """
    k1, V = logits_r.shape
    k = k1 - 1
    flags = 0
    tokens = np.full(k + 1, -1, dtype=np.int32)
    logprobs = np.zeros(k + 1)
    alpha = np.zeros(k)

    # Invalid input (READING): a NaN or +inf logit, or a position whose logits
    # are all -inf, makes the whole row invalid.
    if np.any(np.isnan(logits_r)) or np.any(logits_r == np.inf) or \
            np.any(np.max(logits_r, axis=1) == -np.inf):
        return RowResult(tokens, 0, logprobs, alpha, F_NAN)

    if not params_valid(T, P):
        flags |= F_BAD_PARAM
        T = 0.0            # READING: an invalid row is sampled greedily
    if not (0 < K < V):
        K = 0              # top-k disabled
    if P >= 1.0 or not (P > 0.0):
        P = 1.0            # top-p disabled

    targets = []
    topp_margin = []
    for j in range(k + 1):
        t = target_distribution(logits_r[j], T, K, P)
        if t.topp_margin:
            flags |= F_MARGIN_TOPP
        targets.append(t)
        topp_margin.append(t.topp_margin)

    # alpha_j = sum_v min(p_j(v), q_j(v)) for every draft position
    # [AReno, accept-probability table].  READING: computed whether or not
    # position j is reached; masking by accept length is the caller's.
    for j in range(k):
        alpha[j] = np.sum(np.minimum(targets[j].p, q_r[j]))

    # Exact chain rejection sampling [AReno Phase 2]: accept x_j with
    # probability min(1, p_j(x_j) / q_j(x_j)), written without a division as
    # u_j * q_j(x_j) < p_j(x_j) with u_j uniform in (0, 1).
    # READING: every draft token is validated, reached or not; an
    # out-of-range draft is rejected when the chain reaches it.
    if any(not (0 <= int(x) < V) for x in drafts_r[:k]):
        flags |= F_BAD_TOKEN
    a = k
    accept, margin_accept = [], []
    for j in range(k):
        x = int(drafts_r[j])
        if 0 <= x < V:
            px, qx = targets[j].p[x], q_r[j][x]
        else:
            px, qx = 0.0, 0.0
        u = philox.accept_uniform(seed, row, j)
        acc = bool(u * qx < px)
        if MUTATION == "inverted_accept":
            acc = bool(u * px < qx)
        # The decision is exact when p is exactly 0 or 1; otherwise flag a margin.
        marg = bool(0.0 < px < 1.0 and abs(u * qx - px) < MARGIN)
        accept.append(acc)
        margin_accept.append(marg)
        if marg:
            flags |= F_MARGIN_ACCEPT
        if not acc:
            a = j
            break

    # Draw at position a: from normalise(max(p_a - q_a, 0)) after a rejection,
    # from p_k when every draft was accepted (the bonus token).
    p_a = targets[a].p
    if a < k:
        r = np.maximum(p_a - q_r[a], 0.0)
        q_a = q_r[a]
        if MUTATION == "residual_is_p":
            r = p_a.copy()
    else:
        r = p_a.copy()
        q_a = np.zeros(V)
    if not np.any(r > 0):
        # READING: an empty residual (p_a <= q_a everywhere) falls back to p_a.
        flags |= F_RESIDUAL_EMPTY
        r = p_a.copy()
        q_a = np.zeros(V)
    # READING: a draw is uncertain when the best two scores at either level
    # differ by less than a relative error of MARGIN in p and q would move them.
    y, draw_margin = exponential_race(r, seed, row, a, p_a + q_a)
    if draw_margin:
        flags |= F_MARGIN_DRAW

    for j in range(a):
        tokens[j] = drafts_r[j]
        logprobs[j] = token_logprob(logits_r[j], targets[j], int(drafts_r[j]), T)
    tokens[a] = y
    logprobs[a] = token_logprob(logits_r[a], targets[a], y, T)
    res = RowResult(tokens, a + 1, logprobs, alpha, flags, a=a, accept=accept,
                    margin_accept=margin_accept, topp_margin=topp_margin,
                    draw_margin=bool(draw_margin))
    return res


def verify(logits: np.ndarray, q: np.ndarray, drafts: np.ndarray,
           temperature: np.ndarray, top_k: np.ndarray, top_p: np.ndarray,
           seed: int, rows=None, row_base: int = 0) -> dict:
    """Batched verify over `rows` (default: all rows).

    logits [B, k+1, V] and q [B, k, V] are converted to float64; the returned
    arrays are indexed like `rows`.

    Row r of this batch draws its random numbers as row `row_base + r` of the
    stream keyed by (seed, row, position).  READING: the random stream is
    keyed by the row's index in the whole batch, so a batch split into
    blocks of rows (one block per GPU) reproduces the whole batch's draws
    when every block passes the index of its first row as row_base.  The stream row is a 32-bit counter word, so
    row_base + r wraps modulo 2^32.

    Besides the outputs, the result holds each row's margin record: the
    chain's reach `a`, the accept margins of the tests taken
    (`margin_accept`, [rows, k], False past the chain), the top-p margins per
    position (`topp_margin`, [rows, k+1]) and the draw margin (`draw_margin`).
    """
    B = logits.shape[0]
    k = logits.shape[1] - 1
    rows = list(range(B)) if rows is None else list(rows)
    out = {"tokens": [], "accept_len": [], "logprobs": [], "alpha": [], "flags": [],
           "a": [], "margin_accept": [], "topp_margin": [], "draw_margin": [],
           "rows": np.asarray(rows, dtype=np.int64)}
    for r in rows:
        res = verify_row(np.asarray(logits[r], dtype=np.float64),
                         np.asarray(q[r], dtype=np.float64), np.asarray(drafts[r]),
                         float(temperature[r]), int(top_k[r]), float(top_p[r]), seed,
                         (int(row_base) + int(r)) % (1 << 32))
        out["tokens"].append(res.tokens)
        out["accept_len"].append(res.accept_len)
        out["logprobs"].append(res.logprobs)
        out["alpha"].append(res.alpha)
        out["flags"].append(res.flags)
        out["a"].append(res.a)
        ma = np.zeros(k, dtype=bool)
        ma[:len(res.margin_accept)] = res.margin_accept
        out["margin_accept"].append(ma)
        tm = np.zeros(k + 1, dtype=bool)
        tm[:len(res.topp_margin)] = res.topp_margin
        out["topp_margin"].append(tm)
        out["draw_margin"].append(res.draw_margin)
    for key in ("tokens", "accept_len", "logprobs", "alpha", "flags", "a", "draw_margin"):
        out[key] = np.asarray(out[key])
    out["margin_accept"] = np.asarray(out["margin_accept"], dtype=bool).reshape(len(rows), k)
    out["topp_margin"] = np.asarray(out["topp_margin"], dtype=bool).reshape(len(rows), k + 1)
    return out


def expected_accept_length(alphas) -> float:
    """E[accept_len] = 1 + sum_{i=1..k} prod_{j<i} alpha_j.

    With drafts drawn from q, draft j is accepted with probability alpha_j
    (Leviathan-style closed form, [AReno] accept-probability table); the
    accept length counts the accepted drafts plus the drawn token.
    """
    total, prod = 1.0, 1.0
    for a in alphas:
        prod *= float(a)
        total += prod
    return total


# Negative-control hook for the tests: None in normal use.  A test may set it
# to "residual_is_p" or "inverted_accept" to plant a known mistake in this
# oracle and check that the distribution tests catch it.
MUTATION = None
