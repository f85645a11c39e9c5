"""GPU parity of spec_verify against the oracle (element by element).

Runs through the C ABI (ctypes binding).  Sizes: the tiny, top-p, mixed and
adversarial workloads are compared on every row at their full sizes (the
oracle over the adversarial workload's 256 rows runs in a process pool).
Random small cases cover odd and tiny vocabularies, k = 0..4, both dtypes,
every filter combination, the general threshold paths (top-k above the
candidate limit, top-p without top-k), ties, masked entries and invalid
inputs; top-k 8, 9, 127, 128 and 129 at V = 151936 with exact ties at the
K-th entry cover the hand-over between the candidate lists and the general
path.  A batch split into row blocks with row_base must equal the whole
batch bit for bit, and a wait that runs out must come back as a flagged row.
"""
import numpy as np
import pytest
import torch

from oracle import verify as ov
from speculative_decoding_verify_07_gb300 import synth
from tests.gpu_harness import compare, host_outputs, run_gpu, run_oracle, to_device
from tests.oracle_pool import oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def test_device_philox_matches_oracle():
    from oracle import philox
    from speculative_decoding_verify_07_gb300 import binding as sv
    rng = np.random.default_rng(5)
    n = 1 << 18
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    ctr[:16] = 0
    ctr[16:32] = 0xFFFFFFFF
    for seed in (0, 0x0123456789ABCDEF, 2 ** 64 - 1):
        dev = sv.philox4x32_10(torch.from_numpy(ctr.view(np.int32)).cuda(), seed)
        got = dev.cpu().numpy().view(np.uint32)
        exp = philox.philox4x32_10(ctr, philox.seed_key(seed))
        assert np.array_equal(got, exp)


def test_parity_tiny():
    inp = synth.make_tiny()
    compare(run_gpu(inp), run_oracle(inp), "tiny")


def test_parity_topp_workload():
    inp = synth.make_topp()
    s = compare(run_gpu(inp), run_oracle(inp), "topp")
    assert s["exempt"] <= 2


def test_parity_mixed_workload():
    inp = synth.make_mixed()
    compare(run_gpu(inp), run_oracle(inp), "mixed")


def test_parity_adversarial_all_rows():
    inp = synth.make_adversarial()
    gpu = run_gpu(inp)
    orc = oracle_rows("adversarial", range(256))
    s = compare(gpu, orc, "adversarial")
    # whole-batch properties: the first half rejects early, the second half accepts everything
    assert np.mean(gpu["accept_len"][:128]) < 1.2
    assert np.all(gpu["accept_len"][128:] >= 4)
    assert np.all(gpu["flags"] & (ov.F_NAN | ov.F_BAD_TOKEN | ov.F_BAD_PARAM) == 0)
    assert s["rows"] == 256


def _ktie_case(K, B=4, k=2, V=151936, seed=0):
    """Mixed-recipe bf16 logits with top-k K; in every (row, position) the
    K-th largest value is copied onto three tokens ranked below K, so equal
    keys straddle the K-th entry of the total order."""
    rng = np.random.default_rng(500 + K + seed)
    logits = synth.round_to_bf16(synth._spiked_logits(rng, B, k + 1, V))
    for b in range(B):
        for j in range(k + 1):
            row = logits[b, j]
            order = np.argsort(-row, kind="stable")
            v = row[order[K - 1]]
            for dst in rng.choice(order[K + 10:], size=3, replace=False):
                row[dst] = v
    q = synth._noisy_q(rng, logits, k, 0.7)
    drafts = synth._sample_rows(rng, q.astype(np.float64))
    T = np.full(B, 0.8, np.float32)
    Kk = np.full(B, K, np.int32)
    P = np.array([1.0 if b % 2 == 0 else 0.9 for b in range(B)], np.float32)
    return _Case(logits, q, drafts, T, Kk, P, 1000 + K, "bf16")


@pytest.mark.parametrize("K", [8, 9, 127, 128, 129])
def test_parity_topk_boundary_with_ties(K):
    case = _ktie_case(K)
    compare(run_gpu(case), run_oracle(case), f"top-k {K} ties")


class _Case:
    def __init__(self, logits, q, drafts, T, K, P, seed, dtype):
        self.logits, self.q, self.drafts = logits, q, drafts
        self.temperature, self.top_k, self.top_p = T, K, P
        self.seed, self.dtype = seed, dtype


def _random_case(rng, B, k, V, dtype, param_mode):
    logits = rng.normal(0, 2.5, size=(B, k + 1, V)).astype(np.float32)
    if dtype == "bf16":
        logits = synth.round_to_bf16(logits)
    # coarse values for ties in some rows
    for b in range(0, B, 3):
        logits[b] = np.round(logits[b] * 2) / 2
    if V > 4:
        logits[1 % B, :, : V // 7] = -np.inf       # masked entries
    q = np.empty((B, k, V), np.float32)
    for b in range(B):
        for j in range(k):
            z = logits[b, j].astype(np.float64)
            z = np.where(np.isfinite(z), z, -30.0) + rng.normal(0, 0.8, V)
            e = np.exp(z - z.max())
            q[b, j] = (e / e.sum()).astype(np.float32)
    drafts = np.empty((B, k), np.int32)
    for b in range(B):
        for j in range(k):
            pj = q[b, j].astype(np.float64)
            drafts[b, j] = rng.choice(V, p=pj / pj.sum())
    T = np.ones(B, np.float32)
    K = np.zeros(B, np.int32)
    P = np.ones(B, np.float32)
    for b in range(B):
        mode = param_mode if param_mode != "mix" else ["greedy", "temp", "topk", "topp", "both",
                                                          "bigk", "bigk_topp", "k1"][b % 8]
        if mode == "greedy":
            T[b] = 0.0
        elif mode == "temp":
            T[b] = 0.6
        elif mode == "topk":
            T[b], K[b] = 0.9, max(1, min(V - 1, 20))
        elif mode == "topp":
            T[b], P[b] = 1.1, 0.8
        elif mode == "both":
            T[b], K[b], P[b] = 0.7, max(1, min(V - 1, 40)), 0.9
        elif mode == "bigk":
            T[b], K[b] = 1.0, max(1, min(V - 1, 300))
        elif mode == "bigk_topp":
            T[b], K[b], P[b] = 0.8, max(1, min(V - 1, 500)), 0.95
        elif mode == "k1":
            T[b], K[b] = 1.0, 1
    return _Case(logits, q, drafts, T, K, P, int(rng.integers(0, 2 ** 63)), dtype)


@pytest.mark.parametrize("V", [1, 2, 7, 8, 9, 100, 1000, 4097, 33331])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_parity_random_small(V, dtype):
    rng = np.random.default_rng(V * 7 + (dtype == "bf16"))
    for k in (0, 1, 2, 4):
        case = _random_case(rng, B=16, k=k, V=V, dtype=dtype, param_mode="mix")
        compare(run_gpu(case), run_oracle(case), f"V={V} {dtype} k={k}")


def test_parity_large_topk_and_topp_only():
    rng = np.random.default_rng(123)
    for mode in ("bigk", "bigk_topp", "topp", "both"):
        case = _random_case(rng, B=8, k=2, V=50000, dtype="bf16", param_mode=mode)
        compare(run_gpu(case), run_oracle(case), mode)


def test_parity_topp_fp32_refinement_levels():
    # fp32 keys are dense: the crossing bin spans many keys and takes
    # several refinement levels; coarse rows put exact ties at the crossing
    rng = np.random.default_rng(321)
    for V in (40000, 2048 * 3 + 5):
        case = _random_case(rng, B=8, k=2, V=V, dtype="f32", param_mode="topp")
        compare(run_gpu(case), run_oracle(case), f"top-p fp32 V={V}")


def test_parity_topp_dense_keys_extreme_p_and_full_vocabulary():
    rng = np.random.default_rng(404)
    # bf16 logits packed near zero: a crossing bin holds hundreds of keys, two
    # refinement levels, tiles with more keys than their lists hold (the ties
    # pass runs)
    case = _random_case(rng, B=6, k=2, V=30000, dtype="bf16", param_mode="topp")
    case.logits[:] = synth.round_to_bf16(rng.normal(0, 0.02, size=case.logits.shape).astype(np.float32))
    case.top_p[:] = np.array([0.8, 0.5, 0.95, 0.3, 0.99, 0.7], np.float32)
    compare(run_gpu(case), run_oracle(case), "top-p dense keys")
    # extreme P: the crossing at the maximum, and nearly the whole row
    case = _random_case(rng, B=4, k=2, V=20000, dtype="bf16", param_mode="topp")
    case.top_p[:] = np.array([1e-4, 0.02, 0.9999, 0.99999], np.float32)
    compare(run_gpu(case), run_oracle(case), "top-p extreme P")
    # fp32 at the bench vocabulary: four refinement levels and the ties pass
    case = _random_case(rng, B=4, k=2, V=151936, dtype="f32", param_mode="topp")
    compare(run_gpu(case), run_oracle(case), "top-p fp32 V=151936")


def test_parity_topp_rows_above_the_shared_order_limit():
    # 300 rows (the row order then lives in the workspace), every class, and
    # top-p rows holding NaN, +inf and all -inf positions
    rng = np.random.default_rng(77)
    case = _random_case(rng, B=300, k=2, V=3000, dtype="bf16", param_mode="mix")
    topp = [b for b in range(300) if b % 8 == 3]
    case.logits[topp[0], 1, 17] = np.nan
    case.logits[topp[1], 0, 9] = np.inf
    case.logits[topp[2], 2, :] = -np.inf
    gpu = run_gpu(case)
    compare(gpu, run_oracle(case), "300 rows")
    for r in topp[:3]:
        assert gpu["flags"][r] & ov.F_NAN and gpu["accept_len"][r] == 0


def test_invalid_inputs_set_flags():
    rng = np.random.default_rng(9)
    case = _random_case(rng, B=8, k=2, V=513, dtype="f32", param_mode="temp")
    case.logits[0, 1, 5] = np.nan
    case.logits[1, 2, 7] = np.inf
    case.logits[2, 0, :] = -np.inf
    case.drafts[3, 1] = 513
    case.drafts[4, 0] = -5
    case.temperature[5] = -1.0
    case.top_p[6] = 0.0
    gpu = run_gpu(case)
    compare(gpu, run_oracle(case), "invalid")
    assert gpu["flags"][0] == ov.F_NAN and gpu["accept_len"][0] == 0
    assert np.all(gpu["tokens"][0] == -1)
    assert gpu["flags"][3] & ov.F_BAD_TOKEN and gpu["flags"][5] & ov.F_BAD_PARAM


def test_empty_batch_and_workspace_left_clean():
    from speculative_decoding_verify_07_gb300 import binding as sv
    case = _random_case(np.random.default_rng(1), B=5, k=3, V=1000, dtype="bf16", param_mode="mix")
    logits, q, x, params = to_device(case)
    ws = sv.new_workspace(5, 3, 1000, "cuda")
    for _ in range(3):
        sv.spec_verify(logits, q, x, params, 7, workspace=ws)
    torch.cuda.synchronize()
    # three calls, numbered 0, 1, 2 (tags 1, 2, 3): the last counted in set
    # 0, and set 1, the next call's, is zero, as are the per-row tickets
    # (padded to 256 bytes) and the two tile counters per (row, position)
    # (padded to 256 bytes); the epoch word holds the last call's tag
    B, U = 5, 5 * 4
    tickets = 256
    counters = tickets + 256 * ((B * 4 + 255) // 256)
    records = counters + 256 * ((U * 8 + 255) // 256)
    assert int(ws[24:28].view(torch.int32).item()) == 0
    assert int(ws[64:96].count_nonzero()) == 0
    assert int(ws[tickets:records].count_nonzero()) == 0
    assert int(ws[236:240].view(torch.int32).item()) == 3
    assert int(ws[0:8].view(torch.int64).item()) == 3 * torch.cuda.get_device_properties(0).multi_processor_count
    # dirty records behind them do not matter: every record word carries the
    # call's tag, so results stay identical
    ref = sv.spec_verify(logits, q, x, params, 7, workspace=ws)
    ws[records:].fill_(0xAB)
    again = sv.spec_verify(logits, q, x, params, 7, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(ref.tokens, again.tokens) and torch.equal(ref.logprobs, again.logprobs)
    e = torch.empty((0, 3, 1000), dtype=torch.bfloat16, device="cuda")
    out = sv.spec_verify(e, torch.empty((0, 2, 1000), device="cuda"),
                         torch.empty((0, 2), dtype=torch.int32, device="cuda"),
                         sv.make_params([], [], [], "cuda"), 0)
    assert out.tokens.shape == (0, 3)


def test_parity_many_units_several_settle_rounds():
    # 96 rows at k = 4: more settle tasks than settle warps, so warps take
    # several tasks (the earlier ones draw with the rolled race, the last
    # with the inline one) and the unfiltered rows come in several waves
    rng = np.random.default_rng(8080)
    case = _random_case(rng, B=96, k=4, V=12289, dtype="bf16", param_mode="mix")
    compare(run_gpu(case), run_oracle(case), "96 rows k=4")
    case = _random_case(rng, B=96, k=4, V=12289, dtype="bf16", param_mode="temp")
    compare(run_gpu(case), run_oracle(case), "96 unfiltered rows k=4")


def test_one_workspace_through_calls_of_every_row_class():
    # consecutive calls on one workspace alternate between the two sets of
    # call counters: every call, whatever rows it holds (the top-p passes use
    # the grid barrier count and refinement flags, large top-k rows the
    # general-path counter), starts from a zeroed set and leaves the next
    # one zeroed
    from speculative_decoding_verify_07_gb300 import binding as sv
    rng = np.random.default_rng(2024)
    B, k, V = 24, 2, 20000
    ws = sv.new_workspace(B, k, V, "cuda")
    for i, mode in enumerate(["mix", "topp", "greedy", "bigk", "mix", "topp", "both"]):
        case = _random_case(rng, B=B, k=k, V=V, dtype="bf16", param_mode=mode)
        logits, q, x, params = to_device(case)
        out = host_outputs(sv.spec_verify(logits, q, x, params, case.seed, workspace=ws))
        torch.cuda.synchronize()
        compare(out, run_oracle(case), f"call {i} ({mode})")
        assert _last_call_errors(ws) == 0
        assert int(ws[236:240].view(torch.int32).item()) == i + 1
        cs = int(ws[24:28].view(torch.int32).item())
        assert cs == i % 2
        nxt = 32 + 32 * (1 - cs)
        assert int(ws[nxt:nxt + 32].count_nonzero()) == 0


def test_deterministic_and_graph_replay_bit_identical():
    from speculative_decoding_verify_07_gb300 import binding as sv
    inp = synth.make_mixed(B=16, V=32768)
    logits, q, x, params = to_device(inp)
    ws = sv.new_workspace(16, 2, 32768, "cuda")
    ref = sv.spec_verify(logits, q, x, params, 11, workspace=ws)
    again = sv.spec_verify(logits, q, x, params, 11, workspace=ws)
    torch.cuda.synchronize()
    for name in ("tokens", "accept_len", "logprobs", "alpha", "flags"):
        assert torch.equal(getattr(ref, name), getattr(again, name)), name
    out = sv.VerifyOutputs(16, 2, "cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sv.spec_verify(logits, q, x, params, 11, out=out, workspace=ws)   # warm-up on the side stream
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        sv.spec_verify(logits, q, x, params, 11, out=out, workspace=ws)
    for name in ("tokens", "logprobs"):
        getattr(out, name).fill_(0)
    g.replay()
    torch.cuda.synchronize()
    for name in ("tokens", "accept_len", "logprobs", "alpha", "flags"):
        assert torch.equal(getattr(ref, name), getattr(out, name)), name


def test_row_base_split_equals_whole_batch():
    from speculative_decoding_verify_07_gb300 import binding as sv
    inp = synth.make_mixed(B=16, V=32768)
    logits, q, x, params = to_device(inp)
    whole = host_outputs(sv.spec_verify(logits, q, x, params, 19))
    lo = host_outputs(sv.spec_verify(logits[:9], q[:9], x[:9], params[:9], 19, row_base=0))
    hi = host_outputs(sv.spec_verify(logits[9:], q[9:], x[9:], params[9:], 19, row_base=9))
    torch.cuda.synchronize()
    for key in ("tokens", "accept_len", "logprobs", "alpha", "flags"):
        assert np.array_equal(np.concatenate([lo[key], hi[key]]), whole[key]), key
    # and the second block matches the oracle run on that block with the same base
    orc_hi = ov.verify(inp.logits[9:], inp.q[9:], inp.drafts[9:], inp.temperature[9:], inp.top_k[9:],
                       inp.top_p[9:], 19, row_base=9)
    compare(hi, orc_hi, "row_base 9")
    compare(whole, run_oracle(inp, seed=19), "whole")


def _last_call_errors(ws):
    """The error bits of the last call: its counter set (bytes 24..27) picks
    the word (bytes 52..55 for set 0, 84..87 for set 1)."""
    cs = int(ws[24:28].view(torch.int32).item())
    assert cs in (0, 1)
    off = 52 + 32 * cs
    return int(ws[off:off + 4].view(torch.int32).item())


def test_timed_out_wait_flags_the_row_and_leaves_the_context_usable():
    from speculative_decoding_verify_07_gb300 import binding as sv
    case = _random_case(np.random.default_rng(31), B=4, k=2, V=4096, dtype="bf16", param_mode="mix")
    logits, q, x, params = to_device(case)
    ws = sv.new_workspace(4, 2, 4096, "cuda")
    ws[20:24].view(torch.int32).fill_(1)        # test hook: row 0's finalize waits for nothing
    out = host_outputs(sv.spec_verify(logits, q, x, params, case.seed, workspace=ws))
    torch.cuda.synchronize()
    assert out["flags"][0] & sv.F_TIMEOUT and out["accept_len"][0] == 0
    assert np.all(out["tokens"][0] == -1)
    assert _last_call_errors(ws) & 4       # the record-wait bit of the last call
    orc = run_oracle(case, rows=[1, 2, 3])
    compare(out, orc, "rows after the timeout")
    # the same workspace, hook cleared: every row comes back normally
    ws[20:24].view(torch.int32).fill_(0)
    again = host_outputs(sv.spec_verify(logits, q, x, params, case.seed, workspace=ws))
    torch.cuda.synchronize()
    compare(again, run_oracle(case), "after the timeout")
    assert _last_call_errors(ws) == 0


def test_grid_barrier_that_gives_up_flags_the_top_p_rows():
    from speculative_decoding_verify_07_gb300 import binding as sv
    case = _random_case(np.random.default_rng(32), B=8, k=2, V=5000, dtype="bf16", param_mode="mix")
    logits, q, x, params = to_device(case)
    ws = sv.new_workspace(8, 2, 5000, "cuda")
    ws[20:24].view(torch.int32).fill_(2)        # test hook: one CTA misses a top-p grid barrier
    out = host_outputs(sv.spec_verify(logits, q, x, params, case.seed, workspace=ws))
    torch.cuda.synchronize()
    topp = [3]                                  # the mix gives row 3 top-p without top-k
    for r in topp:
        assert out["flags"][r] & sv.F_TIMEOUT and out["accept_len"][r] == 0
        assert np.all(out["tokens"][r] == -1)
    assert _last_call_errors(ws) & 16       # the barrier bit of the last call
    others = [r for r in range(8) if r not in topp]
    compare(out, run_oracle(case, rows=others), "rows outside the top-p passes")
    # hook cleared: every row comes back normally and no wait gave up
    ws[20:24].view(torch.int32).fill_(0)
    again = host_outputs(sv.spec_verify(logits, q, x, params, case.seed, workspace=ws))
    torch.cuda.synchronize()
    compare(again, run_oracle(case), "after the barrier timeout")
    assert _last_call_errors(ws) == 0


def test_gpu_distribution_preserved_40k_rows():
    """The page's criterion run on the GPU path: 40k rows, drafts drawn from q."""
    from scipy import stats
    from speculative_decoding_verify_07_gb300 import binding as sv
    V, k, B = 6, 2, 40000
    rng = np.random.default_rng(4)
    base = rng.normal(0, 1.2, size=(k + 1, V)).astype(np.float32)
    qrow = rng.dirichlet(np.full(V, 0.6), size=k).astype(np.float32)
    logits = np.broadcast_to(base, (B, k + 1, V)).copy()
    q = np.broadcast_to(qrow, (B, k, V)).copy()
    drafts = np.stack([rng.choice(V, size=B, p=qrow[j] / qrow[j].sum()) for j in range(k)], 1)
    case = _Case(logits, q, drafts.astype(np.int32), np.ones(B, np.float32),
                 np.zeros(B, np.int32), np.ones(B, np.float32), 77, "f32")
    gpu = run_gpu(case)
    p0 = ov.target_distribution(base[0].astype(np.float64), 1.0, 0, 1.0).p
    c = np.bincount(gpu["tokens"][:, 0], minlength=V).astype(float)
    tv = 0.5 * np.abs(c / B - p0).sum()
    pv = stats.chisquare(c, p0 * B).pvalue
    assert tv <= 0.015 and pv > 1e-3, (tv, pv)
    # and the sampled rows agree with the oracle exactly
    compare(gpu, run_oracle(case, rows=list(range(0, B, 997))), "40k")
