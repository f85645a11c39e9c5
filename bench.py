#!/usr/bin/env python3
"""Benchmark of the speculative verify hot path on GB300.

One step = one pass of the whole hot path over one synthetic batch:
  spec_verify  on 64 rows, k=2, V=151936, bf16 logits, mixed per-row params
               (25% greedy, 50% T=0.7 top-k 50 top-p 0.9, 25% T=1), exact
               ties in 1% of positions;
  spec_commit  of those 64 rows' accepted states (accept_len from the verify)
               from a stacked verify buffer of 24 layers x 3 states of fp32
               recurrent state 16x128x128 plus bf16 conv state 4x4096.
Metric: rows/s (whole job), with HBM GB/s against the measured peak.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 launch one process per GPU with torch.distributed.run; every rank
processes its own batch (weak scaling, no collective on the data path).
`--impl reference` times the CPU oracle (the baseline arm) on host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "spec-verify rows/s at V=151936,k=2; achieved HBM GB/s vs GB300 peak"
# spec_verify launches one cooperative kernel; its sources
VERIFY_SOURCES = ["spec_verify.cu", "spec_kernel.cu", "spec_settle.cuh", "spec_general.cuh",
                  "spec_verify_common.cuh", "spec_device.cuh"]
VERIFY_LAUNCHES = 1
B, K, V = 64, 2, 151936
N_SETS = 4   # rotating verify input sets (each ~136 MB, together > L2)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "speculative_decoding_verify_07_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_record(kernel, src_hash):
    """DRAM bytes per launch from the committed ncu summary, if it matches this source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(kernel)
        if rec and rec.get("source_hash") == src_hash:
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def verify_algorithmic_bytes(inp):
    """Bytes the method must move for one verify launch.

    Every logit is read.  q is read in full at positions whose target
    distribution has (potentially) full support; where the kept set is
    bounded (greedy: one entry; top-k <= 128: at most top_k entries) only the
    kept entries, the draft token and the argmax are read.
    """
    Bn, k1, Vn = inp.logits.shape
    k = k1 - 1
    es = 2 if inp.dtype == "bf16" else 4
    total = Bn * k1 * Vn * es
    for r in range(Bn):
        T, Kt = float(inp.temperature[r]), int(inp.top_k[r])
        if T == 0.0:
            total += k * 2 * 4
        elif 0 < Kt <= 128:
            total += k * (Kt + 2) * 4
        else:
            total += k * Vn * 4
    total += Bn * k * 4 + Bn * 16                       # draft tokens, params
    total += Bn * (k1 * 4 + 4 + k1 * 4 + k * 4 + 4)     # outputs
    return total


class ClockSampler:
    """Samples the SM clock and the clock-event reasons while the timed steps
    run: NVML (read-only queries through the driver's libnvidia-ml, one
    sample every 2 ms from a thread), else nvidia-smi every 100 ms."""

    # NVML clock-event reason bits that reject or annotate a measurement
    NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                    0x40: "hw_thermal_slowdown"}

    def __init__(self, index):
        self.proc = None
        self.thread = None
        self.samples = []
        self.path = os.path.join(tempfile.gettempdir(), f"spec_clocks_{os.getpid()}.csv")
        self.index = index

    def _nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return None
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            return None
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
        if reasons_fn is None:
            return None
        return lib, h, reasons_fn

    def _poll(self, lib, h, reasons_fn):
        import ctypes
        mhz, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop:
            if (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0 and
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                    reasons_fn(h, ctypes.byref(rs)) == 0):
                self.samples.append((float(mhz.value), float(mx.value), int(rs.value)))
            time.sleep(0.002)

    def __enter__(self):
        nv = None
        try:
            nv = self._nvml()
        except Exception:
            nv = None
        if nv is not None:
            import threading
            self.stop = False
            self.thread = threading.Thread(target=self._poll, args=nv, daemon=True)
            self.thread.start()
            return self
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.thread is not None:
            self.stop = True
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.thread is not None:
            sm = [x[0] for x in self.samples]
            reasons = sorted({n for x in self.samples for bit, n in self.NVML_REASONS.items() if x[2] & bit})
            return {"sm_mhz": statistics.median(sm) if sm else None,
                    "sm_max_mhz": max(x[1] for x in self.samples) if sm else None,
                    "reasons": reasons, "samples": len(sm), "source": "nvml"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


def dist_setup(n_gpus):
    import torch
    rank, world, local = 0, 1, 0
    if n_gpus > 1 or "RANK" in os.environ:
        import torch.distributed as dist
        rank = int(os.environ.get("RANK", 0))
        world = int(os.environ.get("WORLD_SIZE", 1))
        local = int(os.environ.get("LOCAL_RANK", 0))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """The slowest rank's value (the job's time is the slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_rank, world, elapsed_s):
    """Weak scaling: every rank processes its own batch; throughput counts all ranks."""
    return rows_per_rank * world / elapsed_s


def cpu_oracle_sample(inp, n_rows=16, commit_rows=2):
    """Time the oracle as it stands on a bounded sample of the workload."""
    from oracle import commit as oc
    from oracle import verify as ov
    from speculative_decoding_verify_07_gb300 import synth
    rows = list(range(n_rows))
    t0 = time.perf_counter()
    ov.verify(inp.logits, inp.q, inp.drafts, inp.temperature, inp.top_k, inp.top_p, inp.seed, rows=rows)
    t_verify = (time.perf_counter() - t0) / n_rows
    sh = synth.CommitShape()
    rng = np.random.default_rng(0)
    vrec = rng.standard_normal((sh.L, commit_rows, sh.S, sh.H, sh.Dk, sh.Dv), dtype=np.float32)
    vconv = rng.integers(0, 1 << 16, size=(sh.L, commit_rows, sh.S, sh.W, sh.C), dtype=np.uint16)
    crec = np.zeros((sh.L, commit_rows, sh.H, sh.Dk, sh.Dv), np.float32)
    cconv = np.zeros((sh.L, commit_rows, sh.W, sh.C), np.uint16)
    acc = np.full(commit_rows, 2, np.int32)
    t0 = time.perf_counter()
    oc.commit(vrec, vconv, acc, None, crec, cconv)
    t_commit = (time.perf_counter() - t0) / commit_rows
    per_row = t_verify + t_commit
    return {"value": 1.0 / per_row, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"oracle verify on {n_rows} of the 64 rows + oracle commit of {commit_rows} rows "
                      f"(24 layers); {t_verify * 1e3:.1f} ms/row verify, {t_commit * 1e3:.1f} ms/row commit; "
                      "single thread (NumPy)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", 0))
    if rank != 0:
        return
    from speculative_decoding_verify_07_gb300 import synth
    inp = synth.make_mixed()
    for _ in range(args.warmup):
        cpu_oracle_sample(inp, n_rows=2, commit_rows=1)
    t0 = time.perf_counter()
    per = []
    for _ in range(args.steps):
        per.append(cpu_oracle_sample(inp, n_rows=4, commit_rows=1))
    el = time.perf_counter() - t0
    value = statistics.median(p["value"] for p in per)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "mixed verify 64x2x151936 bf16 + commit 24L x 64 rows (sampled rows)",
                       "sample_per_step": "oracle verify on 4 rows + oracle commit of 1 row"},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": per[0]["sample"]},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_ours(args):
    import torch

    from speculative_decoding_verify_07_gb300 import binding as sv
    from speculative_decoding_verify_07_gb300 import synth

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)

    # ---- inputs resident in HBM ----
    sets = []
    inps = []
    for i in range(N_SETS):
        inp = synth.make_mixed(seed_offset=100 * i)
        inps.append(inp)
        logits = torch.from_numpy(inp.logits).to(torch.bfloat16).to(dev)
        q = torch.from_numpy(inp.q).to(dev)
        x = torch.from_numpy(inp.drafts).to(dev)
        params = sv.make_params(inp.temperature, inp.top_k, inp.top_p, dev)
        sets.append((logits, q, x, params, inp.seed + i))
    sh = synth.CommitShape()
    g = torch.Generator(device=dev)
    g.manual_seed(1004 + rank)
    vrec = torch.empty((sh.L, sh.B, sh.S, sh.H, sh.Dk, sh.Dv), dtype=torch.float32, device=dev)
    vrec.view(torch.int32).random_(generator=g)
    vconv = torch.randint(-32768, 32767, (sh.L, sh.B, sh.S, sh.W, sh.C), dtype=torch.int16,
                          device=dev, generator=g)
    crec = torch.zeros((sh.L, sh.slots, sh.H, sh.Dk, sh.Dv), dtype=torch.float32, device=dev)
    cconv = torch.zeros((sh.L, sh.slots, sh.W, sh.C), dtype=torch.int16, device=dev)
    slot = torch.arange(sh.B, dtype=torch.int32, device=dev)
    ws = sv.new_workspace(B, K, V, dev)
    out = sv.VerifyOutputs(B, K, dev)

    def step(i):
        logits, q, x, params, seed = sets[i % N_SETS]
        sv.spec_verify(logits, q, x, params, seed, out=out, workspace=ws)
        sv.spec_commit(vrec, vconv, out.accept_len, slot, crec, cconv, out.flags)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()

    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # a ~1 ms spin on the stream before the timed region lets the host
        # queue the first steps ahead of the device, so no step's interval
        # holds host launch latency
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(2_000_000)
        start.record(stream)
        for i in range(n):
            logits, q, x, params, seed = sets[i % N_SETS]
            ev[i][0].record(stream)
            sv.spec_verify(logits, q, x, params, seed, out=out, workspace=ws)
            ev[i][1].record(stream)
            sv.spec_commit(vrec, vconv, out.accept_len, slot, crec, cconv, out.flags)
            ev[i][2].record(stream)
        end.record(stream)
        while not end.query():   # short sleeps: the clock sampler thread runs meanwhile
            time.sleep(0.0005)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = max_over_ranks(start.elapsed_time(end), world)
    t_verify = [ev[i][0].elapsed_time(ev[i][1]) for i in range(n)]
    t_commit = [ev[i][1].elapsed_time(ev[i][2]) for i in range(n)]
    acc = out.accept_len.cpu().numpy()

    # ---- end to end through the public API with host buffers ----
    pin = lambda t: t.cpu().pin_memory()
    h_sets = [(pin(s[0]), pin(s[1]), pin(s[2]), pin(s[3]), s[4]) for s in sets]
    h_vrec, h_vconv = pin(vrec), pin(vconv)
    d_out = {k: torch.empty_like(getattr(out, k), device="cpu").pin_memory()
             for k in ("tokens", "accept_len", "logprobs", "alpha", "flags")}
    e2e_steps = max(3, min(n, 10))
    h2d = sum(t.numel() * t.element_size() for t in h_sets[0][:4]) + \
        h_vrec.numel() * 4 + h_vconv.numel() * 2
    d2h = sum(t.numel() * t.element_size() for t in d_out.values())
    dl, dq, dx, dp = (torch.empty_like(t) for t in sets[0][:4])

    def e2e_step(i):
        hl, hq, hx, hp, seed = h_sets[i % N_SETS]
        dl.copy_(hl, non_blocking=True)
        dq.copy_(hq, non_blocking=True)
        dx.copy_(hx, non_blocking=True)
        dp.copy_(hp, non_blocking=True)
        vrec.copy_(h_vrec, non_blocking=True)
        vconv.copy_(h_vconv, non_blocking=True)
        sv.spec_verify(dl, dq, dx, dp, seed, out=out, workspace=ws)
        sv.spec_commit(vrec, vconv, out.accept_len, slot, crec, cconv, out.flags)
        for k_, t in d_out.items():
            t.copy_(getattr(out, k_), non_blocking=True)
        torch.cuda.current_stream().synchronize()

    e2e_step(0)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        e2e_step(i)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peaks()
    vbytes = statistics.mean(verify_algorithmic_bytes(inp) for inp in inps)
    cbytes = sh.bytes_moved(int(np.count_nonzero(acc > 0)))
    tv = statistics.mean(t_verify) * 1e-3
    tc = statistics.mean(t_commit) * 1e-3
    v_hash = kernel_source_hash(VERIFY_SOURCES)
    c_hash = kernel_source_hash(["spec_commit.cu"])

    def roof(name, nbytes, t, h):
        ach = nbytes / t / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": peak,
                "unit": "GB/s", "frac": round(ach / peak, 4), "peak_source": peak_kind,
                "traffic": traffic_record(name, h), "algorithmic_bytes": int(nbytes),
                "avg_us": round(t * 1e6, 2)}

    r_commit = roof("commit_kernel", cbytes, tc, c_hash)
    r_verify = roof("spec_verify", vbytes, tv, v_hash)
    dominant = r_commit if tc >= tv else r_verify
    value = job_rows_per_s(B * n, world, elapsed_ms * 1e-3)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world,
        "steps": n, "warmup": max(args.warmup, 3), "ms_per_step": round(elapsed_ms / n, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "verify 64 rows k=2 V=151936 bf16 mixed params (25% greedy, "
                               "50% T0.7 top-k50 top-p0.9, 25% T1) + commit 24 layers x 64 rows "
                               "(16x128x128 fp32 + 4x4096 bf16 per layer, 3 states)",
                   "l2": f"verify inputs rotate over {N_SETS} sets of 136 MB; commit reads a 4.98 GB buffer",
                   "parallelism": f"rows sharded per GPU (dp{world})"},
        "clocks": clk.summary(),
        "e2e": {"value": round(B * world * e2e_steps / e2e_s, 1), "unit": "rows/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": (VERIFY_LAUNCHES + 1) * n,
        "roofline": dominant,
        "roofline_verify": r_verify,
        "components": {
            "spec_verify": {"us": round(tv * 1e6, 2), "rows_per_s": round(B / tv, 1),
                            "gbs": r_verify["achieved"], "frac": r_verify["frac"],
                            "dense_q_model_bytes": int(inps[0].logits.size * 2 + inps[0].q.size * 4),
                            "us_p50": round(statistics.median(t_verify) * 1e3, 2),
                            "us_max": round(max(t_verify) * 1e3, 2)},
            "spec_commit": {"us": round(tc * 1e6, 2), "gbs": r_commit["achieved"], "frac": r_commit["frac"],
                            "us_p50": round(statistics.median(t_commit) * 1e3, 2),
                            "us_max": round(max(t_commit) * 1e3, 2)},
            "mean_accept_len": float(acc.mean()),
        },
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(inps[0])
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_only(args):
    """Launch one kernel per step on the benchmark workload (for ncu captures)."""
    import torch

    from speculative_decoding_verify_07_gb300 import binding as sv
    from speculative_decoding_verify_07_gb300 import synth

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    if args.only == "verify":
        sets = []
        for i in range(N_SETS):
            inp = synth.make_mixed(seed_offset=100 * i)
            sets.append((torch.from_numpy(inp.logits).to(torch.bfloat16).to(dev),
                         torch.from_numpy(inp.q).to(dev), torch.from_numpy(inp.drafts).to(dev),
                         sv.make_params(inp.temperature, inp.top_k, inp.top_p, dev), inp.seed + i))
        ws = sv.new_workspace(B, K, V, dev)
        out = sv.VerifyOutputs(B, K, dev)
        fn = lambda i: sv.spec_verify(*sets[i % N_SETS][:4], sets[i % N_SETS][4], out=out, workspace=ws)
    else:
        sh = synth.CommitShape(L=args.layers)
        vrec = torch.zeros((sh.L, sh.B, sh.S, sh.H, sh.Dk, sh.Dv), dtype=torch.float32, device=dev)
        vconv = torch.zeros((sh.L, sh.B, sh.S, sh.W, sh.C), dtype=torch.int16, device=dev)
        crec = torch.zeros((sh.L, sh.slots, sh.H, sh.Dk, sh.Dv), dtype=torch.float32, device=dev)
        cconv = torch.zeros((sh.L, sh.slots, sh.W, sh.C), dtype=torch.int16, device=dev)
        acc = torch.from_numpy(synth.commit_indices(sh)[0]).to(dev)
        slot = torch.arange(sh.B, dtype=torch.int32, device=dev)
        fn = lambda i: sv.spec_commit(vrec, vconv, acc, slot, crec, cconv)
    for i in range(max(args.warmup, 3)):
        fn(i)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][0].record()
        fn(i)
        ev[i][1].record()
    torch.cuda.synchronize()
    t = [a.elapsed_time(b) * 1e3 for a, b in ev]
    print(json.dumps({"only": args.only, "steps": args.steps, "mean_us": statistics.mean(t),
                      "median_us": statistics.median(t), "min_us": min(t)}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["verify", "commit"], default=None,
                    help="profiling aid: launch only one kernel per step, print its mean time")
    ap.add_argument("--layers", type=int, default=24, help="profiling aid for --only commit")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
