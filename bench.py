#!/usr/bin/env python3
"""Throughput of batched speculative-sampling verification on GB300.

One step = one spec_verify_sample call (plan kernel + persistent verify kernel) over
one synthetic round of the headline workload: B = 64 requests, gamma = 7,
V = 151936 bf16 logits, full-q verification with the SpecKV draft signals.
The metric is verify rounds/s (whole job, all ranks); the roofline is the HBM
bandwidth of the verify kernel on the bytes the method must read.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 is launched by torchrun: every rank verifies its own request batches
(requests are independent, so the work shards with no data-path exchange:
weak scaling); rank 0 prints one JSON line with the max time over ranks.
--impl reference times the fp64 CPU oracle on the same workload instead.
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

from speculative_decoding_verification_26_gb300 import workloads as W  # noqa: E402

METRIC = "verify rounds/s and HBM GB/s (% of 8 TB/s) at B=64, gamma=7, V=151936 bf16"
UNIT = "rounds/s"
WORKLOAD = "m"
# The headline workload is m; --workload times the other configurations of
# the same seeded generator with the same contract (call kind per config).
WORKLOADS = {
    "m": ("sample", "B=64 gamma=7 V=151936 bf16, full-q stochastic verify + draft signals; T=0.7, "
                    "target N(0,3^2)+Zipf(1.1) bias, draft = target + N(0,1.5^2), y ~ q"),
    "c2": ("greedy", "B=64 gamma=7 V=151936 bf16, greedy verify; target N(0,3^2)+Zipf(1.1) bias, "
                     "y = argmax replaced w.p. 0.3 by a uniform token"),
    "c3": ("sample", "B=32 gamma=4 V=128256 bf16, full-q stochastic verify + draft signals; T=0.7, "
                     "draft = target + N(0,1.5^2), y ~ q"),
    "c4": ("onehot", "B=64 gamma=8 V=151936 bf16, one-hot q verify; T=1, y = argmax(target + N(0,2^2))"),
    "c5": ("sample", "B=256 gamma_b in {2,4,6,8} (G=8) V=151936 bf16, full-q stochastic verify + draft signals; "
                     "T=0.6, draft = target + N(0,1), y ~ q"),
}
WORKLOAD_DESC = WORKLOADS[WORKLOAD][1]
L2_BYTES = 129 * 2**20


# ----------------------------------------------------------------------------
# multi-rank plumbing (also exercised by the gloo tests on CPU)

def rank_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity for one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_rate(units_all_ranks: float, t_max_s: float) -> float:
    return units_all_ranks / t_max_s if t_max_s > 0 else 0.0


def rank_round_index(rank: int, s: int) -> int:
    """Seed index of input set s on `rank`: every rank verifies its own requests."""
    return 1000 * rank + s


# ----------------------------------------------------------------------------
# clocks during the timed region

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# our arm

def source_sha() -> str:
    h = hashlib.sha256()
    for rel in ("speculative_decoding_verification_26_gb300/csrc/verify.cu",
                "speculative_decoding_verification_26_gb300/csrc/common.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes of the verify kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "verify_kernel_b64_g7_v151936_traffic.txt")
    try:
        with open(path) as f:
            d = json.loads(f.read().split("\n---\n")[0])
    except (OSError, ValueError):
        return None
    if d.get("source_sha") != source_sha():
        return None
    return d.get("dram_bytes_per_launch")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def build_inputs(dev, rank, nsets, sv, torch):
    """Seeded input sets resident on the device.  Draft tokens come from the
    workload's stand-in drafter (the same tokens the reference arm uses); the
    argmax drafters of the greedy and one-hot configurations use torch's
    argmax (lowest index on ties)."""
    def bf16_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def argmax_rows(rows):
        x = bf16_dev(rows).float() if rows.dtype == np.uint16 else torch.from_numpy(rows).to(dev)
        return x.argmax(dim=-1).int().cpu().numpy()

    sets = []
    for s in range(nsets):
        wl = W.make(WORKLOAD, rank_round_index(rank, s))
        W.resolve_draft_tokens(wl, argmax_rows)
        sets.append(dict(target=bf16_dev(wl.target), draft=bf16_dev(wl.draft) if wl.draft is not None else None,
                         tokens=torch.from_numpy(wl.draft_tokens).to(dev), gamma=torch.from_numpy(wl.gamma).to(dev),
                         temperature=torch.from_numpy(wl.temperature).to(dev),
                         uniforms=torch.from_numpy(wl.uniforms).to(dev), host=wl))
    return sets


def all_rows_bytes(wl, mode):
    """Bytes of every valid logit row of one round, each read once."""
    gam = wl.gamma.astype(np.int64)
    rows = ((2 * gam + 1) if mode == "sample" else (gam + 1)).sum()
    return int(rows) * wl.V * wl.elem_bytes


def config_dict(wl, world, nsets, F_bytes):
    """The `config` of the JSON line, identical for both arms."""
    return {"workload": WORKLOAD_DESC, "B": wl.B, "gamma": wl.G, "V": wl.V,
            "l2": f"{nsets} rotating input sets of {F_bytes/1e6:.0f} MB ({nsets*F_bytes/1e9:.2f} GB > 4x L2)",
            "parallelism": f"{world} independent request shards, no collective"}


def run_ours(args):
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    rank, world, local = rank_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    L = sv.lib()
    stream = torch.cuda.current_stream(dev)
    sets = build_inputs(dev, rank, args.sets, sv, torch)
    B, G, V = sets[0]["host"].B, sets[0]["host"].G, sets[0]["host"].V
    ws = torch.empty(sv.workspace_bytes(B, G, V), dtype=torch.uint8, device=dev)
    mode = WORKLOADS[WORKLOAD][0]
    out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
               tokens=torch.empty(B, G + 1, dtype=torch.int32, device=dev),
               status=torch.empty(B, dtype=torch.int32, device=dev))
    if mode == "sample":
        out["signals"] = torch.empty(B, 4, dtype=torch.float32, device=dev)

    def call(s):
        if mode == "greedy":
            return sv.verify_greedy(s["target"], s["tokens"], s["gamma"], ws=ws, out=out)
        if mode == "onehot":
            return sv.verify_onehot(s["target"], s["tokens"], s["gamma"], s["temperature"], s["uniforms"],
                                    ws=ws, out=out)
        return sv.verify_sample(s["target"], s["draft"], s["tokens"], s["gamma"], s["temperature"], s["uniforms"],
                                signals=True, ws=ws, out=out)

    def step(k):
        return call(sets[k % len(sets)])

    # per-set outcome (accept lengths) -> committed tokens and algorithmic bytes
    rows_needed, committed = [], []
    for k in range(len(sets)):
        r = step(k)
        torch.cuda.synchronize()
        kk = r["accept_len"].cpu().numpy().astype(np.int64)
        gam = sets[k]["host"].gamma.astype(np.int64)
        # target rows 0..k, and with the signals every draft row
        rows_needed.append(int(np.sum(kk + 1) + (np.sum(gam) if mode == "sample" else 0)))
        committed.append(int(np.sum(kk + 1)))
        # no request may fail (SPEC_ST_GUARDED and SPEC_ST_ZERO_RESIDUAL are informational)
        assert int((r["status"] & ~(sv._lib.ST_GUARDED | sv._lib.ST_ZERO_RESIDUAL)).abs().sum()) == 0
    es = 2
    F_bytes = all_rows_bytes(sets[0]["host"], mode)

    # warm-up (at least W calls and ~0.5 s so clocks settle)
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid is not None else local)
    sampler.start()
    t0 = time.time()
    n = 0
    while n < args.warmup or time.time() - t0 < args.min_warmup_s:
        step(n)
        n += 1
    torch.cuda.synchronize()

    # The K timed steps are replayed from captured CUDA graphs: a step is one
    # library call (its kernels, as launched by the C ABI), and replaying a
    # graph removes the Python/ctypes launch overhead from the timing.
    K = args.steps
    per_graph = 4 * len(sets)
    lc0 = sv.launch_count()
    step(0)
    torch.cuda.synchronize()
    per_call = sv.launch_count() - lc0                  # kernels per call
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    g_big, g_one = torch.cuda.CUDAGraph(), []
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_big, stream=side):
            for k in range(per_graph):
                step(k)
        for k in range(len(sets)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                step(k)
            g_one.append(g)
    stream.wait_stream(side)
    for _ in range(3):
        g_big.replay()
    torch.cuda.synchronize()
    n_full, rem = divmod(K, per_graph)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_full):
        g_big.replay()
    for j in range(rem):
        g_one[(n_full * per_graph + j) % len(sets)].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    launches = per_call * K
    t_local = e0.elapsed_time(e1) / 1e3
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    t_max = max_over_ranks(t_local, world, dev)
    rounds_all = sum_over_ranks(float(K), world, dev)
    value = job_rate(rounds_all, t_max)

    # verify-kernel duration, live, with events around that kernel only
    nprof = min(K, 200)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nprof)]
    for a, b in evs:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for k in range(nprof):
        sv.profile_next_call(*evs[k])
        step(k)
    torch.cuda.synchronize()
    t_kern = statistics.mean(a.elapsed_time(b) for a, b in evs) / 1e3
    nsets = len(sets)
    N_bytes = statistics.mean(rows_needed[k % nsets] for k in range(nprof)) * V * es
    hbm_peak, peak_kind = peaks()
    achieved = N_bytes / t_kern / 1e9
    traffic = profiled_traffic()

    # end to end: pinned host inputs -> device, call, results -> host, every step
    e2e = None
    if not args.no_e2e:
        host = []
        for s in sets:
            h = {}
            keys = {"greedy": ("target", "tokens", "gamma"),
                    "onehot": ("target", "tokens", "gamma", "temperature", "uniforms")}.get(
                mode, ("target", "draft", "tokens", "gamma", "temperature", "uniforms"))
            for key in keys:
                h[key] = torch.empty_like(s[key], device="cpu").pin_memory()
                h[key].copy_(s[key])
            host.append(h)
        # two device input buffers: the inputs of step k+1 cross the host link
        # (on a copy stream) while step k's call and result readback run
        dbufs = [{key: torch.empty_like(sets[0][key]) for key in host[0]} for _ in range(2)]
        hout = {key: torch.empty_like(v, device="cpu").pin_memory() for key, v in out.items()}
        h2d = sum(v.numel() * v.element_size() for v in host[0].values())
        d2h = sum(v.numel() * v.element_size() for v in hout.values())
        Ke = min(K, args.e2e_steps)
        copy_stream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]

        def h2d_copy(k):
            j = k % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(consumed[j])       # step k-2 is done with this buffer
                h = host[k % len(host)]
                for key in h:
                    dbufs[j][key].copy_(h[key], non_blocking=True)
                copied[j].record(copy_stream)

        def e2e_run(k0, n):
            """Steps k0 .. k0+n-1; each step's inputs go host -> device and its
            results device -> host inside the run."""
            copy_stream.wait_stream(stream)     # no copy starts before the run does
            h2d_copy(k0)
            for k in range(k0, k0 + n):
                j = k % 2
                if k + 1 < k0 + n:
                    h2d_copy(k + 1)
                stream.wait_event(copied[j])
                r = call(dbufs[j])
                consumed[j].record(stream)
                for key in hout:
                    hout[key].copy_(r[key], non_blocking=True)
            stream.synchronize()
        e2e_run(0, 3)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_run(0, Ke)
        b.record(stream)
        torch.cuda.synchronize()
        te = max_over_ranks(a.elapsed_time(b) / 1e3, world, dev)
        e2e = {"value": job_rate(sum_over_ranks(float(Ke), world, dev), te), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": Ke}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(sets[0]["host"], args.cpu_seconds, mode)

    if rank == 0:
        mean_committed = statistics.mean(committed)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": t_max / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": config_dict(sets[0]["host"], world, nsets, F_bytes),
            "roofline": {"bound": "hbm", "kernel": "verify_kernel", "achieved": achieved, "peak": hbm_peak,
                         "unit": "GB/s", "frac": achieved / hbm_peak, "peak_kind": peak_kind,
                         "frac_label": f"of {peak_kind} peak ({hbm_peak:.0f} GB/s copy bandwidth)",
                         "frac_of_8tbs": achieved / 8000.0, "target_frac": 0.70,
                         "traffic": traffic,
                         "dram_gbs": (traffic / t_kern / 1e9) if traffic else None,
                         "algorithmic_bytes_per_launch": N_bytes,
                         "kernel_ms": t_kern * 1e3},
            "gpu_launches": int(launches),
            "clocks": clocks,
            "tokens_per_s": value * mean_committed,
            "committed_tokens_per_round": mean_committed,
            "hbm_gbs_step": N_bytes * value / world / 1e9,
            "all_rows_bytes": F_bytes,
            "needed_bytes_mean": N_bytes,
            "rounds_per_s_at_peak_all_rows": hbm_peak * 1e9 / F_bytes,
            "rounds_per_s_at_peak_needed_rows": hbm_peak * 1e9 / N_bytes,
        }
        if e2e:
            line["e2e"] = e2e
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# the oracle on the host cores

def oracle_round(o, wl, mode, idx, cores):
    """The fp64 oracle on requests `idx` of one round (OpenMP over requests)."""
    if mode == "greedy":
        o.verify_greedy(wl.target[idx], wl.draft_tokens[idx], wl.gamma[idx], nthreads=cores)
    elif mode == "onehot":
        o.verify_onehot(wl.target[idx], wl.draft_tokens[idx], wl.gamma[idx], wl.temperature[idx], wl.uniforms[idx],
                        nthreads=cores)
    else:
        o.verify_sample(wl.target[idx], wl.draft[idx], wl.draft_tokens[idx], wl.gamma[idx], wl.temperature[idx],
                        wl.uniforms[idx], want_signals=True, nthreads=cores)


def cpu_baseline(wl, seconds, mode="sample"):
    """The fp64 oracle (test infrastructure, as it stands) on full rounds of the
    same workload, repeated on one input set for about `seconds` of wall time."""
    import oracle
    o = oracle.load()
    cores = os.cpu_count() or 1
    idx = np.arange(wl.B)
    t0 = time.perf_counter()
    n = 0
    while n < 1 or time.perf_counter() - t0 < seconds:
        oracle_round(o, wl, mode, idx, cores)
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} full rounds (B={wl.B} requests each) of one input set, {dt:.1f} s, "
                      f"OpenMP over requests on {cores} threads"}


def run_reference(args):
    """The reference arm: the fp64 oracle, as it stands, on the host cores, on
    the same input sets, draft tokens, metric and config as our arm.  A step
    verifies `per_step` requests of the rotating rounds (a full round when K
    rounds fit in about a minute, else a divisor of B sized so they do); the
    requests of consecutive steps are verified a round at a time (one oracle
    call, OpenMP over that round's requests), so a step of a few requests
    costs what it costs inside a full round."""
    rank, world, _ = rank_env()
    if rank != 0:
        return
    import oracle
    o = oracle.load()
    cores = os.cpu_count() or 1
    mode = WORKLOADS[WORKLOAD][0]

    def argmax_rows(rows):
        return o.run(oracle.GREEDY, target=np.ascontiguousarray(rows)[:, None, :], G=0)["tokens"][:, 0]

    sets = []
    for s in range(args.sets):
        wl = W.make(WORKLOAD, rank_round_index(0, s))
        W.resolve_draft_tokens(wl, argmax_rows)
        sets.append(wl)
    B = sets[0].B
    t0 = time.perf_counter()
    oracle_round(o, sets[0], mode, np.arange(B), cores)          # one round: size the steps
    t_round = time.perf_counter() - t0
    budget_s = args.ref_seconds
    divisors = [d for d in range(1, B + 1) if B % d == 0]
    per_step = max([d for d in divisors if args.steps * t_round * d / B <= budget_s] or [1])

    def run_steps(k0, n):
        """Steps k0 .. k0+n-1: their requests, a round (input set) at a time."""
        r0, r1 = k0 * per_step, (k0 + n) * per_step             # request counter range
        while r0 < r1:
            rnd, off = divmod(r0, B)
            m = min(B - off, r1 - r0)
            oracle_round(o, sets[rnd % len(sets)], mode, np.arange(off, off + m), cores)
            r0 += m
    run_steps(0, max(args.warmup, 1))
    t0 = time.perf_counter()
    run_steps(args.warmup, args.steps)
    dt = time.perf_counter() - t0
    rounds = args.steps * per_step / B
    value = rounds / dt
    F_bytes = all_rows_bytes(sets[0], mode)
    sample = (f"each step: {per_step} of the {B} requests of a round (fp64 oracle); the {args.steps} timed steps "
              f"({rounds:g} rounds of {len(sets)} rotating input sets) run a round's requests per call, "
              f"OpenMP over requests on {cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(sets[0], world, len(sets), F_bytes),
            "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": sample, "value": value, "unit": UNIT},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# the calls beside the verification, timed on the headline shapes

def run_op(args):
    """--op divergence|filter|gamma: one JSON line per case, not the headline.
    CUDA events on the current stream, inputs resident in HBM; divergence
    rotates --sets input sets (L2 flush by footprint); filter restores its rows
    between calls outside the timed events (the call filters in place)."""
    import torch

    import speculative_decoding_verification_26_gb300 as sv
    sv.lib()
    dev = torch.device("cuda:0")
    peak, peak_kind = peaks()
    steps, warm = min(args.steps, 400), max(args.warmup, 3)

    def bf16_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def emit(case, us, algo_bytes, extra):
        gbs = algo_bytes / (us * 1e-6) / 1e9 if algo_bytes else None
        line = {"op": args.op, "case": case, "metric": f"{args.op} us per call", "value": round(us, 2),
                "unit": "us", "higher_is_better": False, "steps": steps, "warmup": warm,
                "algorithmic_bytes": algo_bytes, "achieved_gbs": round(gbs, 1) if gbs else None,
                "frac": round(gbs / peak, 4) if gbs else None, "frac_label": f"of {peak_kind} {peak:.1f} GB/s",
                "data": "synthetic", **extra}
        print(json.dumps(line), flush=True)

    if args.op == "divergence":
        sets = []
        for k in range(args.sets):
            wl = W.make("m", k)
            sets.append((bf16_dev(wl.target), bf16_dev(wl.draft), torch.from_numpy(wl.gamma).to(dev),
                         torch.from_numpy(wl.temperature).to(dev)))
        pairs = int(wl.gamma.sum())
        for i in range(warm):
            sv.divergence_stats(*sets[i % len(sets)])
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            sv.divergence_stats(*sets[i % len(sets)])
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / steps
        emit("b64_g7_v151936", us, pairs * 2 * wl.V * 2,
             {"config": {"workload": "divergence statistics of 64 requests, gamma 7, V 151936 bf16",
                         "pairs": pairs, "l2": f"{args.sets} rotating input sets"}})
    elif args.op == "filter":
        wl = W.make("m", 0)
        base = bf16_dev(wl.target).reshape(-1, wl.V)
        n = base.shape[0]
        work = base.clone()
        T = torch.full((n,), 0.7, dtype=torch.float32, device=dev)
        for case, k, p in (("top_k50", 50, None), ("top_p0.9", None, 0.9), ("top_k50_top_p0.9", 50, 0.9)):
            kt = None if k is None else torch.full((n,), k, dtype=torch.int32, device=dev)
            pt = None if p is None else torch.full((n,), p, dtype=torch.float32, device=dev)
            for _ in range(warm):
                work.copy_(base)
                sv.filter_top_k_top_p(work, kt, pt, T)
            torch.cuda.synchronize()
            changed = int((work.view(torch.int16).reshape(n, -1, 8) != base.view(torch.int16).reshape(n, -1, 8))
                          .any(-1).sum())
            tot = 0.0
            for _ in range(steps):
                work.copy_(base)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                sv.filter_top_k_top_p(work, kt, pt, T)
                e1.record()
                torch.cuda.synchronize()
                tot += e0.elapsed_time(e1)
            kept = int(torch.isfinite(work.float()).sum())
            emit(case, tot * 1e3 / steps, n * wl.V * 2 + changed * 16,
                 {"config": {"workload": f"top-k/top-p filtering of {n} rows of V {wl.V} bf16 at T 0.7",
                             "rows": n, "kept_per_row": round(kept / n, 2), "changed_16B_vectors": changed}})
    else:
        for B in (64, 4096):
            g = torch.Generator().manual_seed(B)
            sig = torch.rand(B, 4, generator=g).to(dev)
            model = (torch.randn(141, generator=g) * 0.3).to(dev)
            model[6:12] = 1.0                                  # standard deviations
            for _ in range(warm):
                sv.gamma_select(sig, model)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                sv.gamma_select(sig, model)
            e1.record()
            torch.cuda.synchronize()
            emit(f"b{B}", e0.elapsed_time(e1) * 1e3 / steps, None,
                 {"config": {"workload": f"SpecKV gamma selector, {B} requests", "B": B}})


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sets", type=int, default=4, help="rotating input sets (L2 flush by footprint)")
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="reference arm: size its steps so the timed ones take about this long")
    ap.add_argument("--min-warmup-s", type=float, default=0.5, help="keep warming up at least this long")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--op", choices=["verify", "divergence", "filter", "gamma"], default="verify",
                    help="verify (default) is the headline step; the others time the calls beside it")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="m",
                    help="m (default) is the headline; c2..c5 time the other configurations")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    global WORKLOAD, WORKLOAD_DESC, METRIC
    WORKLOAD = args.workload
    WORKLOAD_DESC = WORKLOADS[WORKLOAD][1]
    if WORKLOAD != "m":
        c = W.CONFIGS[WORKLOAD]
        METRIC = (f"verify rounds/s and HBM GB/s (% of 8 TB/s) at B={c['B']}, gamma={c['G']}, V={c['V']} bf16, "
                  f"{WORKLOADS[WORKLOAD][0]}")
    if args.op != "verify":
        run_op(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
