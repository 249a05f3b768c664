#!/usr/bin/env python
"""Benchmark of the GB300 verify step.

One step = one pass of the whole verify path (statistics, c* labels, accept
test, first-rejection cut, replacement / bonus draw) over one batch of the
synthetic workload, inputs resident in HBM: one launch of the rows kernel,
which finishes the requests in its tail (filtered workloads: the row kernel
and the request kernel).
Default workload: B = 32 requests, block 16 (15 drafted positions + bonus),
V = 151,936, bf16 logits, T = 1 sampling with labels -- the workload on which
the 70%-of-HBM goal is stated.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and torch.cuda.synchronize(); CUDA events on the launch stream.  Two copies of
the inputs (2 x 301 MB, each larger than the 129 MB L2) alternate between
steps.  The step's launch (filtered: the row kernel) is additionally
bracketed by events each step to give its own duration for the roofline.
Multi-GPU: one process per GPU, each
verifying its own independent batch (requests are independent units; no
collective on the data path), time = max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload I] [--mode sample|greedy]

After the headline line's own workload, the same line carries
``per_workload``: every one of the five synthetic workloads in each of its
modes, timed the same way (inputs larger than L2 alternate; smaller ones
get an L2 flush before each step, outside the step's events), with the
dominant kernel's HBM fraction and the oracle's check of one call on a
sample of requests (near ties, open accept chains, mismatches).

--component schedule prints one line for the DSpark prefix scheduler instead
(spec_verify_schedule on a pool of 256 requests x 15 positions whose
confidences are the verify step's own labels on the ragged workload; the
SPS curve is synthetic: flat to 1,024 tokens, then falling as 1/B), with the
fp64 oracle timed beside it.

--component split prints one line for the vocabulary-split verify
(include/spec_verify_shard.h) on the same workload: the columns of every row
split over --split-world ranks whose steps run in lockstep on this one GPU
(the all-gathers are stacks in rank order), each phase timed with CUDA
events and divided by the number of ranks to give one rank's time, L2
flushed before both passes over the logits (the statistics pass and the
masses pass).
"""

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from speculative_decoding_verification_16_gb300 import workloads as W  # noqa: E402

PKG = os.path.join(ROOT, "speculative_decoding_verification_16_gb300")
FALLBACK_HBM_GBS = 6800.0
METRIC = "verified draft positions/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "draft positions/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--mode", choices=("sample", "greedy"), default="sample")
    ap.add_argument("--requests", type=int, default=0,
                    help="run the workload with this many requests instead of its own B "
                         "(small cases for profiling; the timed default keeps B)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the per-workload lines (all five workloads in their modes)")
    ap.add_argument("--component", choices=("verify", "schedule", "split"), default="verify")
    ap.add_argument("--split-world", type=int, default=8,
                    help="--component split: ranks the vocabulary is split over")
    ap.add_argument("--top-k", type=int, default=None, help="override the workload's top_k")
    ap.add_argument("--top-p", type=float, default=None, help="override the workload's top_p")
    return ap.parse_args()


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------- clocks
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index):
        self.proc = None
        self.path = os.path.join("/tmp", f"sv_clocks_{os.getpid()}.csv")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)], stdout=self.fh, stderr=subprocess.DEVNULL)
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
        self.fh.close()
        sm, smax, reasons = [], [], set()
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(REASONS, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------- roofline inputs
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return float(json.load(open(path))["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Source files that make up each kernel whose DRAM traffic is recorded under
# profiles/ (the kernel's own header, the headers it includes, the launch code).
KERNEL_SOURCES = {
    "rows_kernel": ["csrc/sv_rows.cuh", "csrc/sv_finalize.cuh", "csrc/sv_common.cuh",
                    "csrc/sv_ptx.cuh", "csrc/spec_verify.cu", "../include/spec_verify.h"],
    "filter_rows_kernel": ["csrc/sv_filter.cuh", "csrc/sv_common.cuh", "csrc/sv_ptx.cuh",
                           "csrc/spec_verify.cu", "../include/spec_verify.h"],
    "gfilter_rows_kernel": ["csrc/sv_gfilter.cuh", "csrc/sv_filter.cuh", "csrc/sv_common.cuh",
                            "csrc/sv_ptx.cuh", "csrc/spec_verify.cu", "../include/spec_verify.h"],
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(PKG, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload_name):
    """DRAM bytes per launch of ``kernel`` on the workload from the committed
    ncu summary, or None when that kernel's sources changed since the
    capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    ent = rec.get(f"{kernel}/{workload_name}")
    if not ent or ent.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


# --------------------------------------------------------------------- oracle (CPU legs)
def oracle_rate(w, spec, mode, budget_s, ell_cap=None, start=0, top_k=None, top_p=None):
    """Time the fp64 oracle on requests of ``w`` -- each cut to at most
    ``ell_cap`` target rows (a shorter request is itself a valid verify
    problem) -- until ``budget_s`` of oracle time has elapsed (at least one
    request).  Rows are copied to the host outside the timing.  Returns
    (draft positions/s, positions, seconds, requests)."""
    import oracle
    lens = w.verify_lens.cpu().numpy()
    offs = w.row_offsets.cpu().numpy()
    dt = W.dtype_name(w.target)
    pos, secs, nreq, r = 0, 0.0, 0, start
    while nreq == 0 or secs < budget_s:
        rr = r % w.B
        r += 1
        off, ell = int(offs[rr]), int(lens[rr])
        if ell_cap is not None:
            ell = min(ell, ell_cap)
        if ell < 2:
            continue
        doff = off - rr
        t = W.bits_of(w.target[off:off + ell])
        d = W.bits_of(w.draft[doff:doff + ell - 1])
        x = w.draft_tokens[doff:doff + ell - 1].cpu().numpy()
        u = w.uniforms[off:off + ell].double().cpu().numpy()
        t0 = time.perf_counter()
        oracle.verify_request(oracle.decode_logits(t, dt),
                              oracle.decode_logits(d, dt).reshape(ell - 1, -1), x, u,
                              spec.temperature, spec.top_k if top_k is None else top_k,
                              spec.top_p if top_p is None else top_p, mode, want_conf=True)
        secs += time.perf_counter() - t0
        pos += ell - 1
        nreq += 1
    return pos / secs, pos, secs, nreq


def oracle_check(w, out, spec, mode, top_k, top_p, budget_s, seed=0):
    """The fp64 oracle on a seeded sample of the workload's requests (whole
    requests, at least one, until ``budget_s`` of oracle time): its rate, and
    how the library's outputs of one call compare with it -- requests with a
    decision margin below 1e-6 (near ties), requests whose accept chain such
    a margin leaves open (not compared), final tokens checked against a set
    of admissible tokens, and mismatches (must be 0)."""
    import numpy as np

    import oracle
    lens = w.verify_lens.cpu().numpy()
    offs = w.row_offsets.cpu().numpy()
    toks = out.tokens.cpu().numpy()
    acc = out.accept_len.cpu().numpy()
    dt = W.dtype_name(w.target)
    order = np.random.default_rng(seed).permutation(w.B)
    c = {"requests": 0, "positions": 0, "near_tie": 0, "open": 0, "final_sets": 0,
         "mismatches": 0}
    secs = 0.0
    for r in order:
        if c["requests"] and secs >= budget_s:
            break
        off, ell = int(offs[r]), int(lens[r])
        doff = off - r
        t = oracle.decode_logits(W.bits_of(w.target[off:off + ell]), dt)
        d = oracle.decode_logits(W.bits_of(w.draft[doff:doff + ell - 1]), dt).reshape(ell - 1, w.V)
        x = w.draft_tokens[doff:doff + ell - 1].cpu().numpy()
        u = w.uniforms[off:off + ell].double().cpu().numpy()
        t0 = time.perf_counter()
        ex = oracle.verify_request(t, d, x, u, spec.temperature, top_k, top_p, mode)
        secs += time.perf_counter() - t0
        adm = oracle.admissible_outcomes(t, d, x, u, spec.temperature, top_k, top_p, mode)
        c["requests"] += 1
        c["positions"] += ell - 1
        c["near_tie"] += bool(ex["near_tie"])
        if not adm["determined"]:
            c["open"] += 1
            continue
        a = adm["accept_len"]
        got = toks[off:off + ell].tolist()
        ok = (acc[r] == a and got[:a] == ex["tokens"][:a].tolist() and got[a] in adm["finals"]
              and all(v == -1 for v in got[a + 1:]))
        c["mismatches"] += not ok
        c["final_sets"] += len(adm["finals"]) > 1
    rate = c["positions"] / secs if secs > 0 else None
    return c, rate, secs


def run_reference(args, world, rank):
    """Reference arm: the CPU oracle, as it stands, on this host's cores."""
    if rank != 0:
        return
    spec = W.WORKLOADS[args.workload]
    mode = W.SAMPLE if args.mode == "sample" else W.GREEDY
    w = W.make_workload(spec, mode, seed=1000 * args.workload, device="cpu")
    # size each step so that the whole run stays within about two minutes
    per_step = max(0.0, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    _, pos1, sec1, _ = oracle_rate(w, spec, mode, 0.0)
    t_pos = sec1 / pos1  # oracle seconds per drafted position (2 rows each)
    ell_cap = max(2, min(spec.max_len, int(per_step / t_pos) + 1))
    tot_pos, tot_sec, nreq_all = 0, 0.0, 0
    for i in range(args.warmup + args.steps):
        _, pos, sec, nreq = oracle_rate(w, spec, mode, per_step, ell_cap, start=i)
        if i >= args.warmup:
            tot_pos += pos
            tot_sec += sec
            nreq_all += nreq
    value = tot_pos / tot_sec
    sample = (f"{args.steps} timed steps over {nreq_all} requests of the {spec.name} workload "
              f"cut to <= {ell_cap} target rows each, >= {per_step * 1e3:.0f} ms of "
              f"single-thread fp64 oracle time per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_sec / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.name, "B": spec.B, "block": spec.max_len, "V": spec.V,
                   "logits": spec.dtype, "mode": args.mode, "temperature": spec.temperature,
                   "top_k": spec.top_k, "top_p": spec.top_p},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours
L2_BYTES = 129 * 1024 * 1024


def row_kernel_name(top_k, top_p, V):
    """The launch that streams the logits (the dominant kernel)."""
    if not ((0 < top_k < V) or top_p < 1.0):
        return "rows_kernel"
    return "filter_rows_kernel" if 0 < top_k <= 64 else "gfilter_rows_kernel"


class Prepared:
    """Input sets of one workload on the device with their marshalled calls:
    unfiltered, one launch per step (the rows kernel finishes the requests in
    its tail); filtered, the row kernel then the request kernel."""

    def __init__(self, L, spec, mode, dev, stream, seed, top_k, top_p, requests=0, n_sets=2):
        kw = {"B": requests} if requests > 0 else {}
        self.sets = [W.make_workload(spec, mode, seed=seed + 100 * i, device=dev, **kw)
                     for i in range(n_sets)]
        w = self.sets[0]
        if any(s.n_target_rows != w.n_target_rows for s in self.sets):
            self.sets = self.sets[:1]  # ragged sets of other lengths: keep one
        self.w = w
        self.filtered = (0 < top_k < w.V) or top_p < 1.0
        self.kernel = row_kernel_name(top_k, top_p, w.V)
        self.out = L.alloc_outputs(w.n_target_rows, w.B, dev, want_conf=True)
        self.ws = L.alloc_workspace(w.B, w.n_target_rows, dev)
        self.kw = dict(max_len=spec.max_len, temperature=spec.temperature, top_k=top_k,
                       top_p=top_p, mode=mode, out=self.out, workspace=self.ws, stream=stream)
        self.calls = []
        for st in self.sets:
            a = (st.target, st.draft, st.draft_tokens, st.uniforms, st.verify_lens, st.row_offsets)
            if self.filtered:
                self.calls.append((L.prepare("spec_verify_rows", *a, **self.kw),
                                   L.prepare("spec_verify_finalize", *a, **self.kw)))
            else:
                self.calls.append((L.prepare("spec_verify", *a, **self.kw), lambda: None))
        self.launches = 2 if self.filtered else 1
        self.positions = w.n_draft_rows
        self.bytes = w.logit_bytes()
        self.l2_cover = self.bytes * len(self.sets) > 2 * L2_BYTES


def time_steps(prep, K, stream, flush=None, end=None):
    """K steps; per step CUDA events around the row launch and around the
    whole step (both on the launch stream).  ``flush``: a buffer larger than
    L2 overwritten before each step, outside the events.  ``end``: an event
    recorded after the last step, before the host waits.  Returns (per-step
    row-launch ms, per-step ms)."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    for i in range(K):
        if flush is not None:
            flush.add_(1)
        rows, fin = prep.calls[i % len(prep.calls)]
        e0, e1, e2 = ev[i]
        e0.record(stream)
        rows()
        e1.record(stream)
        fin()
        e2.record(stream)
    if end is not None:
        end.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b, _ in ev], [a.elapsed_time(c) for a, _, c in ev]


def measure_workload(L, spec, mode, dev, stream, top_k, top_p, oracle_budget_s, flush):
    """One entry of ``per_workload``: drafted positions/s over the summed step
    times, the dominant kernel's mean launch time and its fraction of the HBM
    peak, and the oracle's check of one call on a sample of requests."""
    prep = Prepared(L, spec, mode, dev, stream, seed=5000 + 7 * WORKLOAD_INDEX[spec.name],
                    top_k=top_k, top_p=top_p)
    use_flush = None if prep.l2_cover else flush
    rows_ms, step_ms = time_steps(prep, 5, stream, use_flush)  # warm-up and size
    assert int(prep.out.dev_error.item()) == 0, f"device error flags on {spec.name}"
    K = int(max(20, min(2000, 0.5e3 / max(1e-3, statistics.fmean(step_ms)))))
    rows_ms, step_ms = time_steps(prep, K, stream, use_flush)
    assert int(prep.out.dev_error.item()) == 0, f"device error flags on {spec.name}"
    peak, _ = hbm_peak()
    kernel_ms = statistics.fmean(rows_ms)
    gbs = prep.bytes / (kernel_ms / 1e3) / 1e9
    ent = {"workload": spec.name, "mode": "sample" if mode == W.SAMPLE else "greedy",
           "B": prep.w.B, "V": prep.w.V, "logits": spec.dtype, "top_k": top_k, "top_p": top_p,
           "positions_per_s": prep.positions * K / (sum(step_ms) / 1e3),
           "ms_per_step": statistics.fmean(step_ms), "steps": K,
           "launches_per_step": prep.launches, "kernel": prep.kernel,
           "kernel_mean_ms": kernel_ms, "bytes_per_launch": prep.bytes,
           "achieved_gbs": gbs, "frac": gbs / peak,
           "traffic": recorded_traffic(prep.kernel, spec.name),
           "l2": ("inputs larger than L2: input sets alternate" if prep.l2_cover
                  else "L2 flushed before each step (outside the events)")}
    if oracle_budget_s > 0:
        # one more call, then the oracle on a sample of its requests
        prep.out.dev_error.zero_()
        rows, fin = prep.calls[0]
        rows()
        fin()
        torch.cuda.synchronize()
        counts, rate, secs = oracle_check(prep.w, prep.out, spec, mode, top_k, top_p,
                                          oracle_budget_s)
        ent["oracle_check"] = counts
        ent["oracle_positions_per_s"] = rate
        ent["oracle_seconds"] = secs
    del prep
    torch.cuda.empty_cache()
    return ent


WORKLOAD_INDEX = {s.name: i for i, s in enumerate(W.WORKLOADS)}


def run_ours(args, world, rank, local):
    from speculative_decoding_verification_16_gb300 import binding as L

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    spec = W.WORKLOADS[args.workload]
    mode = W.SAMPLE if args.mode == "sample" else W.GREEDY
    stream = torch.cuda.current_stream(dev)
    top_k = spec.top_k if args.top_k is None else args.top_k
    top_p = spec.top_p if args.top_p is None else args.top_p
    prep = Prepared(L, spec, mode, dev, stream, seed=1000 * args.workload + rank, top_k=top_k,
                    top_p=top_p, requests=args.requests)
    w, out = prep.w, prep.out
    B, V = w.B, w.V
    flush = None
    if not prep.l2_cover:  # small workloads: overwrite 2 x L2 before each step
        flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    for i in range(args.warmup):
        if flush is not None:
            flush.add_(1)
        rows, fin = prep.calls[i % len(prep.calls)]
        rows()
        fin()
    torch.cuda.synchronize(dev)
    assert int(out.dev_error.item()) == 0, "device error flags during warm-up"

    K = args.steps
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    barrier(world)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    rows_ms, step_ms = time_steps(prep, K, stream, flush, end=end)
    barrier(world)
    clocks = sampler.stop() if sampler else None
    # with a flush, only the steps' own events count; else the whole loop
    elapsed_ms = sum(step_ms) if flush is not None else start.elapsed_time(end)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    total_pos = sum_over_ranks(prep.positions * K, world, dev)
    value = total_pos / (elapsed_ms / 1e3)
    assert int(out.dev_error.item()) == 0, "device error flags during the timed steps"

    mean_rows_ms = statistics.fmean(rows_ms)
    achieved = prep.bytes / (mean_rows_ms / 1e3) / 1e9
    peak, peak_src = hbm_peak()
    traffic = recorded_traffic(prep.kernel, spec.name) if args.requests <= 0 else None

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(L, w, spec, mode, dev, stream, prep.kw, K, world)

    cpu = None
    host_cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        counts, rate, secs = oracle_check(w, out, spec, mode, top_k, top_p, 8.0)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "host_cores": host_cores,
               "host_cpu_count": os.cpu_count(), "kind": "oracle",
               "sample": f"{counts['requests']} whole requests ({counts['positions']} drafted "
                         f"positions) of the same workload, {secs:.1f} s of single-thread fp64 "
                         f"oracle time",
               "oracle_check": counts}
    l2_note = (f"inputs larger than L2: {len(prep.sets)} input sets of "
               f"{prep.bytes / 1e6:.0f} MB alternate between steps" if flush is None
               else "L2 flushed before each step (outside the step events)")
    launches = prep.launches
    per = None
    if rank == 0 and world == 1 and not args.no_per_workload:
        del prep
        torch.cuda.empty_cache()
        per = []
        if flush is None:
            flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        budget = 0.0 if args.no_cpu_baseline else 3.0
        for idx, sp in enumerate(W.WORKLOADS):
            for m in sp.modes:
                mm = W.SAMPLE if m == "sample" else W.GREEDY
                per.append(measure_workload(L, sp, mm, dev, stream, sp.top_k, sp.top_p, budget,
                                            flush))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": spec.name, "B": B, "block": spec.max_len, "V": V,
                       "logits": spec.dtype, "mode": args.mode,
                       "temperature": spec.temperature, "top_k": top_k,
                       "top_p": top_p, "labels": True,
                       "l2": l2_note,
                       "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": row_kernel_name(top_k, top_p, V),
                         "bytes_per_launch": w.logit_bytes(),
                         "mean_launch_ms": mean_rows_ms, "peak_source": peak_src},
            "hbm_gbs_step": w.logit_bytes() / (elapsed_ms / K / 1e3) / 1e9,
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks,
            "gpu_launches": launches * K,
            "per_workload": per,
        }
        print(json.dumps(line), flush=True)


def run_e2e(L, w, spec, mode, dev, stream, kw, K, world):
    """Same metric through the public call with host buffers: every step
    copies its inputs from pinned host memory, verifies, and reads the
    outputs back.  As in a serving loop, the upload of the next step's inputs
    (on a copy stream, into the other of two device input sets) overlaps the
    current step's verify; each step still waits for its own upload."""
    host = {n: getattr(w, n).cpu().pin_memory() for n in
            ("target", "draft", "draft_tokens", "uniforms", "verify_lens", "row_offsets")}
    devbufs = [{n: torch.empty_like(t, device=dev) for n, t in host.items()} for _ in range(2)]
    out = kw["out"]
    h_out = [torch.empty(out.tokens.shape, dtype=torch.int32).pin_memory(),
             torch.empty(out.accept_len.shape, dtype=torch.int32).pin_memory(),
             torch.empty(out.conf.shape, dtype=torch.float32).pin_memory()]
    calls = [L.prepare("spec_verify", d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                       d["verify_lens"], d["row_offsets"], **kw) for d in devbufs]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    steps = max(3, min(K, 30))
    copy_stream = torch.cuda.Stream(dev)
    done = [torch.cuda.Event(), torch.cuda.Event()]  # verify of the set finished reading it
    for e in done:
        e.record(stream)

    def upload(i):
        copy_stream.wait_event(done[i % 2])  # the set is free again
        with torch.cuda.stream(copy_stream):
            for n in host:
                devbufs[i % 2][n].copy_(host[n], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(copy_stream)
        return ev

    def run(n_steps):
        ready = upload(0)
        for i in range(n_steps):
            stream.wait_event(ready)
            nxt = upload(i + 1) if i + 1 < n_steps else None
            calls[i % 2]()
            done[i % 2].record(stream)
            h_out[0].copy_(out.tokens, non_blocking=True)
            h_out[1].copy_(out.accept_len, non_blocking=True)
            h_out[2].copy_(out.conf, non_blocking=True)
            ready = nxt

    run(2)
    torch.cuda.synchronize(dev)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    copy_stream.wait_stream(stream)  # the first upload starts inside the timed region
    run(steps)
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    value = sum_over_ranks(steps * w.n_draft_rows, world, dev) / (ms / 1e3)
    # the bound: one step's upload alone (pinned host -> device, copy stream)
    torch.cuda.synchronize(dev)
    ua, ub = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ua.record(copy_stream)
    for i in range(3):
        upload(i)
    ub.record(copy_stream)
    torch.cuda.synchronize(dev)
    up_ms = ua.elapsed_time(ub) / 3
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "overlap": "next step's upload during this step's verify",
            "h2d_gbs_in_loop": h2d * steps / (ms / 1e3) / 1e9,
            "h2d_gbs_upload_alone": h2d / (up_ms / 1e3) / 1e9}


def run_schedule(args, rank):
    """DSpark prefix scheduler: schedules per second on a 256 x 15 pool."""
    import numpy as np

    from speculative_decoding_verification_16_gb300 import binding as L

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    spec = W.WORKLOADS[3]  # ragged, B = 256, block 16
    w = W.make_workload(spec, W.SAMPLE, seed=3000, device=dev)
    out = L.verify_workload(w)
    torch.cuda.synchronize()
    K = spec.max_len - 1
    conf = torch.zeros((w.B, K), dtype=torch.float32, device=dev)
    lens = w.verify_lens.cpu().tolist()
    offs = w.row_offsets.cpu().tolist()
    for r in range(w.B):  # drafted positions of request r; missing ones stay 0
        n = lens[r] - 1
        if n > 0:
            conf[r, :n] = out.conf[offs[r] - r:offs[r] - r + n]
    b = np.arange(w.B * (K + 1) + 2, dtype=np.float64)
    sps_np = 1e4 / np.maximum(1024.0, b)
    sps = torch.tensor(sps_np, device=dev)
    out_lens = torch.empty(w.B, dtype=torch.int32, device=dev)
    theta = torch.empty(2, dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        L.spec_verify_schedule(conf, sps, out_lens=out_lens, out_theta=theta, stream=stream)
    torch.cuda.synchronize()
    K_steps = min(args.steps, 2000)
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K_steps):
        L.spec_verify_schedule(conf, sps, out_lens=out_lens, out_theta=theta, stream=stream)
    e.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / K_steps
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        t0, n = time.perf_counter(), 0
        c_np = conf.cpu().numpy()
        while time.perf_counter() - t0 < 5.0 or n == 0:
            oracle.schedule_prefix(c_np, sps_np)
            n += 1
        cpu = {"value": n / (time.perf_counter() - t0), "unit": "schedules/s", "cores": 1,
               "kind": "oracle", "sample": f"{n} schedules of the same pool, 5 s of one core"}
    if rank == 0:
        print(json.dumps({
            "metric": "DSpark prefix schedules/s (256 requests x 15 positions)",
            "value": 1e3 / ms, "unit": "schedules/s", "n_gpus": 1, "steps": K_steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "dspark_pool_b256_k15",
                       "confidences": "verify labels c* of dspark_ragged_b256_v129280",
                       "sps": "synthetic: 1e4 / max(1024, B)",
                       "added": int(theta[1].item()), "theta": float(theta[0].item())},
            "roofline": {"bound": "latency", "achieved": None, "peak": None, "unit": None,
                         "frac": None, "traffic": None, "kernel": "schedule_kernel"},
            "cpu_baseline": cpu, "gpu_launches": K_steps,
        }), flush=True)


def run_split(args, rank):
    """Vocabulary-split verify: one rank's kernel times, emulated in lockstep."""
    from speculative_decoding_verification_16_gb300.sharded import ShardRank, split_columns

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    spec = W.WORKLOADS[args.workload]
    mode = W.SAMPLE if args.mode == "sample" else W.GREEDY
    w = W.make_workload(spec, mode, seed=args.workload, device=dev)
    n_t, V = w.target.shape
    n_d = w.draft.shape[0]
    world = args.split_world
    ranks = [ShardRank(q, world, v0, V, w.target[:, v0:v0 + vq].contiguous(),
                       w.draft[:, v0:v0 + vq].contiguous(), w.draft_tokens, w.uniforms,
                       w.verify_lens, w.row_offsets, max_len=spec.max_len,
                       temperature=spec.temperature, mode=mode, want_conf=True)
             for q, (v0, vq) in enumerate(split_columns(V, world))]
    sample = mode == W.SAMPLE
    flush = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    names = ["stats", "gather 1", "merge", "masses", "gather 2", "draw", "gather 3", "finish"]

    def step(ev):
        # ev: events before each phase and one after the last (or None)
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        flush.add_(1)
        mark(0)
        for r in ranks:
            r.stats()
        mark(1)
        recs = torch.stack([r.rec for r in ranks])
        mark(2)
        for r in ranks:
            r.merge(recs)
        if ev is not None:
            ev[3].record(stream)
        flush.add_(1)  # the masses pass re-reads the columns from HBM
        mark(4)
        for r in ranks:
            r.masses()
        mark(5)
        masses = torch.stack([r.mass for r in ranks])
        mark(6)
        for r in ranks:
            r.draw(masses)
        mark(7)
        if sample:
            cands = torch.stack([r.cand for r in ranks])
            mark(8)
            for r in ranks:
                r.finish(cands)
        else:
            mark(8)
        mark(9)

    for _ in range(max(3, args.warmup)):
        step(None)
    torch.cuda.synchronize()
    K = min(args.steps, 200)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(10)] for _ in range(K)]
    for k in range(K):
        step(evs[k])
    torch.cuda.synchronize()
    # phase ms per step; [3] -> [4] is the flush, not a phase
    spans = [(0, 1), (1, 2), (2, 3), (4, 5), (5, 6), (6, 7), (7, 8), (8, 9)]
    ph = {n: statistics.mean(e[a].elapsed_time(e[b]) for e in evs) for n, (a, b) in zip(names, spans)}
    per_rank = {n: ph[n] / world for n in names if not n.startswith("gather")}
    rank_ms = sum(per_rank.values())
    es = w.target.element_size()
    vq_max = max(vq for _, vq in split_columns(V, world))
    rank_bytes = (n_t + n_d) * vq_max * es  # one pass over the widest rank's columns
    top = max(("stats", "masses"), key=lambda n: per_rank[n])
    peak, src = hbm_peak()
    ach = rank_bytes / (per_rank[top] * 1e-3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "vocabulary-split verify: drafted positions/s of one rank's kernels",
            "value": n_d / (rank_ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": rank_ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": spec.name, "world": world, "mode": args.mode,
                       "labels": True,
                       "ranks": "emulated in lockstep on one GPU; each phase's time / world",
                       "l2": "flushed before the stats pass and before the masses pass"},
            "phases_us_per_rank": {n: 1e3 * v for n, v in per_rank.items()},
            "gather_us_all_ranks": {n: 1e3 * ph[n] for n in names if n.startswith("gather")},
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s",
                         "frac": ach / peak, "traffic": None, "kernel": f"shard_{top}_kernel",
                         "bytes_per_launch": rank_bytes,
                         "mean_launch_ms": per_rank[top], "peak_source": src},
            "gpu_launches": K * world * (5 if sample else 4),
        }), flush=True)


def main():
    args = parse()
    world, rank, local = dist_setup()
    if args.component == "schedule":
        run_schedule(args, rank)
    elif args.component == "split":
        run_split(args, rank)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
