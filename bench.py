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

--component schedule prints one line for the DSpark prefix scheduler instead
(spec_verify_schedule on a pool of 256 requests x 15 positions whose
confidences are the verify step's own labels on the ragged workload; the
SPS curve is synthetic: flat to 1,024 tokens, then falling as 1/B), with the
fp64 oracle timed beside it.
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
    ap.add_argument("--component", choices=("verify", "schedule"), default="verify")
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


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(PKG, "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name):
    """DRAM bytes per launch of the rows kernel from the committed ncu summary,
    or None when the kernel sources changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "rows_kernel_traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    ent = rec.get(workload_name)
    if not ent or ent.get("source_sha256") != kernel_source_hash():
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
def run_ours(args, world, rank, local):
    from speculative_decoding_verification_16_gb300 import binding as L

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    spec = W.WORKLOADS[args.workload]
    mode = W.SAMPLE if args.mode == "sample" else W.GREEDY
    seed = 1000 * args.workload + rank
    kw = {"B": args.requests} if args.requests > 0 else {}
    sets = [W.make_workload(spec, mode, seed=seed + 100 * i, device=dev, **kw) for i in range(2)]
    w = sets[0]
    B, Nt, Nd, V = w.B, w.n_target_rows, w.n_draft_rows, w.V
    stream = torch.cuda.current_stream(dev)
    out = L.alloc_outputs(Nt, B, dev, want_conf=True)
    ws = L.alloc_workspace(B, Nt, dev)
    top_k = spec.top_k if args.top_k is None else args.top_k
    top_p = spec.top_p if args.top_p is None else args.top_p
    kw = dict(max_len=spec.max_len, temperature=spec.temperature, top_k=top_k,
              top_p=top_p, mode=mode, out=out, workspace=ws, stream=stream)
    # unfiltered: one launch per step (the rows kernel finishes the requests
    # in its tail), timed whole; filtered: the row kernel, timed alone, then
    # the request kernel
    filtered = (0 < top_k < V) or top_p < 1.0
    # kept sets of at most 64 tokens take the small-set row kernel
    row_kernel = ("filter_rows_kernel" if 0 < top_k <= 64 else "gfilter_rows_kernel") \
        if filtered else "rows_kernel"
    calls = []
    for s in sets:
        args_ = (s.target, s.draft, s.draft_tokens, s.uniforms, s.verify_lens, s.row_offsets)
        if filtered:
            calls.append((L.prepare("spec_verify_rows", *args_, **kw),
                          L.prepare("spec_verify_finalize", *args_, **kw)))
        else:
            calls.append((L.prepare("spec_verify", *args_, **kw), lambda: None))
    launches_per_step = 2 if filtered else 1
    # (sets use their own lengths; for ragged workloads the second set is
    # drawn with a different seed, so row counts may differ)
    n_rows = [s.n_target_rows + s.n_draft_rows for s in sets]
    n_pos = [s.n_draft_rows for s in sets]
    if n_rows[0] != n_rows[1]:
        sets, calls, n_rows, n_pos = sets[:1], calls[:1], n_rows[:1], n_pos[:1]

    for i in range(args.warmup):
        rows, fin = calls[i % len(calls)]
        rows()
        fin()
    torch.cuda.synchronize(dev)
    assert int(out.dev_error.item()) == 0, "device error flags during warm-up"

    K = args.steps
    ev_rows = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.3 if sampler else 0.0)
    barrier(world)
    torch.cuda.synchronize(dev)
    start.record(stream)
    positions = 0
    for i in range(K):
        rows, fin = calls[i % len(calls)]
        e0, e1 = ev_rows[i]
        e0.record(stream)
        rows()
        e1.record(stream)
        fin()
        positions += n_pos[i % len(calls)]
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop() if sampler else None
    elapsed_ms = start.elapsed_time(end)
    rows_ms = [a.elapsed_time(b) for a, b in ev_rows]
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    total_pos = sum_over_ranks(positions, world, dev)
    value = total_pos / (elapsed_ms / 1e3)
    assert int(out.dev_error.item()) == 0, "device error flags during the timed steps"

    esize = w.target.element_size()
    bytes_per_launch = (sum(n_rows) / len(n_rows)) * V * esize
    mean_rows_ms = statistics.fmean(rows_ms)
    achieved = bytes_per_launch / (mean_rows_ms / 1e3) / 1e9
    peak, peak_src = hbm_peak()
    # the recorded traffic is for the full-size workload only
    traffic = recorded_traffic(spec.name) if args.requests <= 0 else None

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(L, sets[0], spec, mode, dev, stream, kw, K, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, pos, secs, nreq = oracle_rate(w, spec, mode, 10.0, top_k=top_k, top_p=top_p)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{nreq} whole requests ({pos} drafted positions) of the same "
                         f"workload, {secs:.1f} s of single-thread fp64 oracle time"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": spec.name, "B": B, "block": spec.max_len, "V": V,
                       "logits": spec.dtype, "mode": args.mode,
                       "temperature": spec.temperature, "top_k": top_k,
                       "top_p": top_p, "labels": True,
                       "l2": f"inputs larger than L2: {len(sets)} input sets of "
                             f"{bytes_per_launch / 1e6:.0f} MB alternate between steps",
                       "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": row_kernel,
                         "bytes_per_launch": bytes_per_launch,
                         "mean_launch_ms": mean_rows_ms, "peak_source": peak_src},
            "hbm_gbs_step": bytes_per_launch / (elapsed_ms / K / 1e3) / 1e9,
            "e2e": e2e, "cpu_baseline": cpu, "clocks": clocks,
            "gpu_launches": launches_per_step * K,
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
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "overlap": "next step's upload during this step's verify"}


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


def main():
    args = parse()
    world, rank, local = dist_setup()
    if args.component == "schedule":
        run_schedule(args, rank)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
