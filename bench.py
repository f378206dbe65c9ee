"""Benchmark of the speculative-sampling verification step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config c4]

A step is one verification call over one batch of the workload (default: the
largest single-GPU workload, B=256 sequences, K=4 drafts, V=256000, fp32
logits, T=1). Inputs are seeded synthetic logits, drawn on the device and
resident in HBM before timing starts; a step streams more than twice the L2
(smaller workloads rotate over input sets, or flush L2 between steps). The K
steps are captured in one CUDA graph, which is replayed back to back until at
least --min-seconds have passed, timed with CUDA events on the launching
stream; a second graph with events between the two kernels gives each
kernel's time for the roofline figure.

Rank 0 prints one JSON line. `value` is verified draft positions per second
over all ranks (B*K per step); `e2e` is the same metric through the
host-buffer entry points (host->device copy of each step's inputs from pinned
memory, device->host copy of its outputs, inside the timed region).
`cpu_baseline` is the fp64 oracle on a bounded sample of the same step, on one
core and on every host core, and `parity` compares the GPU's decisions with
the oracle's on that sample. `workloads` holds sub-records (ms per step,
GB/s, mean accepted length) for the 64x8x128256 workload and the 20 cells of
the acceptance sweep. `--impl reference` times the fp64 CPU oracle on the
host cores instead.
"""

from __future__ import annotations

import argparse
import json
import os
import platform
import shutil
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from synthetic import (SWEEP_K, SWEEP_NOISE, get_workload, make_batch, make_inputs,  # noqa: E402
                       make_topk_inputs, make_topp_inputs)

L2_BYTES = 129 * 1024 * 1024
METRIC = "verified draft positions/sec (and achieved HBM GB/s, % of GB300 peak)"
UNIT = "draft_positions/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c4", help="c1..c4 or sweep-k{K}-n{noise}")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="verify: replay the K-step graph until this much time has passed")
    ap.add_argument("--sub", default="c3,sweep",
                    help="verify: workloads measured after the headline, as sub-records")
    ap.add_argument("--no-sub", action="store_true")
    ap.add_argument("--ncu-case", type=int, default=0,
                    help="verify: run --steps calls on the workload cut to this many sequences "
                         "and exit (a small case for ncu captures)")
    ap.add_argument("--path", choices=["auto", "pair", "fused"], default="auto",
                    help="verify, --ncu-case: force the kernel pair or the fused kernel")
    ap.add_argument("--op", choices=["verify", "draft_sample", "greedy", "topk", "topp",
                                     "lmhead"],
                    default="verify",
                    help="verify: the verification step (default); draft_sample: the draft-side "
                         "sampler over every draft row of the workload; greedy: greedy-mode "
                         "verification of the workload's target rows; topk: verification on "
                         "top-k filtered distributions (--top-k); topp: verification on nucleus "
                         "filtered distributions (--top-p); lmhead: the scoring step's "
                         "projection fused with the row statistics (tensor cores)")
    ap.add_argument("--top-k", type=int, default=50)
    ap.add_argument("--top-p", type=float, default=0.9)
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def reduce_max(x: float, world: int, device=None) -> float:
    """Maximum of a per-rank float over all ranks (identity at world size 1)."""
    if world <= 1:
        return float(x)
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: int, world: int, seconds_max: float) -> float:
    """Whole-job throughput: units every rank processed over the slowest rank's time."""
    return world * units_per_rank / seconds_max


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def load_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if the
    summary was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
        ent = data[f"{kernel}@{workload}"]
    except Exception:
        return None
    import hashlib

    src = os.path.join(ROOT, "speculative_sampling_verification_gb300", "csrc", "sv_kernels.cu")
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return ent["dram_bytes_per_launch"] if ent.get("source_sha") == h else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 50 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [p for (t, p) in self.samples if t0 - 0.1 <= t <= t1 + 0.1] or \
               [p for (_, p) in self.samples]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][1]), "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- the host and the oracle on its cores

def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def host_info() -> dict:
    return {"nproc": os.cpu_count(), "cores_available": host_cores(), "cpu_model": cpu_model(),
            "arch": platform.machine()}


def _scratch_dir() -> str:
    """A directory for the oracle's input files: /dev/shm when it has room,
    else the default temporary directory."""
    try:
        if shutil.disk_usage("/dev/shm").free > (16 << 30):
            return "/dev/shm"
    except Exception:
        pass
    return tempfile.gettempdir()


def _to_np(t: torch.Tensor) -> np.ndarray:
    """CPU numpy copy of a tensor; bf16 is kept as its raw 16-bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def save_oracle_job(tmp: str, tag: str, inp: dict, seqs) -> list:
    """Write sequences `seqs` of an input dict (CPU or GPU tensors) to .npy
    files under `tmp`; returns their paths (target, draft, tokens, uniforms)."""
    idx = torch.as_tensor(list(seqs), dtype=torch.long)
    paths = []
    for k in ("target", "draft", "tokens", "uniforms"):
        x = inp[k]
        x = x[idx.to(x.device)]
        p = os.path.join(tmp, f"{tag}-{k}.npy")
        np.save(p, _to_np(x))
        paths.append(p)
    return paths


def _load_oracle_job(paths):
    t, d, k, u = (np.load(p, mmap_mode="r") for p in paths)
    if t.dtype == np.uint16:  # bf16 bit patterns: widen exactly to fp32
        t = (t.astype(np.uint32) << np.uint32(16)).view(np.float32)
        d = (d.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return (np.ascontiguousarray(t), np.ascontiguousarray(d), np.asarray(k).astype(np.int64),
            np.asarray(u))


def oracle_job(job):
    """One oracle job (run in this process or in a spawned worker): the fp64
    oracle over the sequences stored in `paths`, repeated for `seconds` (at
    least once). Returns (sequences verified, seconds, the first result)."""
    import oracle

    paths, temperature, seconds = job
    t, d, k, u = _load_oracle_job(paths)
    t0 = time.perf_counter()
    n, first = 0, None
    while True:
        r = oracle.verify(t, d, k, u, temperature)
        n += t.shape[0]
        if first is None:
            first = r
        if time.perf_counter() - t0 >= seconds:
            break
    return n, time.perf_counter() - t0, first


class OracleHost:
    """The fp64 oracle on the host's cores: a spawn pool fed through .npy files."""

    def __init__(self, workers: int):
        import multiprocessing as mp

        self.workers = max(1, workers)
        self.tmp = tempfile.mkdtemp(prefix="sv-oracle-", dir=_scratch_dir())
        self.pool = mp.get_context("spawn").Pool(self.workers)

    def close(self):
        self.pool.terminate()
        self.pool.join()
        shutil.rmtree(self.tmp, ignore_errors=True)


def oracle_sample_plan(w, cores: int, call_s: float = 0.25):
    """Sequences per oracle call, sized so that one call takes about `call_s`
    on one core (about 25 ns per logit element)."""
    per_seq = (2 * w.K + 1) * w.V * 25e-9
    return max(1, min(w.B, int(call_s / per_seq)))


def cpu_baselines(w, inp: dict, host: OracleHost, seconds: float = 10.0):
    """The oracle, as it stands, on a bounded sample of one step of `w`
    (`inp`, the GPU's own inputs): one thread in this process, then every
    host core through the pool, each job on different sequences. Returns
    (single, all_cores, the per-sequence oracle results with their indices)."""
    per = oracle_sample_plan(w, host.workers)
    jobs = []
    for j in range(host.workers):
        seqs = [(j * per + i) % w.B for i in range(per)]
        jobs.append((seqs, save_oracle_job(host.tmp, f"{w.name}-{j}", inp, seqs)))
    T = inp["temperature"]
    n1, dt1, _ = oracle_job((jobs[0][1], T, seconds))
    single = {"value": n1 * w.K / dt1, "unit": UNIT, "cores": 1, "kind": "oracle",
              "sample": f"{n1 // per} oracle calls over {per} sequences of {w.name} in "
                        f"{dt1:.1f} s (fp64 numpy oracle, 1 thread)"}
    res = host.pool.map(oracle_job, [(p, T, seconds) for _, p in jobs])
    rate = sum(n / dt for n, dt, _ in res) * w.K
    calls = sum(n for n, _, _ in res) // per
    every = {"value": rate, "unit": UNIT, "cores": host.workers, "kind": "oracle",
             "sample": f"{calls} oracle calls over {per} sequences each of {w.name}, one process "
                       f"per core on {host.workers} cores, {seconds:.0f} s each (fp64 numpy "
                       f"oracle)"}
    checked = [(seqs, r) for (seqs, _), (_, _, r) in zip(jobs, res)]
    return single, every, checked


def parity_sample(checked, out: np.ndarray, nacc: np.ndarray, tokens: np.ndarray) -> dict:
    """Decisions of the GPU's step against the oracle's on the sampled sequences."""
    from tests import _parity

    rep = _parity.ParityReport()
    seen = set()
    for seqs, r in checked:
        keep = [i for i, b in enumerate(seqs) if b not in seen]
        seen.update(seqs)
        if not keep:
            continue
        b = np.asarray(seqs)[keep]
        sub = type(r)(*[getattr(r, f)[keep] for f in r.__dataclass_fields__])
        rep.add(_parity.compare(out[b], nacc[b], sub, tokens[b]))
    d = rep.as_dict()
    d["margin"] = _parity.MARGIN
    return d


# ---------------------------------------------------------------- timing helpers

def make_sets(w, n_sets: int, dev, step_base: int):
    """`n_sets` input sets of `w`, drawn on the device by the batched generator."""
    return [make_batch(w, step=step_base + i, device=dev) for i in range(n_sets)]


def l2_plan(set_bytes: int, max_sets: int = 2):
    """Input sets to rotate over, and whether L2 must be flushed between steps:
    a step whose logits exceed twice the L2 needs neither."""
    if set_bytes >= 2 * L2_BYTES:
        return 1, False
    n = min(max_sets, -(-2 * L2_BYTES // set_bytes))
    return n, n * set_bytes < 2 * L2_BYTES


def time_sub_workload(sv, name: str, dev, stream, reps_min_s: float = 0.25, steps: int = 20):
    """ms per step, GB/s and mean accepted length of one workload (a
    sub-record): `steps` calls in one CUDA graph, each bracketed by its own
    events, L2 flushed between calls when the inputs fit in it."""
    w = get_workload(name)
    dt_code = sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32
    B, K, V, es = w.B, w.K, w.V, w.elem_bytes
    set_bytes = B * (2 * K + 1) * V * es
    n_sets, flush = l2_plan(set_bytes)
    sets = make_sets(w, n_sets, dev, 500)
    outs = [(torch.empty(B, K + 1, dtype=torch.int32, device=dev),
             torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(n_sets)]
    ws = sv.new_workspace(B, K, V, dt_code, dev)
    scrub = torch.empty(3 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    T = w.temperature
    # external: recorded inside the graph as timing nodes
    evs = [(torch.cuda.Event(enable_timing=True, external=True),
            torch.cuda.Event(enable_timing=True, external=True)) for _ in range(steps)]

    def call(i):
        s = sets[i % n_sets]
        o, n = outs[i % n_sets]
        rc = sv.spec_verify(s["target"], s["draft"], s["tokens"], s["uniforms"], T, o, n, ws)
        if rc != 0:
            raise RuntimeError(f"spec_verify failed: {sv.sv_status_string(rc)}")

    with torch.cuda.stream(stream):
        call(0)
        for a, b in evs:
            a.record(stream)
            b.record(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(steps):
            if scrub is not None:
                scrub.fill_(float(i))
            evs[i][0].record(stream)
            call(i)
            evs[i][1].record(stream)
    torch.cuda.synchronize()
    g.replay()  # warm-up
    torch.cuda.synchronize()
    per_rep, t0 = [], time.perf_counter()
    while not per_rep or time.perf_counter() - t0 < reps_min_s:
        g.replay()
        torch.cuda.synchronize()
        per_rep.append(float(np.mean([a.elapsed_time(b) for a, b in evs])))
    if sv.sv_read_device_status(ws, stream) != 0:
        raise RuntimeError(f"bad device status on {name}")
    ms = float(np.median(per_rep))
    nacc = torch.stack([n for _, n in outs]).cpu().numpy()
    peak, _ = load_peaks()
    ideal = w.ideal_bytes_per_step()
    fused = sv.sv_kernels_per_call(B, K, V, dt_code) == 1
    del sets, outs, ws, scrub, g
    torch.cuda.empty_cache()
    return {"workload": w.name, "ms_per_step": ms, "draft_positions_per_s": B * K / (ms * 1e-3),
            "sequences_per_s": B / (ms * 1e-3), "hbm_gbs_ideal_bytes": ideal / (ms * 1e-3) / 1e9,
            "frac_of_peak_ideal_bytes": ideal / (ms * 1e-3) / 1e9 / peak,
            "mean_accepted": float(nacc.mean()), "sequences_for_mean": int(nacc.size),
            "path": "fused_kernel" if fused else "stats_kernel + draw_kernel",
            "l2": "flushed between calls" if flush else f"inputs rotate over {n_sets} sets "
                                                         f"(> 2x L2)",
            "repeats": len(per_rep)}


# ---------------------------------------------------------------- the verification step

def run_reference(args, w, world, rank):
    """The reference arm: the fp64 oracle, as it stands, on every host core.
    A step is one oracle call per core over a bounded sample of the workload's
    sequences (one process per core, each on its own sequences)."""
    if rank != 0:
        return
    steps = max(1, args.steps)
    cores = host_cores()
    host = OracleHost(cores)
    try:
        per = oracle_sample_plan(w, cores)
        seqs_all = sorted({(j * per + i) % w.B for j in range(cores) for i in range(per)})
        inp = make_inputs(w, step=20_000, seqs=seqs_all)
        pos = {b: i for i, b in enumerate(seqs_all)}
        jobs = [save_oracle_job(host.tmp, f"ref-{j}", inp,
                                [pos[(j * per + i) % w.B] for i in range(per)])
                for j in range(cores)]
        T = inp["temperature"]
        for _ in range(max(1, args.warmup)):
            host.pool.map(oracle_job, [(p, T, 0.0) for p in jobs])
        t0 = time.perf_counter()
        for _ in range(steps):
            host.pool.map(oracle_job, [(p, T, 0.0) for p in jobs])
        dt = time.perf_counter() - t0
    finally:
        host.close()
    value = steps * cores * per * w.K / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": dt / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": bench_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: {cores} processes, one per core, each running "
                                   f"the oracle once over {per} sequences of {w.name}",
                         "host": host_info()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_config(w) -> dict:
    """The `config` object of the verification step's line (both arms)."""
    return {"workload": w.name, "detail": w.describe()}


def run_ncu_case(args, w, dev, sv):
    """A small case of the workload for ncu: its first `--ncu-case` sequences,
    `--steps` verification calls on one input set, on the chosen kernel path."""
    from synthetic.configs import shrink

    w = shrink(w, B=min(w.B, args.ncu_case))
    sv.sv_force_path({"auto": 0, "pair": 1, "fused": 2}[args.path])
    inp = make_batch(w, step=1, device=dev)
    dt_code = sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32
    ws = sv.new_workspace(w.B, w.K, w.V, dt_code, dev)
    out = torch.empty(w.B, w.K + 1, dtype=torch.int32, device=dev)
    nacc = torch.empty(w.B, dtype=torch.int32, device=dev)
    for _ in range(max(1, args.steps)):
        rc = sv.spec_verify(inp["target"], inp["draft"], inp["tokens"], inp["uniforms"],
                            w.temperature, out, nacc, ws)
        if rc != 0:
            raise RuntimeError(sv.sv_status_string(rc))
    torch.cuda.synchronize()
    if sv.sv_read_device_status(ws) != 0:
        raise RuntimeError("bad device status")
    print(json.dumps({"ncu_case": w.name, "B": w.B, "path": args.path, "calls": args.steps,
                      "mean_accepted": float(nacc.float().mean())}))


def run_ours(args, w, world, rank, local):
    import speculative_sampling_verification_gb300 as sv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sv.load_library(build=True)
    if args.ncu_case:
        return run_ncu_case(args, w, dev, sv)
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    host = OracleHost(host_cores()) if want_cpu else None  # spawned before any GPU work
    try:
        _run_ours(args, w, world, rank, local, dev, sv, host)
    finally:
        if host is not None:
            host.close()


def _run_ours(args, w, world, rank, local, dev, sv, host):
    dt_code = sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32
    B, K, V, es = w.B, w.K, w.V, w.elem_bytes
    set_bytes = B * (2 * K + 1) * V * es
    n_sets, flush = l2_plan(set_bytes, max_sets=64)
    sets = make_sets(w, n_sets, dev, 1000 * rank)
    outs = [(torch.empty(B, K + 1, dtype=torch.int32, device=dev),
             torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(n_sets)]
    ws = sv.new_workspace(B, K, V, dt_code, dev)
    T = w.temperature
    stream = torch.cuda.Stream(dev)
    scrub = torch.empty(3 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    def call(i, evs=None):
        s = sets[i % n_sets]
        o, n = outs[i % n_sets]
        if evs is None:
            rc = sv.spec_verify(s["target"], s["draft"], s["tokens"], s["uniforms"], T, o, n, ws)
        else:
            rc = sv.spec_verify_profiled(s["target"], s["draft"], s["tokens"], s["uniforms"], T,
                                         o, n, ws, *evs)
        if rc != 0:
            raise RuntimeError(f"spec_verify failed: {sv.sv_status_string(rc)}")

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        call(0)  # first call on the device: kernel set-up, before any capture
    torch.cuda.synchronize()

    steps, warmup = args.steps, max(3, args.warmup)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
            torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for trio in evs:  # torch creates the CUDA event on its first record
        for e in trio:
            e.record(stream)
    torch.cuda.synchronize()
    # g_timed is the product path (plain calls, the draw kernel launched as a
    # programmatic dependent of the streaming kernel) and gives `value`;
    # g_prof repeats the steps with events between the two kernels (which
    # makes the draw an ordinary launch) and gives the per-kernel times.
    g_warm, g_timed, g_prof = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()

    def steps_into(graph, first, n, with_evs=False):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n):
                if scrub is not None:
                    scrub.fill_(float(i))
                call(first + i, evs[i] if with_evs else None)

    steps_into(g_warm, 0, warmup)
    steps_into(g_timed, warmup, steps)
    steps_into(g_prof, warmup, steps, with_evs=True)
    torch.cuda.synchronize()

    # The timed region: the K-step graph replayed back to back until at least
    # a second has passed, inside one barrier + synchronise bracket.
    g_warm.replay()
    torch.cuda.synchronize()
    t_est = time.perf_counter()
    g_timed.replay()
    torch.cuda.synchronize()
    est = max(time.perf_counter() - t_est, 1e-4)
    reps = max(1, int(np.ceil(args.min_seconds / est)))
    rep_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for a, b in rep_evs:
            a.record(stream)
            g_timed.replay()
            b.record(stream)
        end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = start.elapsed_time(end)
    rep_ms = [a.elapsed_time(b) for a, b in rep_evs]
    g_prof.replay()
    torch.cuda.synchronize()
    time.sleep(0.3)
    clocks.stop()

    status = sv.sv_read_device_status(ws, stream)
    nacc_all = torch.stack([n for _, n in outs]).cpu().numpy()
    out_all = torch.stack([o for o, _ in outs]).cpu().numpy()
    drawn = np.take_along_axis(out_all, np.clip(nacc_all, 0, K)[..., None], axis=-1)
    bad_outputs = int((drawn < 0).sum())
    if status != 0 or (nacc_all < 0).any() or (nacc_all > K).any() or bad_outputs:
        raise RuntimeError(f"bad device status {status}, n_accepted out of range or "
                           f"{bad_outputs} undrawn tokens")

    stats_ms = float(np.mean([a.elapsed_time(b) for a, b, _ in evs]))
    draw_ms = float(np.mean([b.elapsed_time(c) for _, b, c in evs]))
    elapsed_ms = reduce_max(elapsed_ms, world, dev)

    # End to end through the host-buffer entry points: every step copies its
    # inputs from pinned host memory and reads its outputs back. `e2e` is a
    # serving loop over two lanes (stream, staging, workspace, host outputs)
    # with spec_verify_host_async, so that one step's copies overlap the
    # previous step's kernels; each step's results are read, its status
    # checked and its drawn tokens counted, before its lane is reused.
    # `e2e_sync` is one blocking spec_verify_host call per step.
    host_sets = [{k: (v.cpu().pin_memory() if torch.is_tensor(v) else v) for k, v in s.items()}
                 for s in sets[:2]]
    n_host = len(host_sets)
    e2e_steps = args.e2e_steps or max(8, min(steps, int(np.ceil(0.5 / (est / steps)))))
    lanes = []
    for j in range(2):
        lanes.append({
            "stream": stream if j == 0 else torch.cuda.Stream(dev),
            "staging": torch.empty(sv.sv_staging_size(B, K, V, dt_code), dtype=torch.uint8,
                                   device=dev),
            "ws": ws if j == 0 else sv.new_workspace(B, K, V, dt_code, dev),
            "out": torch.empty(B, K + 1, dtype=torch.int32).pin_memory(),
            "nacc": torch.empty(B, dtype=torch.int32).pin_memory()})
    h_out, h_nacc, staging = lanes[0]["out"], lanes[0]["nacc"], lanes[0]["staging"]

    def host_call(i):
        h = host_sets[i % n_host]
        rc = sv.spec_verify_host(h["target"], h["draft"], h["tokens"], h["uniforms"], T, h_out,
                                 h_nacc, staging, ws, stream=stream)
        if rc != 0:
            raise RuntimeError(f"spec_verify_host: {rc}")

    def pipelined(n):
        undrawn = 0
        for i in range(n + 2):
            lane = lanes[i % 2]
            if i >= 2:  # step i-2 on this lane: wait, check and read its results
                lane["stream"].synchronize()
                if sv.sv_read_device_status(lane["ws"], lane["stream"]) != 0:
                    raise RuntimeError("bad device status in the e2e loop")
                o, na = lane["out"].numpy(), lane["nacc"].numpy()
                undrawn += int((o[np.arange(B), na] < 0).sum())
            if i < n:
                h = host_sets[i % n_host]
                rc = sv.spec_verify_host_async(h["target"], h["draft"], h["tokens"],
                                               h["uniforms"], T, lane["out"], lane["nacc"],
                                               lane["staging"], lane["ws"], stream=lane["stream"])
                if rc != 0:
                    raise RuntimeError(f"spec_verify_host_async: {rc}")
        return undrawn

    for i in range(3):
        host_call(i)
    pipelined(4)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        host_call(i)
    e2e_sync_s = reduce_max(time.perf_counter() - t0, world, dev)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    undrawn = pipelined(e2e_steps)
    e2e_s = reduce_max(time.perf_counter() - t0, world, dev)
    if undrawn:
        raise RuntimeError(f"{undrawn} undrawn tokens (-1 at position n_accepted) in the e2e loop")
    del host_sets, lanes

    if rank != 0:
        return
    timed_steps = steps * reps
    per_step_s = elapsed_ms / 1e3 / timed_steps
    value = aggregate(B * K, world, per_step_s)
    ideal = w.ideal_bytes_per_step()
    peak, peak_kind = load_peaks()
    fused = sv.sv_kernels_per_call(B, K, V, dt_code) == 1
    # Rows the draw reads per step: two per residual draw, one per bonus draw.
    draw_rows = float(np.where(nacc_all < K, 2, 1).sum(axis=1).mean())
    stream_bytes = B * (2 * K + 1) * V * es
    draw_bytes = draw_rows * V * es
    if fused:
        # One launch streams the B(2K+1) rows and re-reads the draw's rows.
        kern = {"kernel": "fused_kernel (streaming, scan and draw)", "ms": stats_ms,
                "bytes": stream_bytes + draw_bytes,
                "basis": "B(2K+1) rows once, plus 2 rows per residual draw and 1 per bonus "
                         "draw"}
        traffic = load_traffic("fused_kernel", w.name)
        draw_rec = {"ms_per_launch": None, "note": "inside fused_kernel",
                    "rows_reread_per_step": draw_rows}
    else:
        stats = {"kernel": "stats_kernel (streaming row statistics)", "ms": stats_ms,
                 "bytes": stream_bytes, "basis": "B(2K+1) rows of V elements, once"}
        draw = {"kernel": "draw_sum_kernel + draw_finish_kernel (residual / bonus draw)",
                "ms": draw_ms,
                "bytes": draw_bytes, "basis": "2 rows per residual draw, 1 per bonus draw"}
        kern = stats if stats_ms >= draw_ms else draw
        traffic = load_traffic("stats_kernel" if kern is stats else "draw_kernel", w.name)
        draw_rec = {"ms_per_launch": draw_ms, "rows_reread_per_step": draw_rows,
                    "achieved_gbs": draw_bytes / (draw_ms * 1e-3) / 1e9,
                    "frac": draw_bytes / (draw_ms * 1e-3) / 1e9 / peak,
                    "stats_ms_per_launch": stats_ms}
    achieved = kern["bytes"] / (kern["ms"] * 1e-3) / 1e9
    h2d = B * (K + 1) * V * es + B * K * V * es + B * K * 4 + B * (K + 2) * 4
    d2h = B * (K + 1) * 4 + B * 4 + 4

    cpu = parity = None
    if host is not None:
        s0 = sets[0]
        single, every, checked = cpu_baselines(w, s0, host)
        cpu = dict(every, single_thread=single, host=host_info())
        parity = parity_sample(checked, out_all[0], nacc_all[0], s0["tokens"].cpu().numpy())
        parity["sample"] = (f"the timed step's outputs on input set 0 against the oracle "
                            f"results of the cpu_baseline leg ({parity['sequences']} sequences)")
    subs = []
    if world == 1 and not args.no_sub:
        del sets, outs, ws, scrub, g_warm, g_timed, g_prof
        torch.cuda.empty_cache()
        for name in args.sub.split(","):
            for cell in expand_sub(name):
                if get_workload(cell).name != w.name:
                    subs.append(time_sub_workload(sv, cell, dev, stream))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": per_step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": bench_config(w),
        "input_dtype": w.dtype,
        "timing": {"l2": (f"inputs rotate over {n_sets} resident sets of "
                          f"{set_bytes / 1e6:.1f} MB" if not flush else
                          f"L2 flushed (a {3 * L2_BYTES // 4 / 1e6:.0f} MB write) between steps")
                         if n_sets > 1 or flush else "each step streams more than twice the L2",
                   "method": "K plain steps captured in one CUDA graph; the graph replayed "
                             "back to back until at least min_seconds passed, CUDA events on "
                             "the launching stream around the whole region (value) and around "
                             "each replay (median); kernel split from a second graph with "
                             "events between the two kernels",
                   "repeats": reps, "timed_steps": timed_steps,
                   "ms_per_step_median_repeat": float(np.median(rep_ms)) / steps,
                   "min_seconds": args.min_seconds},
        "sequences_per_s": world * B / per_step_s,
        "hbm_gbs_ideal_bytes": ideal / per_step_s / 1e9 * world,
        "frac_of_peak_ideal_bytes": ideal / per_step_s / 1e9 / peak,
        "mean_accepted": float(nacc_all.mean()),
        "roofline": {"bound": "hbm", "kernel": kern["kernel"], "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "traffic": traffic,
                     "bytes_per_launch": kern["bytes"], "ms_per_launch": kern["ms"],
                     "bytes_basis": kern["basis"]},
        "draw_kernel": draw_rec,
        "e2e": {"value": aggregate(B * K * e2e_steps, world, e2e_s), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "spec_verify_host_async, two lanes: a step's copies overlap the previous "
                       "step's kernels; every step's outputs read back, its status checked and "
                       "its drawn tokens counted (-1 at n_accepted would be an undrawn token)"},
        "e2e_sync": {"value": aggregate(B * K * e2e_steps, world, e2e_sync_s),
                     "unit": UNIT, "api": "spec_verify_host, one blocking call per step"},
        "gpu_launches": timed_steps * sv.sv_kernels_per_call(B, K, V, dt_code),
        "clocks": clocks.summary(t_wall0, t_wall1),
        "cpu_baseline": cpu,
        "parity": parity,
        "parity_at_scale": load_parity_at_scale(),
        "workloads": subs,
    }
    print(json.dumps(line), flush=True)


def expand_sub(name: str):
    """Workload keys of a --sub entry ("sweep": the 20 cells of the acceptance sweep)."""
    if name == "sweep":
        return [f"sweep-k{k}-n{n:g}" for k in SWEEP_K for n in SWEEP_NOISE]
    return [name]


def load_parity_at_scale():
    """The committed summary of the last whole-batch parity run, if any."""
    path = os.path.join(ROOT, "profiles", "parity_at_scale.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"file": "profiles/parity_at_scale.json", "when": d.get("when"),
                "totals": d.get("totals")}
    except Exception:
        return None


SAMPLE_METRIC = "draft tokens sampled/sec (and achieved HBM GB/s, % of GB300 peak)"
SAMPLE_UNIT = "tokens/s"


def sample_sets(w, n_sets: int, base: int, pin: bool):
    """Draft rows [B*K, V] of the workload's steps, with seeded uniforms [B*K]."""
    out = []
    for i in range(n_sets):
        inp = make_inputs(w, step=base + i)
        g = torch.Generator().manual_seed(base + i)
        u = torch.rand(w.B * w.K, generator=g, dtype=torch.float32)
        lg = inp["draft"].reshape(w.B * w.K, w.V)
        out.append((lg.pin_memory() if pin else lg, u.pin_memory() if pin else u))
    return out


def sampler_launches(n: int, V: int) -> int:
    """Kernels of one sampler call: the single-pass sum kernel and the finish
    kernel."""
    return 2


def run_sampler_reference(args, w, world, rank):
    if rank != 0:
        return
    import oracle

    steps = max(1, args.steps)
    sets = sample_sets(w, min(4, steps), 30_000, pin=False)
    wide = [(lg.to(torch.float64).numpy(), u.to(torch.float64).numpy()) for lg, u in sets]
    for i in range(args.warmup):
        oracle.draft_sample(*wide[i % len(wide)], w.temperature)
    t0 = time.perf_counter()
    for i in range(steps):
        oracle.draft_sample(*wide[i % len(wide)], w.temperature)
    dt = time.perf_counter() - t0
    n = w.B * w.K
    value = steps * n / dt
    print(json.dumps({
        "impl": "reference", "op": "draft_sample", "metric": SAMPLE_METRIC, "value": value,
        "unit": SAMPLE_UNIT, "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + "-draft-rows", "rows": n, "V": w.V},
        "cpu_baseline": {"value": value, "unit": SAMPLE_UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{steps} calls over the {n} draft rows of {w.name} "
                                   f"(fp64 numpy oracle, 1 thread)"},
        "e2e": {"value": value, "unit": SAMPLE_UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_sampler(args, w, world, rank, local):
    """A step is one spec_draft_sample call over all B*K draft rows of one
    step of the workload (both of its kernels)."""
    import speculative_sampling_verification_gb300 as sv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sv.load_library(build=True)
    n, V, es = w.B * w.K, w.V, w.elem_bytes
    dt_code = sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32
    set_bytes = n * V * es
    n_sets = max(2, min(64, -(-2 * L2_BYTES // set_bytes) + 1))
    host = sample_sets(w, n_sets, 40_000 + 1000 * rank, pin=True)
    sets = [(lg.to(dev), u.to(dev)) for lg, u in host]
    outs = [torch.empty(n, dtype=torch.int32, device=dev) for _ in range(n_sets)]
    ws = torch.empty(max(256, sv.sv_sample_workspace_size(n, V, dt_code)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.Stream(dev)
    T = w.temperature

    def call(i):
        lg, u = sets[i % n_sets]
        rc = sv.spec_draft_sample(lg, u, T, outs[i % n_sets], ws, stream=stream)
        if rc != 0:
            raise RuntimeError(f"spec_draft_sample failed: {sv.sv_status_string(rc)}")

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        call(0)
    torch.cuda.synchronize()
    steps, warmup = args.steps, max(3, args.warmup)
    g_warm, g_timed = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm, stream=stream):
        for i in range(warmup):
            call(i)
    with torch.cuda.graph(g_timed, stream=stream):
        for i in range(steps):
            call(warmup + i)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    g_warm.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        g_timed.replay()
        end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = reduce_max(start.elapsed_time(end), world, dev)
    time.sleep(0.3)
    clocks.stop()
    status = sv.sv_read_device_status(ws, stream)
    toks = torch.stack(outs).cpu().numpy()
    if status != 0 or (toks < 0).any() or (toks >= V).any():
        raise RuntimeError(f"bad device status {status} or token out of range")

    # End to end: pinned host rows -> device, the call, tokens -> host.
    e2e_steps = args.e2e_steps or min(steps, 200)
    h_out = torch.empty(n, dtype=torch.int32).pin_memory()
    d_lg = torch.empty(n, V, dtype=sets[0][0].dtype, device=dev)
    d_u = torch.empty(n, dtype=torch.float32, device=dev)

    def host_call(i):
        lg, u = host[i % n_sets]
        with torch.cuda.stream(stream):
            d_lg.copy_(lg, non_blocking=True)
            d_u.copy_(u, non_blocking=True)
            rc = sv.spec_draft_sample(d_lg, d_u, T, outs[0], ws, stream=stream)
            if rc != 0:
                raise RuntimeError(f"spec_draft_sample: {rc}")
            h_out.copy_(outs[0], non_blocking=True)
        stream.synchronize()

    for i in range(3):
        host_call(i)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        host_call(i)
    e2e_s = reduce_max(time.perf_counter() - t0, world, dev)
    if rank != 0:
        return
    per_step_s = elapsed_ms / 1e3 / steps
    peak, peak_kind = load_peaks()
    achieved = set_bytes / per_step_s / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        wide = [(lg.to(torch.float64).numpy(), u.to(torch.float64).numpy()) for lg, u in host[:2]]
        t0, k = time.perf_counter(), 0
        while time.perf_counter() - t0 < 12.0 and k < 2000:
            oracle.draft_sample(*wide[k % len(wide)], T)
            k += 1
        dt = time.perf_counter() - t0
        cpu = {"value": k * n / dt, "unit": SAMPLE_UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{k} calls over the {n} draft rows of {w.name} in {dt:.1f} s "
                         f"(fp64 numpy oracle, 1 thread)"}
    print(json.dumps({
        "op": "draft_sample", "metric": SAMPLE_METRIC, "value": aggregate(n, world, per_step_s),
        "unit": SAMPLE_UNIT, "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": per_step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name + "-draft-rows", "rows": n, "V": V, "input_dtype": w.dtype,
                   "l2": f"inputs rotate over {n_sets} resident sets of {set_bytes / 1e6:.1f} MB",
                   "timing": "K calls in one CUDA graph, CUDA events on the launching stream"},
        "roofline": {"bound": "hbm", "kernel": "sample_sum_kernel and sample_finish_kernel (one sampler call)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                     "bytes_per_launch": set_bytes, "ms_per_launch": per_step_s * 1e3,
                     "bytes_basis": "N rows of V elements, once (both kernels' time)"},
        "e2e": {"value": aggregate(n * e2e_steps, world, e2e_s), "unit": SAMPLE_UNIT,
                "h2d_bytes_per_step": set_bytes + 4 * n, "d2h_bytes_per_step": 4 * n,
                "steps": e2e_steps},
        "gpu_launches": steps * sampler_launches(n, V),
        "clocks": clocks.summary(t_wall0, t_wall1),
        "cpu_baseline": cpu,
    }), flush=True)


def run_greedy_reference(args, w, world, rank):
    if rank != 0:
        return
    import oracle

    steps = max(1, args.steps)
    sets = [make_inputs(w, step=50_000 + i) for i in range(min(4, steps))]
    wide = [(s["target"].to(torch.float64).numpy(), s["tokens"].numpy()) for s in sets]
    for i in range(args.warmup):
        oracle.verify_greedy(*wide[i % len(wide)])
    t0 = time.perf_counter()
    for i in range(steps):
        oracle.verify_greedy(*wide[i % len(wide)])
    dt = time.perf_counter() - t0
    value = steps * w.B * w.K / dt
    print(json.dumps({
        "impl": "reference", "op": "greedy", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + "-greedy", "detail": w.describe()},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{steps} greedy steps of {w.name} (fp64 numpy oracle, 1 thread)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_greedy(args, w, world, rank, local):
    """A step is one spec_verify_greedy call over the B sequences of one step
    of the workload (its K+1 target rows; the draft rows are not read)."""
    import speculative_sampling_verification_gb300 as sv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sv.load_library(build=True)
    B, K, V, es = w.B, w.K, w.V, w.elem_bytes
    dt_code = sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32
    set_bytes = B * (K + 1) * V * es
    n_sets = max(2, min(64, -(-2 * L2_BYTES // set_bytes) + 1))
    host = []
    for i in range(n_sets):
        inp = make_inputs(w, step=60_000 + 1000 * rank + i)
        host.append((inp["target"].pin_memory(), inp["tokens"].to(torch.int32).pin_memory()))
    sets = [(t.to(dev), k.to(dev)) for t, k in host]
    outs = [(torch.empty(B, K + 1, dtype=torch.int32, device=dev),
             torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(n_sets)]
    ws = torch.empty(max(256, sv.sv_greedy_workspace_size(B, K, V, dt_code)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.Stream(dev)

    def call(i):
        t, k = sets[i % n_sets]
        o, n = outs[i % n_sets]
        rc = sv.spec_verify_greedy(t, k, o, n, ws, stream=stream)
        if rc != 0:
            raise RuntimeError(f"spec_verify_greedy failed: {sv.sv_status_string(rc)}")

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        call(0)
    torch.cuda.synchronize()
    steps, warmup = args.steps, max(3, args.warmup)
    g_warm, g_timed = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm, stream=stream):
        for i in range(warmup):
            call(i)
    with torch.cuda.graph(g_timed, stream=stream):
        for i in range(steps):
            call(warmup + i)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    g_warm.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        g_timed.replay()
        end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = reduce_max(start.elapsed_time(end), world, dev)
    time.sleep(0.3)
    clocks.stop()
    status = sv.sv_read_device_status(ws, stream)
    nacc_all = torch.stack([n for _, n in outs]).cpu().numpy()
    if status != 0 or (nacc_all < 0).any() or (nacc_all > K).any():
        raise RuntimeError(f"bad device status {status} or n_accepted out of range")

    e2e_steps = args.e2e_steps or min(steps, 200)
    d_t = torch.empty_like(sets[0][0])
    d_k = torch.empty_like(sets[0][1])
    h_out = torch.empty(B, K + 1, dtype=torch.int32).pin_memory()
    h_n = torch.empty(B, dtype=torch.int32).pin_memory()

    def host_call(i):
        t, k = host[i % n_sets]
        with torch.cuda.stream(stream):
            d_t.copy_(t, non_blocking=True)
            d_k.copy_(k, non_blocking=True)
            rc = sv.spec_verify_greedy(d_t, d_k, outs[0][0], outs[0][1], ws, stream=stream)
            if rc != 0:
                raise RuntimeError(f"spec_verify_greedy: {rc}")
            h_out.copy_(outs[0][0], non_blocking=True)
            h_n.copy_(outs[0][1], non_blocking=True)
        stream.synchronize()

    for i in range(3):
        host_call(i)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        host_call(i)
    e2e_s = reduce_max(time.perf_counter() - t0, world, dev)
    if rank != 0:
        return
    per_step_s = elapsed_ms / 1e3 / steps
    peak, peak_kind = load_peaks()
    achieved = set_bytes / per_step_s / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        wide = [(t.to(torch.float64).numpy(), k.to(torch.int64).numpy()) for t, k in host[:2]]
        t0, k = time.perf_counter(), 0
        while time.perf_counter() - t0 < 12.0 and k < 5000:
            oracle.verify_greedy(*wide[k % len(wide)])
            k += 1
        dt = time.perf_counter() - t0
        cpu = {"value": k * B * K / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{k} greedy steps of {w.name} in {dt:.1f} s (fp64 numpy oracle, 1 thread)"}
    print(json.dumps({
        "op": "greedy", "metric": METRIC, "value": aggregate(B * K, world, per_step_s),
        "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": per_step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name + "-greedy", "detail": w.describe(),
                   "l2": f"inputs rotate over {n_sets} resident sets of {set_bytes / 1e6:.1f} MB",
                   "timing": "K calls in one CUDA graph, CUDA events on the launching stream"},
        "roofline": {"bound": "hbm", "kernel": "greedy_kernel (one launch per call)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                     "bytes_per_launch": set_bytes, "ms_per_launch": per_step_s * 1e3,
                     "bytes_basis": "B(K+1) target rows of V elements, once (call time)"},
        "e2e": {"value": aggregate(B * K * e2e_steps, world, e2e_s), "unit": UNIT,
                "h2d_bytes_per_step": set_bytes + 4 * B * K,
                "d2h_bytes_per_step": 4 * B * (K + 2), "steps": e2e_steps},
        "gpu_launches": steps,
        "clocks": clocks.summary(t_wall0, t_wall1),
        "cpu_baseline": cpu,
    }), flush=True)


def _filter_mode(args, w):
    """(label, input maker, oracle call, workload suffix) of --op topk / topp.
    The oracle is imported only when its call runs (the CPU baseline and the
    reference arm)."""

    def ref(*a):
        import oracle

        if args.op == "topk":
            return oracle.verify_topk(*a, w.temperature, args.top_k)
        return oracle.verify_topp(*a, w.temperature, args.top_p)

    if args.op == "topk":
        kk = args.top_k
        return f"top-{kk}", lambda step: make_topk_inputs(w, kk, step=step), ref, f"-top{kk}"
    pp = args.top_p
    return f"top-p {pp:g}", lambda step: make_topp_inputs(w, pp, step=step), ref, f"-topp{pp:g}"


def run_filter_reference(args, w, world, rank):
    if rank != 0:
        return
    label, make, ref, suffix = _filter_mode(args, w)
    steps = max(1, args.steps)
    sets = [make(70_000 + i) for i in range(min(2, steps))]
    wide = [tuple(s[x].to(torch.float64).numpy() for x in ("target", "draft"))
            + (s["tokens"].numpy(), s["uniforms"].to(torch.float64).numpy()) for s in sets]
    for i in range(args.warmup):
        ref(*wide[i % len(wide)])
    t0 = time.perf_counter()
    for i in range(steps):
        ref(*wide[i % len(wide)])
    dt = time.perf_counter() - t0
    value = steps * w.B * w.K / dt
    print(json.dumps({
        "impl": "reference", "op": args.op, "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name + suffix, "detail": w.describe()},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{steps} {label} steps of {w.name} (fp64 numpy oracle, 1 thread)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_filter(args, w, world, rank, local):
    """A step is one filtered verification call over the B sequences of one
    step of the workload. topk: the row selection kernel over all 2K+1 rows,
    then the verification kernel on the kept entries. topp: the per-row cut
    kernel (which also leaves each row's kept mass), the scan, then the draw
    with the kept sets applied on load."""
    import speculative_sampling_verification_gb300 as sv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sv.load_library(build=True)
    label, make, ref, suffix = _filter_mode(args, w)
    kk, pp = args.top_k, args.top_p
    B, K, V, es = w.B, w.K, w.V, w.elem_bytes
    dt_code = sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32
    set_bytes = B * (2 * K + 1) * V * es
    n_sets = max(2, min(64, -(-2 * L2_BYTES // set_bytes) + 1))
    names = ("target", "draft", "tokens", "uniforms")
    host = []
    for i in range(n_sets):
        inp = make(80_000 + 1000 * rank + i)
        host.append(tuple(inp[x].pin_memory() for x in names))
    sets = [tuple(t.to(dev) for t in h) for h in host]
    outs = [(torch.empty(B, K + 1, dtype=torch.int32, device=dev),
             torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(n_sets)]
    if args.op == "topk":
        ws_bytes = sv.sv_topk_workspace_size(B, K, V, dt_code, kk)
        launches = 2
        kernel = "topk_select_kernel + topk_verify_kernel (call time)"
    else:
        ws_bytes = sv.sv_topp_workspace_size(B, K, V, dt_code)
        launches = sv.sv_topp_kernels_per_call(B, K, V, dt_code)
        kernel = "topp_cluster_kernel + scan_kernel + the masked draw (call time)"
    ws = torch.empty(max(256, ws_bytes), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def call(i, tensors=None, o=None):
        t = tensors or sets[i % n_sets]
        o = o or outs[i % n_sets]
        if args.op == "topk":
            rc = sv.spec_verify_topk(*t, w.temperature, kk, o[0], o[1], ws, stream=stream)
        else:
            rc = sv.spec_verify_topp(*t, w.temperature, pp, o[0], o[1], ws, stream=stream)
        if rc != 0:
            raise RuntimeError(f"{args.op} call failed: {sv.sv_status_string(rc)}")

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        call(0)
    torch.cuda.synchronize()
    steps, warmup = args.steps, max(3, args.warmup)
    g_warm, g_timed = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm, stream=stream):
        for i in range(warmup):
            call(i)
    with torch.cuda.graph(g_timed, stream=stream):
        for i in range(steps):
            call(warmup + i)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    g_warm.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        g_timed.replay()
        end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = reduce_max(start.elapsed_time(end), world, dev)
    time.sleep(0.3)
    clocks.stop()
    status = sv.sv_read_device_status(ws, stream)
    nacc_all = torch.stack([n for _, n in outs]).cpu().numpy()
    if status != 0 or (nacc_all < 0).any() or (nacc_all > K).any():
        raise RuntimeError(f"bad device status {status} or n_accepted out of range")

    e2e_steps = args.e2e_steps or min(steps, 200)
    dev_in = tuple(torch.empty_like(t) for t in sets[0])
    h_out = torch.empty(B, K + 1, dtype=torch.int32).pin_memory()
    h_n = torch.empty(B, dtype=torch.int32).pin_memory()

    def host_call(i):
        h = host[i % n_sets]
        with torch.cuda.stream(stream):
            for d, x in zip(dev_in, h):
                d.copy_(x, non_blocking=True)
            call(0, dev_in, outs[0])
            h_out.copy_(outs[0][0], non_blocking=True)
            h_n.copy_(outs[0][1], non_blocking=True)
        stream.synchronize()

    for i in range(3):
        host_call(i)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        host_call(i)
    e2e_s = reduce_max(time.perf_counter() - t0, world, dev)
    if rank != 0:
        return
    per_step_s = elapsed_ms / 1e3 / steps
    peak, peak_kind = load_peaks()
    achieved = set_bytes / per_step_s / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle

        wide = [tuple(x.to(torch.float64).numpy() for x in h[:2]) + (h[2].to(torch.int64).numpy(),
                h[3].to(torch.float64).numpy()) for h in host[:2]]
        t0, n = time.perf_counter(), 0
        while time.perf_counter() - t0 < 12.0 and n < 5000:
            ref(*wide[n % len(wide)])
            n += 1
        dt = time.perf_counter() - t0
        cpu = {"value": n * B * K / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{n} {label} steps of {w.name} in {dt:.1f} s (fp64 numpy oracle, 1 thread)"}
    in_bytes = sum(t.numel() * t.element_size() for t in host[0])
    print(json.dumps({
        "op": args.op, "metric": METRIC, "value": aggregate(B * K, world, per_step_s),
        "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": per_step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name + suffix, "detail": w.describe(),
                   ("top_k" if args.op == "topk" else "top_p"): kk if args.op == "topk" else pp,
                   "l2": f"inputs rotate over {n_sets} resident sets of {set_bytes / 1e6:.1f} MB",
                   "timing": "K calls in one CUDA graph, CUDA events on the launching stream"},
        "roofline": {"bound": "hbm", "kernel": kernel,
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                     "bytes_per_launch": set_bytes, "ms_per_launch": per_step_s * 1e3,
                     "bytes_basis": "B(2K+1) rows of V elements, once (the whole call's time)"},
        "e2e": {"value": aggregate(B * K * e2e_steps, world, e2e_s), "unit": UNIT,
                "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": 4 * B * (K + 2),
                "steps": e2e_steps},
        "gpu_launches": steps * launches,
        "clocks": clocks.summary(t_wall0, t_wall1),
        "cpu_baseline": cpu,
    }), flush=True)


LMH_METRIC = ("scored rows/sec of the fused projection + row statistics (and tensor "
              "TFLOP/s, % of GB300 bf16 peak)")
LMH_UNIT = "rows/s"


def lmh_oracle_sample(w, inp, rows):
    """The oracle's statistics of `rows` (a bounded sample) and its time."""
    import oracle

    h = inp["hidden"][rows].cpu().to(torch.float64).numpy()
    wt = inp["weight"].cpu().to(torch.float64).numpy()
    tok = inp["tokens"][rows].cpu().numpy()
    t0 = time.perf_counter()
    ref = oracle.lm_head_stats(h, wt, w.temperature, tok)
    dt = time.perf_counter() - t0
    return ref, dt, h, wt, tok


def run_lmhead_reference(args, world, rank):
    if rank != 0:
        return
    from synthetic import LMHEAD_WORKLOADS, make_lmhead_inputs

    w = LMHEAD_WORKLOADS["lmhead-c3"]
    inp = make_lmhead_inputs(w.N, w.D, w.V, w.logit_std, w.seed, device="cpu")
    rows = list(range(4))
    steps = max(1, args.steps)
    for _ in range(max(1, args.warmup)):
        lmh_oracle_sample(w, inp, rows)
    dt = 0.0
    for _ in range(steps):
        dt += lmh_oracle_sample(w, inp, rows)[1]
    value = steps * len(rows) / dt
    print(json.dumps({
        "impl": "reference", "op": "lmhead", "metric": LMH_METRIC, "value": value,
        "unit": LMH_UNIT, "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "N": w.N, "D": w.D, "V": w.V},
        "cpu_baseline": {"value": value, "unit": LMH_UNIT, "cores": host_cores(),
                         "kind": "oracle",
                         "sample": f"each step: the oracle (numpy fp64 matmul, its BLAS on the "
                                   f"host cores) over {len(rows)} rows of {w.name}",
                         "host": host_info()},
        "e2e": {"value": value, "unit": LMH_UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_lmhead(args, world, rank, local):
    """A step is one sv_lmhead_stats call over the N scored rows: the logits of
    the N x D hidden states against the V x D projection on the tensor cores,
    reduced to row statistics on chip."""
    import speculative_sampling_verification_gb300 as sv
    from synthetic import LMHEAD_WORKLOADS, make_lmhead_inputs

    w = LMHEAD_WORKLOADS["lmhead-c3"]
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    sv.load_library(build=True)
    inp = make_lmhead_inputs(w.N, w.D, w.V, w.logit_std, w.seed + rank, device=dev)
    ws = torch.empty(sv.sv_lmhead_workspace_size(w.N, w.D, w.V), dtype=torch.uint8, device=dev)
    rm = torch.empty(w.N, dtype=torch.float64, device=dev)
    lse = torch.empty(w.N, dtype=torch.float64, device=dev)
    at = torch.empty(w.N, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def call():
        rc = sv.sv_lmhead_stats(inp["hidden"], inp["weight"], inp["tokens"], w.temperature, rm,
                                lse, at, ws, stream=stream)
        if rc != 0:
            raise RuntimeError(f"sv_lmhead_stats: {sv.sv_status_string(rc)}")

    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    steps, warmup = max(1, args.steps), max(3, args.warmup)
    g_warm, g = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm, stream=stream):
        for _ in range(warmup):
            call()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(steps):
            call()
    g_warm.replay()
    torch.cuda.synchronize()
    t_est = time.perf_counter()
    g.replay()
    torch.cuda.synchronize()
    est = max(time.perf_counter() - t_est, 1e-4)
    reps = max(1, int(np.ceil(args.min_seconds / est)))
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    time.sleep(0.3)
    clocks.stop()
    if sv.sv_read_device_status(ws, stream) != 0:
        raise RuntimeError("bad device status")
    elapsed_ms = reduce_max(start.elapsed_time(end), world, dev)
    per_s = elapsed_ms / 1e3 / (steps * reps)

    # End to end: the hidden states (the model's activations) copied from
    # pinned host memory every step and the three outputs read back; the
    # projection weights are model parameters, resident in HBM.
    h_host = inp["hidden"].cpu().pin_memory()
    h_dev = torch.empty_like(inp["hidden"])
    o_host = [torch.empty(w.N, dtype=t.dtype).pin_memory() for t in (rm, lse, at)]
    e2e_steps = max(8, min(100, int(0.5 / per_s)))

    def host_step():
        with torch.cuda.stream(stream):
            h_dev.copy_(h_host, non_blocking=True)
            rc = sv.sv_lmhead_stats(h_dev, inp["weight"], inp["tokens"], w.temperature, rm, lse,
                                    at, ws, stream=stream)
            if rc != 0:
                raise RuntimeError(sv.sv_status_string(rc))
            for o, d in zip(o_host, (rm, lse, at)):
                o.copy_(d, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        host_step()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        host_step()
    e2e_s = reduce_max(time.perf_counter() - t0, world, dev)
    if rank != 0:
        return
    tflops = w.flops() / per_s / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        peak, kind = 1900.0, "fallback"
    cpu = parity = None
    if world == 1 and not args.no_cpu_baseline:
        rows = [0, 1, 2, 3]
        ref, dt, h, wt, tok = lmh_oracle_sample(w, inp, rows)
        cpu = {"value": len(rows) / dt, "unit": LMH_UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"{len(rows)} rows of {w.name} in {dt:.2f} s (numpy fp64 matmul, its "
                         f"BLAS on the host cores)", "host": host_info()}
        bound = (np.abs(h) @ np.abs(wt).T * 2.0 ** -20).max(axis=1) / np.float32(w.temperature)
        g_rm, g_lse = rm[rows].cpu().numpy(), lse[rows].cpu().numpy()
        parity = {"rows": len(rows),
                  "row_max_within_bound": bool(np.all(np.abs(g_rm - ref.row_max) <= bound)),
                  "lse_within_bound": bool(np.all(np.abs(g_lse - ref.lse)
                                                  <= bound + 1e-6 * np.abs(ref.lse))),
                  "max_abs_diff_lse": float(np.max(np.abs(g_lse - ref.lse))),
                  "bound": "2^-20 sum_d |h_d w_vd| / T per row (fp32 accumulation)"}
    print(json.dumps({
        "op": "lmhead", "metric": LMH_METRIC, "value": aggregate(w.N, world, per_s),
        "unit": LMH_UNIT, "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": per_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "N": w.N, "D": w.D, "V": w.V},
        "timing": {"repeats": reps, "timed_steps": steps * reps,
                   "l2": f"the {w.weight_bytes() / 1e9:.2f} GB projection is read once per "
                         f"step, more than L2"},
        "tflops": tflops,
        "roofline": {"bound": "tensor", "kernel": "lmhead_kernel (tcgen05 bf16 GEMM + on-chip "
                     "row statistics) with its combine kernel", "achieved": tflops, "peak": peak,
                     "unit": "TFLOP/s", "frac": tflops / peak,
                     "peak_kind": f"{kind} cuBLAS bf16 (burst)", "traffic": None,
                     "flops_per_launch": w.flops(), "ms_per_launch": per_s * 1e3},
        "e2e": {"value": aggregate(w.N * e2e_steps, world, e2e_s), "unit": LMH_UNIT,
                "h2d_bytes_per_step": w.N * w.D * 2, "d2h_bytes_per_step": w.N * 20,
                "steps": e2e_steps, "api": "sv_lmhead_stats with the hidden states copied "
                "from pinned host memory every step; weights resident"},
        "gpu_launches": steps * reps * 2,
        "clocks": clocks.summary(t_wall0, t_wall1),
        "cpu_baseline": cpu,
        "parity": parity,
    }), flush=True)


def main():
    args = parse()
    w = get_workload(args.config)
    world, rank, local = dist_setup(args)
    try:
        if args.op == "lmhead":
            if args.impl == "reference":
                run_lmhead_reference(args, world, rank)
            else:
                run_lmhead(args, world, rank, local)
        elif args.op == "draft_sample":
            if args.impl == "reference":
                run_sampler_reference(args, w, world, rank)
            else:
                run_sampler(args, w, world, rank, local)
        elif args.op == "greedy":
            if args.impl == "reference":
                run_greedy_reference(args, w, world, rank)
            else:
                run_greedy(args, w, world, rank, local)
        elif args.op in ("topk", "topp"):
            if args.impl == "reference":
                run_filter_reference(args, w, world, rank)
            else:
                run_filter(args, w, world, rank, local)
        elif args.impl == "reference":
            run_reference(args, w, world, rank)
        else:
            run_ours(args, w, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
