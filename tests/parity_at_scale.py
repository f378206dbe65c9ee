"""Parity at scale: the CUDA path against the fp64 oracle over whole batches.

    python -m tests.parity_at_scale [--configs c2,c3,c4,sweep] [--min-decisions 100000]
                                    [--min-decisions-cell 10000] [--out FILE]
                                    [--op verify|topk|topp|greedy|sample] [--top-k 50]
                                    [--top-p 0.9]

For every workload, steps are drawn on the GPU by the batched seeded
generator, verified there through the C ABI (spec_verify_debug, whole batch),
and every sequence of every step is verified again by the fp64 oracle on the
host cores (a spawn pool, one process per core, fed through .npy files). Steps
are added until the oracle has taken at least --min-decisions decisions (for
each of the 20 cells of the acceptance sweep, --min-decisions-cell).

With --op topk or topp the filtered verification (spec_verify_topk /
spec_verify_topp) is checked against verify_topk / verify_topp the same way;
for the nucleus, a row whose kept count differs from the oracle's is allowed
only where top_p lies within 1e-9 of the oracle's cumulative sums at its cut
(`cut_excused_rows`; their sequences' decisions are not compared), as in the
GPU tests. With --op greedy, greedy verification must match verify_greedy
exactly (its decisions are integer comparisons). With --op sample, the draft
sampler draws one token per draft row (the uniforms of the first K draws of
each sequence) and is held to the verification draw's margin rule against
draft_sample. These paths export no intermediates.

Per workload the record holds the sequences and decisions checked, the
decisions whose uniform lies within 1e-6 of the oracle's threshold
(`near_threshold`: a property of the inputs), the differences at such
decisions (`excused_differences`), and any other difference
(`unexcused_differences`, which must be 0). It also holds the largest
relative differences of the intermediate values (per-row log-sum-exp and
maximum, thresholds, ratios q/p, drawn token's probability) and how many
exceed their tolerance. The parity bar is the verification step's: no
unexcused difference, and excused differences below 1e-5 of the decisions.
"""

from __future__ import annotations

import argparse
import collections
import json
import os
import shutil
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from tests import _parity  # noqa: E402

# Relative tolerances of the intermediate values (those of tests/test_gpu_parity.py).
TOL = {"row_lse": 1e-5, "thresholds": 1e-5, "ratios": 1e-5, "row_max": 1e-12,
       "sample_prob": 1e-8}
MAX_EXCUSED_RATE = 1e-5


# ---------------------------------------------------------------- oracle side (spawned workers)

def _load(paths):
    t, d, k, u = (np.load(p, mmap_mode="r") for p in paths)
    if t.dtype == np.uint16:  # bf16 bit patterns: widen exactly to fp32
        t = (t.astype(np.uint32) << np.uint32(16)).view(np.float32)
        d = (d.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return (np.ascontiguousarray(t), np.ascontiguousarray(d), np.asarray(k).astype(np.int64),
            np.asarray(u))


CUT_MARGIN = 1e-9


def oracle_job(job):
    """The fp64 oracle over the sequences stored in `paths` (a worker process)."""
    import oracle

    paths, temperature, op, param = job
    if op == "topk":
        return oracle.verify_topk(*_load(paths), temperature, param)
    if op == "topp":
        return oracle.verify_topp(*_load(paths), temperature, param)
    if op == "greedy":
        t, _, k, _ = _load(paths)
        return oracle.verify_greedy(t, k)
    if op == "sample":
        _, d, _, u = _load(paths)
        n, K, V = d.shape
        return oracle.draft_sample(d.reshape(n * K, V), np.ascontiguousarray(u[:, :K]).reshape(-1),
                                   temperature)
    return oracle.verify(*_load(paths), temperature)


def compare_greedy(out, nacc, ref) -> _parity.ParityReport:
    """Greedy verification: the outputs must be identical (each decision is an
    exact comparison of integer argmaxes)."""
    out, nacc = np.asarray(out).astype(np.int64), np.asarray(nacc).astype(np.int64)
    ok = ref.status == 0
    rep = _parity.ParityReport(sequences=len(nacc),
                               decisions=int(np.sum(ref.n_accepted[ok] + 1)))
    for b in np.nonzero((out != ref.out_tokens).any(axis=1) | (nacc != ref.n_accepted))[0]:
        rep.failures.append((int(b), "greedy", out[b].tolist(), ref.out_tokens[b].tolist()))
    return rep


def compare_sample(tokens, ref) -> _parity.ParityReport:
    """Draft sampling: one draw per row, the margin rule of the verification's
    draw (a differing token is tolerated only within MARGIN of its CDF ends)."""
    tokens = np.asarray(tokens).astype(np.int64).reshape(-1)
    ok = ref.status == 0
    rep = _parity.ParityReport(sequences=len(tokens), decisions=int(ok.sum()))
    rep.near_threshold = int(np.sum(ref.sample_margin[ok] < _parity.MARGIN))
    bad = (~ok) & (tokens != -1)
    diff = ok & (tokens != ref.tokens)
    excused = diff & (ref.sample_margin < _parity.MARGIN)
    rep.excused = int(excused.sum())
    for i in np.nonzero(bad | (diff & ~excused))[0][:50]:
        rep.failures.append((int(i), "draw", int(tokens[i]), int(ref.tokens[i]),
                             float(ref.sample_margin[i])))
    return rep


def _subset(res, rows):
    import dataclasses

    return type(res)(*[getattr(res, f.name)[rows] for f in dataclasses.fields(res)])


# ---------------------------------------------------------------- GPU side

def _to_np(t):
    import torch

    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _scratch_dir() -> str:
    try:
        if shutil.disk_usage("/dev/shm").free > (24 << 30):
            return "/dev/shm"
    except Exception:
        pass
    return tempfile.gettempdir()


def _rel_err(got, ref):
    """Largest relative difference over entries finite on both sides, and the
    count of entries whose infinities or NaNs differ."""
    got, ref = np.asarray(got, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(got) & np.isfinite(ref)
    mismatch = int(np.sum(~fin & ~((got == ref) | (np.isnan(got) & np.isnan(ref)))))
    if not fin.any():
        return 0.0, mismatch
    den = np.maximum(np.abs(ref[fin]), 1e-300)
    return float(np.max(np.abs(got[fin] - ref[fin]) / den)), mismatch


class Intermediates:
    def __init__(self):
        self.max_rel = {k: 0.0 for k in TOL}
        self.over = {k: 0 for k in TOL}

    def add(self, dbg, ref, seqs):
        ok = ref.status == 0
        pairs = {"row_lse": ref.lse, "thresholds": ref.thresholds, "ratios": ref.ratios,
                 "row_max": ref.row_max, "sample_prob": ref.sample_prob}
        for k, r in pairs.items():
            g = dbg[k][seqs][ok]
            r = r[ok]
            # the tests' absolute floors: thresholds 1e-9, lse 1e-6, probabilities 1e-15
            floor = {"row_lse": 1e-6, "thresholds": 1e-9, "sample_prob": 1e-15}.get(k, 0.0)
            err, bad = _rel_err(g, r)
            self.max_rel[k] = max(self.max_rel[k], err)
            fin = np.isfinite(g) & np.isfinite(r)
            over = np.abs(g[fin] - r[fin]) > TOL[k] * np.abs(r[fin]) + floor
            self.over[k] += int(over.sum()) + bad

    def as_dict(self):
        return {"tolerance": TOL, "max_rel_diff": self.max_rel, "over_tolerance": self.over}


def check_workload(sv, w, dev, pool, workers, tmp, min_decisions, max_steps=100_000,
                   step_base=7000, depth=None, log=print, op="verify", param=None):
    """Whole-batch parity of workload `w` (for `op`): returns its record."""
    import torch

    from synthetic import make_batch

    B, K, V = w.B, w.K, w.V
    dt = sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32
    ws = sv.new_workspace(B, K, V, dt, dev) if op == "verify" else None
    cut_rows = cut_bad = 0
    per_seq = (2 * K + 1) * V * 25e-9
    per = max(1, min(B, int(0.25 / per_seq)))
    chunks = [list(range(s, min(B, s + per))) for s in range(0, B, per)]
    depth = depth or max(2, -(-2 * workers // len(chunks)))
    rep = _parity.ParityReport()
    inter = Intermediates()
    pending = collections.deque()
    statuses = 0
    step = 0
    need_steps = max_steps
    t0 = time.time()

    def settle(item):
        nonlocal need_steps, cut_rows, cut_bad
        s, jobs, out, nacc, tokens, dbg, files = item
        for seqs, res in jobs:
            ref = res.get()
            if op == "topp":
                kept = dbg["kept"][seqs]
                mism = kept != ref.kept
                cut_rows += int(mism.sum())
                cut_bad += int(np.sum(mism & ~(ref.cut_margin < CUT_MARGIN)))
                ok = ~mism.any(axis=1)
                sub = np.asarray(seqs)[ok]
                rep.add(_parity.compare(out[sub], nacc[sub], _subset(ref.result, ok), tokens[sub]))
            elif op == "topk":
                rep.add(_parity.compare(out[seqs], nacc[seqs], ref, tokens[seqs]))
            elif op == "greedy":
                rep.add(compare_greedy(out[seqs], nacc[seqs], ref))
            elif op == "sample":
                rep.add(compare_sample(out[seqs], ref))
            else:
                rep.add(_parity.compare(out[seqs], nacc[seqs], ref, tokens[seqs]))
                inter.add(dbg, ref, seqs)
        for f in files:
            try:
                os.remove(f)
            except OSError:
                pass
        if need_steps == max_steps and rep.decisions:
            done = s - step_base + 1
            need_steps = min(max_steps,
                             int(np.ceil(1.08 * min_decisions * done / rep.decisions)))

    while True:
        if step >= need_steps:
            while pending:
                settle(pending.popleft())
            if rep.decisions >= min_decisions or step >= max_steps:
                break
            need_steps = min(max_steps, step + int(np.ceil(
                1.1 * (min_decisions - rep.decisions) * step / max(1, rep.decisions))) + 1)
        inp = make_batch(w, step=step_base + step, device=dev)
        args = (inp["target"], inp["draft"], inp["tokens"], inp["uniforms"], inp["temperature"])
        if op == "topk":
            out, nacc = sv.verify_topk(*args, param)
            dbg_np = {}
        elif op == "topp":
            out, nacc, kept = sv.verify_topp(*args, param)
            dbg_np = {"kept": kept.cpu().numpy()}
        elif op == "greedy":
            out, nacc = sv.verify_greedy(inp["target"], inp["tokens"])
            dbg_np = {}
        elif op == "sample":
            u = inp["uniforms"][:, :K].contiguous().reshape(-1)
            tok = sv.draft_sample(inp["draft"].reshape(B * K, V), u, inp["temperature"])
            out, nacc = tok.reshape(B, K), torch.zeros(B, dtype=torch.int32, device=dev)
            dbg_np = {}
        else:
            out, nacc, dbg = sv.verify(*args, workspace=ws, debug=True)
            dbg_np = {k: v.cpu().numpy() for k, v in dbg.items() if k != "workspace"}
            del dbg
        torch.cuda.synchronize()
        if ws is not None:
            statuses |= sv.sv_read_device_status(ws)
        files, jobs = [], []
        for ci, seqs in enumerate(chunks):
            idx = torch.as_tensor(seqs, device=dev)
            paths = []
            for k in ("target", "draft", "tokens", "uniforms"):
                p = os.path.join(tmp, f"{w.name}-{step}-{ci}-{k}.npy")
                np.save(p, _to_np(inp[k].index_select(0, idx)))
                paths.append(p)
            files += paths
            jobs.append((seqs, pool.apply_async(oracle_job,
                                                ((paths, inp["temperature"], op, param),))))
        pending.append((step_base + step, jobs, out.cpu().numpy(), nacc.cpu().numpy(),
                        inp["tokens"].cpu().numpy(), dbg_np, files))
        del inp, out, nacc
        step += 1
        while pending and (len(pending) > depth or all(r.ready() for _, r in pending[0][1])):
            settle(pending.popleft())
    dt = time.time() - t0
    d = rep.as_dict()
    d.update({"workload": w.name, "op": op, "steps": step, "device_status": statuses,
              "excused_rate": rep.excused / max(1, rep.decisions),
              "intermediates": inter.as_dict() if op == "verify" else None,
              "seconds": round(dt, 1), "failures": [str(f)[:300] for f in rep.failures[:5]]})
    if op == "topk":
        d["top_k"] = param
    if op == "topp":
        d.update({"top_p": param, "cut_excused_rows": cut_rows - cut_bad,
                  "cut_unexcused_rows": cut_bad})
    d["pass"] = (not rep.failures and statuses == 0 and rep.excused <= MAX_EXCUSED_RATE
                 * rep.decisions and not any(inter.over.values()) and cut_bad == 0)
    log(json.dumps({k: d[k] for k in ("workload", "steps", "sequences", "decisions",
                                      "near_threshold", "excused_differences",
                                      "unexcused_differences", "seconds", "pass")}))
    del ws
    torch.cuda.empty_cache()
    return d


def workload_list(configs: str):
    from synthetic import SWEEP_K, SWEEP_NOISE, get_workload

    out = []
    for name in configs.split(","):
        if name == "sweep":
            out += [(get_workload(f"sweep-k{k}-n{n:g}"), True) for k in SWEEP_K
                    for n in SWEEP_NOISE]
        else:
            out.append((get_workload(name), False))
    return out


def run(configs="c2,c3,c4,sweep", min_decisions=100_000, min_decisions_cell=10_000,
        workers=None, out=None, log=print, op="verify", top_k=50, top_p=0.9):
    import multiprocessing as mp

    workers = workers or max(1, len(os.sched_getaffinity(0)) - 1)
    pool = mp.get_context("spawn").Pool(workers)  # before any CUDA work
    tmp = tempfile.mkdtemp(prefix="sv-parity-", dir=_scratch_dir())
    try:
        import torch

        import speculative_sampling_verification_gb300 as sv

        sv.load_library(build=True)
        dev = torch.device("cuda:0")
        records = []
        for w, cell in workload_list(configs):
            records.append(check_workload(sv, w, dev, pool, workers, tmp,
                                          min_decisions_cell if cell else min_decisions,
                                          log=log, op=op,
                                          param={"topk": top_k, "topp": top_p}.get(op)))
    finally:
        pool.terminate()
        pool.join()
        shutil.rmtree(tmp, ignore_errors=True)
    tot = _parity.ParityReport()
    for r in records:
        tot.add(_parity.ParityReport(r["sequences"], r["decisions"], r["excused_differences"],
                                     r["near_threshold"]))
    totals = tot.as_dict()
    totals["unexcused_differences"] = sum(r["unexcused_differences"] for r in records)
    totals["excused_rate"] = tot.excused / max(1, tot.decisions)
    summary = {"when": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime()), "op": op,
               "command": "python -m tests.parity_at_scale " + " ".join(sys.argv[1:]),
               "margin": _parity.MARGIN, "max_excused_rate": MAX_EXCUSED_RATE,
               "oracle_workers": workers, "totals": totals,
               "pass": all(r["pass"] for r in records), "workloads": records}
    if out:
        with open(out, "w") as f:
            json.dump(summary, f, indent=1)
    return summary


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--configs", default="c2,c3,c4,sweep")
    ap.add_argument("--min-decisions", type=int, default=100_000)
    ap.add_argument("--min-decisions-cell", type=int, default=10_000)
    ap.add_argument("--workers", type=int, default=None)
    ap.add_argument("--out", default=None)
    ap.add_argument("--op", choices=["verify", "topk", "topp", "greedy", "sample"],
                    default="verify")
    ap.add_argument("--top-k", type=int, default=50)
    ap.add_argument("--top-p", type=float, default=0.9)
    a = ap.parse_args()
    s = run(a.configs, a.min_decisions, a.min_decisions_cell, a.workers, a.out, op=a.op,
            top_k=a.top_k, top_p=a.top_p)
    print(json.dumps({"pass": s["pass"], "totals": s["totals"]}))
    sys.exit(0 if s["pass"] else 1)


if __name__ == "__main__":
    main()
