#!/usr/bin/env python3
"""Benchmark of the fused Indexer-TopK (LiteTopK-style) on one GB300.

Workload (default): one 8192-query prefill chunk at 1M context -- queries at
positions 1040384..1048575, S = 1048576 keys, H = 64, d = 128, k = 2048,
bf16 q/k, fp32 w -- with the previous chunk's top-3k as the sample.  A step is
one pass of the whole path: the previous-chunk sample (ltk_make_sample) plus
the fused Sample -> Filter -> Select call (ltk_indexer_topk).

Printed (rank 0, one JSON line): scored (visible) query-key pairs/s over the
timed steps, ms per chunk, the score kernel's roofline fraction (CUDA events
around that kernel on its launch stream, inside the timed region), the
end-to-end number through the host-buffer C-ABI call, SM clocks sampled during
the timed region, the same-GPU decoupled baseline, and the CPU oracle baseline.

``--impl reference`` times the CPU oracle (the plain definition: fp64 scores
and a full sort) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import signal
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "scored query-key pairs/s and ms per 8K-query chunk at 1M ctx, k=2048 (1 GB300)"
UNIT = "pairs/s"
FLOP_PER_PAIR = 2 * 64 * 128          # H * d multiply-adds per visible pair
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0                    # nominal dense ratio (4.5 / 2.25 PFLOP/s)

WORKLOADS = {
    # name: (current chunk, previous chunk)
    "1m": ("1m", "1m_prev"),
    "256k": ("256k", "256k_prev"),
    "128k": ("128k_chunk2", "128k_chunk1"),
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ltk", "reference"], default="ltk")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["retrieval", "decode"], default="1m")
    ap.add_argument("--dtype", choices=["bf16", "fp8"], default="bf16")
    ap.add_argument("--queries", type=int, default=0,
                    help="run only the first N queries of the chunk (profiling a single wave)")
    ap.add_argument("--cpu-queries", type=int, default=64,
                    help="queries of the chunk the CPU oracle baseline scores")
    ap.add_argument("--ref-queries", type=int, default=2,
                    help="queries per step of the reference (oracle) arm")
    ap.add_argument("--k", type=int, default=0,
                    help="retrieval workload: k (default 1000; the pages sweep 1024..8192)")
    ap.add_argument("--corpus", type=int, default=0,
                    help="retrieval workload: corpus rows (default 8388608; smaller for profiling)")
    ap.add_argument("--engine", choices=["auto", "tensor", "cuda"], default="auto",
                    help="scorer: tensor cores (default where the shape allows) or CUDA cores")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-decoupled", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="1M bf16 run only: skip the e4m3, 256K and decode sub-records")
    ap.add_argument("--cpu-single-queries", type=int, default=16,
                    help="queries of the chunk the single-threaded CPU oracle baseline scores")
    ap.add_argument("--oracle-child", default="",
                    help=argparse.SUPPRESS)   # internal: time the oracle on a saved sample
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, device) -> float:
    """Largest value over all ranks (the job's time is its slowest rank's)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(pairs_per_step: int, steps: int, world: int, elapsed_ms: float) -> float:
    """Visible pairs scored by all ranks (one chunk each per step) per second."""
    return world * pairs_per_step * steps / (elapsed_ms * 1e-3)


def host_cpu() -> str:
    """CPU model of this host (lscpu, else /proc/cpuinfo, else the machine
    type), reported beside the CPU baseline's core count."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name:"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine() or "unknown"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


SCORE_TC_SOURCES = ["indexer_topk_long_gb300/csrc/k_score_tc.cu", "indexer_topk_long_gb300/csrc/ltk_internal.cuh"]
RETRIEVAL_SOURCES = ["indexer_topk_long_gb300/csrc/k_retrieval_tc.cu", "indexer_topk_long_gb300/csrc/ltk_internal.cuh"]


def kernel_source_hash(sources=None) -> str:
    """Hash of the kernel's code (comments and blank space removed, so that a
    documentation edit does not retire a recorded measurement)."""
    h = hashlib.sha256()
    for rel in sources or SCORE_TC_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(profile: str, sources=None):
    """DRAM bytes per filter-kernel launch from the committed ncu summary
    profiles/<profile>.md, if it was captured on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"{profile}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    hsh = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    if not m or not hsh or hsh.group(1) != kernel_source_hash(sources):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms.  The raw
    samples go to clocks_<pid>.csv in $LTK_CLOCKS_DIR (default: the system
    temporary directory)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.proc = None
        self.uuid = uuid
        self.path = os.path.join(os.environ.get("LTK_CLOCKS_DIR") or tempfile.gettempdir(),
                                 f"clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = float(parts[2])
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def build_inputs(workload: str, dtype: str, seed: int, queries: int = 0):
    """Host inputs of the current and previous chunk (shared key cache).
    ``queries`` > 0 keeps only the first queries of each chunk."""
    import dataclasses
    from indexer_topk_long_gb300 import datagen
    cur, prev = WORKLOADS[workload]
    wl = datagen.WORKLOADS[cur]
    wlp = datagen.WORKLOADS[prev]
    if queries:
        wl = dataclasses.replace(wl, T=min(queries, wl.T))
        wlp = dataclasses.replace(wlp, T=min(queries, wlp.T))
    keys = datagen.keys_fp32(wl.S, wl.d, seed)
    inp = datagen.make_indexer_inputs(wl.T, wl.first_pos, wl.S, wl.H, wl.d, seed, dtype, keys=keys)
    inp_prev = datagen.make_indexer_inputs(wlp.T, wlp.first_pos, wlp.S, wlp.H, wlp.d, seed, dtype,
                                           keys=keys)
    return wl, inp, inp_prev


def to_dev(inp, torch, dev):
    import numpy as np
    if inp.dtype == "bf16":
        q = torch.from_numpy(inp.q.view(np.int16)).to(dev)
        k = torch.from_numpy(inp.k.view(np.int16)).to(dev)
        qs = ks = None
    else:
        q = torch.from_numpy(inp.q).to(dev)
        k = torch.from_numpy(inp.k).to(dev)
        qs = torch.from_numpy(inp.q_scale).to(dev)
        ks = torch.from_numpy(inp.k_scale).to(dev)
    return dict(q=q, w=torch.from_numpy(inp.w).to(dev), k_cache=k,
                positions=torch.from_numpy(inp.positions).to(dev), q_scale=qs, k_scale=ks)


def _sample_queries(T: int, n: int) -> list[int]:
    """n queries evenly spaced over the chunk, first and last included."""
    import numpy as np
    return sorted(set(np.linspace(0, T - 1, max(n, 1)).astype(int).tolist()))


def oracle_child(path: str) -> int:
    """Child process of the CPU baseline: load a saved sample of the chunk, time
    the oracle on it with the BLAS/OpenMP thread count its environment sets,
    print one JSON line {seconds, pairs}."""
    import numpy as np
    import oracle.indexer_topk as orc
    z = np.load(path)

    class Chunk:   # the fields the oracle reads
        dtype = str(z["dtype"])
        q, w, k, positions = z["q"], z["w"], z["k"], z["positions"]
        q_scale = z["q_scale"] if "q_scale" in z else None
        k_scale = z["k_scale"] if "k_scale" in z else None
    keys64 = orc.widen_keys(Chunk)
    sel = list(range(Chunk.q.shape[0]))
    pairs = sum(orc.visible_count(Chunk.positions[t], keys64.shape[0], True) for t in sel)
    t0 = time.perf_counter()
    orc.indexer_topk(Chunk, int(z["k_top"]), queries=sel, keys64=keys64)
    print(json.dumps({"seconds": time.perf_counter() - t0, "pairs": int(pairs)}), flush=True)
    return 0


def cpu_oracle_rate(inp, k: int, n_queries: int, threads: int):
    """Oracle (plain fp64 definition + full sort) on a bounded sample of the
    chunk's queries, in a child process whose BLAS/OpenMP pools hold
    ``threads`` threads; returns (pairs/s, seconds, sample description)."""
    import numpy as np
    sel = _sample_queries(inp.T, n_queries)
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    try:
        extra = {}
        if inp.dtype == "fp8":
            extra = {"q_scale": inp.q_scale[sel], "k_scale": inp.k_scale}
        np.savez(path, dtype=np.array(inp.dtype), q=inp.q[sel], w=inp.w[sel], k=inp.k,
                 positions=inp.positions[sel], k_top=np.array(k), **extra)
        env = dict(os.environ)
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                    "BLIS_NUM_THREADS", "VECLIB_MAXIMUM_THREADS"):
            env[var] = str(threads)
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", path],
                             env=env, capture_output=True, text=True, timeout=900, check=True)
        res = json.loads(out.stdout.strip().splitlines()[-1])
    finally:
        os.unlink(path)
    dt, pairs = res["seconds"], res["pairs"]
    return pairs / dt, dt, (f"{len(sel)} of {inp.T} queries evenly spaced over the chunk "
                            f"(first and last included), {pairs} visible pairs; key cache "
                            f"widened to fp64 once before timing")


def cpu_baseline_record(inp, k: int, n_single: int, n_all: int) -> dict:
    """The oracle timed single-threaded (the baseline) and on all host cores."""
    cores = os.cpu_count() or 1
    r1, s1, d1 = cpu_oracle_rate(inp, k, n_single, 1)
    rn, sn, dn = cpu_oracle_rate(inp, k, n_all, cores)
    return {"value": r1, "unit": UNIT, "cores": 1, "threads": 1, "cpu": host_cpu(),
            "kind": "oracle", "sample": d1, "seconds": s1,
            "single_thread": {"value": r1, "threads": 1, "seconds": s1, "sample": d1},
            "all_cores": {"value": rn, "threads": cores, "cores": cores, "seconds": sn,
                          "sample": dn},
            "how": ("oracle in a child process with OMP/OPENBLAS/MKL thread counts set to "
                    "1 (single_thread) and to the host's cores (all_cores)")}


def run_reference(args):
    """Reference arm: the CPU oracle, bounded sample per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle.indexer_topk as orc
    wl, inp, _ = build_inputs(args.workload, args.dtype, 20260715)
    keys64 = orc.widen_keys(inp)
    T = inp.T
    rng = np.random.default_rng(1)
    def step():
        sel = sorted(rng.choice(T, size=args.ref_queries, replace=False).tolist())
        t0 = time.perf_counter()
        orc.indexer_topk(inp, wl.k, queries=sel, keys64=keys64)
        return sum(orc.visible_count(inp.positions[t], inp.S, True) for t in sel), time.perf_counter() - t0
    for _ in range(args.warmup):
        step()
    pairs = secs = 0.0
    for _ in range(args.steps):
        p, s = step()
        pairs += p
        secs += s
    value = pairs / secs
    # one chunk at the measured rate (the oracle scores only a sample of it)
    ms_per_chunk = wl.visible_pairs / value * 1e3
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_chunk,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded hot-key/topic generator)",
        "ms_per_step_is_extrapolated": True,
        "measured_ms_per_step": secs / args.steps * 1e3,
        "extrapolation": (f"ms_per_step = one whole chunk ({wl.visible_pairs} visible pairs) at the "
                          f"measured rate; each timed step scores {args.ref_queries} queries"),
        "config": {"workload": f"{args.workload} chunk, {args.dtype} inputs widened to fp64, k={wl.k}",
                   "sample": f"{args.ref_queries} random queries of the chunk per step",
                   "threads": "numpy's default BLAS pool (all host cores)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "threads": cores, "cpu": host_cpu(),
                         "kind": "oracle",
                         "sample": f"{args.ref_queries} queries per step x {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


RETRIEVAL = dict(T=1024, N=8388608, d=768, k=1000, sample=3000)
RETRIEVAL_METRIC = "scored query-vector pairs/s, vector retrieval 1024 x 8.4M, d=768 (1 GB300)"


def retrieval_record(dev, steps: int, warmup: int, k: int = 0, corpus: int = 0, queries: int = 0,
                     rank: int = 0, world: int = 1, e2e: bool = True, decoupled: bool = True,
                     cpu: bool = True) -> dict:
    """Vector-retrieval workload: one head, plain inner product, no mask."""
    import numpy as np
    import torch
    from indexer_topk_long_gb300 import IndexerTopK, datagen
    R = dict(RETRIEVAL)
    if k:
        R["k"] = k
        R["sample"] = min(3 * k, 16384)
    if corpus:
        R["N"] = corpus
    T = queries or R["T"]
    q, c = datagen.retrieval_inputs_torch(R["N"], T, R["d"], seed=20260715 + rank, device=dev)
    w = torch.ones((T, 1), dtype=torch.float32, device=dev)
    qi, ci = q.view(torch.int16), c.view(torch.int16)
    op = IndexerTopK(max_T=T, max_S=R["N"], k=R["k"], heads=1, dim=R["d"], sample_size=R["sample"],
                     enable_host_io=1 if e2e else 0)
    stream = torch.cuda.current_stream()
    out = (torch.empty((T, R["k"]), dtype=torch.int32, device=dev),
           torch.empty((T, R["k"]), dtype=torch.float32, device=dev))
    step = lambda: op(qi, w, ci, None, k=R["k"], out=out)
    for _ in range(max(warmup, 0)):
        step()
    torch.cuda.synchronize()
    launches0 = op.stats()["launches"]
    op.set_timing(True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(device_uuid(torch, dev))
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    st = op.stats()
    op.set_timing(False)
    elapsed = max_over_ranks(e0.elapsed_time(e1), dev)
    pairs = T * R["N"]
    assert st["visible_pairs"] == pairs and st["device_status"] == 0
    peaks, kind = measured_peaks()
    peak = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    flop = 2 * R["d"] * pairs
    achieved = flop / (st["ms_filter"] * 1e-3) / 1e12
    line = {
        "metric": (RETRIEVAL_METRIC if R["N"] == RETRIEVAL["N"]
                   else RETRIEVAL_METRIC.replace("8.4M", str(R["N"]))),
        "value": whole_job_value(pairs, steps, world, elapsed),
        "unit": UNIT, "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": elapsed / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (clustered Gaussian corpus; MSMARCO unavailable)",
        "config": {"workload": f"vector retrieval: {T} queries x {R['N']} corpus rows, d={R['d']}, "
                               f"k={R['k']}, H=1, no ReLU, no mask, {R['sample']} random sample rows",
                   "l2": f"inputs larger than L2 (corpus {R['N'] * R['d'] * 2 / 1e9:.1f} GB)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "frac_clock_normalised": clock_normalised(achieved, peak, clock_info, peaks),
                     "traffic": (recorded_traffic(f"retrieval_filter_8m_k{R['k']}", RETRIEVAL_SOURCES)
                                 if R["N"] == RETRIEVAL["N"] and T == RETRIEVAL["T"] else None),
                     "kernel": "retrieval_tc_kernel<filter>",
                     "peak_source": f"{kind} bf16 sustained", "algorithmic_flop_per_launch": flop},
        "gpu_launches": st["launches"] - launches0, "clocks": clock_info,
        "stages_ms": {"sample": st["ms_sample"], "filter": st["ms_filter"], "select": st["ms_select"],
                      "rescue": st["ms_rescue"]},
        "candidates_per_query": st["cand_written"] / T, "n_overflow": st["n_overflow"],
    }
    if decoupled and world == 1:
        op.close()
        dec = IndexerTopK(max_T=T, max_S=R["N"], k=R["k"], heads=1, dim=R["d"], enable_decoupled=1)
        di, ds = dec.decoupled(qi, w, ci, None, k=R["k"])
        torch.cuda.synchronize()
        dec.set_timing(True)
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        dec.decoupled(qi, w, ci, None, k=R["k"], out=(di, ds))
        a1.record(stream)
        torch.cuda.synchronize()
        dst = dec.stats()
        dec_ms = a0.elapsed_time(a1)
        line["decoupled"] = {"ms_per_step": dec_ms, "score_kernel_ms": dst["ms_filter"],
                             "select_ms": dst["ms_select"], "fused_speedup": dec_ms / line["ms_per_step"],
                             "identical_output": bool(torch.equal(di, out[0]) and torch.equal(ds, out[1]))}
        dec.close()
        del dec, di, ds
        torch.cuda.empty_cache()
        op = IndexerTopK(max_T=T, max_S=R["N"], k=R["k"], heads=1, dim=R["d"], sample_size=R["sample"],
                         enable_host_io=1 if e2e else 0)
    if e2e:
        hq, hw, hc = qi.cpu().pin_memory(), w.cpu().pin_memory(), ci.cpu().pin_memory()
        hout = (torch.empty((T, R["k"]), dtype=torch.int32, pin_memory=True),
                torch.empty((T, R["k"]), dtype=torch.float32, pin_memory=True))
        op.topk_host(hq, hw, hc, None, k=R["k"], out=hout)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(steps):
            op.topk_host(hq, hw, hc, None, k=R["k"], out=hout)
        a1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a0.elapsed_time(a1), dev)
        line["e2e"] = {"value": whole_job_value(pairs, steps, world, e_ms), "unit": UNIT,
                       "h2d_bytes_per_step": hq.numel() * 2 + hw.numel() * 4 + hc.numel() * 2,
                       "d2h_bytes_per_step": T * R["k"] * 8, "ms_per_step": e_ms / steps}
    if cpu and world == 1 and rank == 0:
        import oracle.indexer_topk as orc
        n_rows = R["N"]   # the whole corpus (~10 s of widening and products on the host)
        sel = sorted({0, T // 3, (2 * T) // 3, T - 1})
        qh = qi[sel].cpu().numpy().view(np.uint16)
        ch = ci[:n_rows].cpu().numpy().view(np.uint16)
        t0 = time.perf_counter()
        orc.retrieval_topk(qh, ch, R["k"])
        secs = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": len(sel) * n_rows / secs, "unit": UNIT, "cores": os.cpu_count(),
                                "threads": os.cpu_count(), "cpu": host_cpu(),
                                "kind": "oracle", "seconds": secs,
                                "sample": f"{len(sel)} queries against the whole corpus ({n_rows} rows)"}
    op.close()
    del q, c, qi, ci, out
    torch.cuda.empty_cache()
    return line


def run_retrieval(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    line = retrieval_record(dev, args.steps, args.warmup, k=args.k, corpus=args.corpus,
                            queries=args.queries, rank=rank, world=world, e2e=not args.no_e2e,
                            decoupled=not args.no_decoupled, cpu=not args.no_cpu)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


DECODE_METRIC = "decode: scored query-key pairs/s and ms per call, T new tokens at 1M ctx, k=2048 (1 GB300)"


def decode_record(T: int, dtype: str, engine: str, steps: int, warmup: int, dev, rank: int = 0,
                  world: int = 1) -> dict:
    """Decode / small-T: T queries at the end of a 1M-token cache, previous-step
    sample; the key range is split over the GPU.  Returns the JSON record."""
    import torch
    from indexer_topk_long_gb300 import IndexerTopK, datagen
    S = 1 << 20
    keys = datagen.keys_fp32(S, 128, 20260715 + rank)
    inp = datagen.make_indexer_inputs(T, S - T, S, dtype=dtype, seed=20260715 + rank, keys=keys)
    d = to_dev(inp, torch, dev)
    op = IndexerTopK(max_T=T, max_S=S, k=2048, dtype=dtype,
                     engine={"auto": 0, "tensor": 1, "cuda": 2}[engine])
    out = (torch.empty((T, 2048), dtype=torch.int32, device=dev),
           torch.empty((T, 2048), dtype=torch.float32, device=dev))
    first = op(d["q"], d["w"], d["k_cache"], d["positions"], k=2048, q_scale=d["q_scale"], k_scale=d["k_scale"])
    sample = op.make_sample(first[0], S, 6144)
    stream = torch.cuda.current_stream()
    step = lambda: op(d["q"], d["w"], d["k_cache"], d["positions"], k=2048, prev_topk=sample,
                      q_scale=d["q_scale"], k_scale=d["k_scale"], out=out)
    for _ in range(max(warmup, 0)):
        step()
    torch.cuda.synchronize()
    op.set_timing(True)
    launches0 = op.stats()["launches"]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    st = op.stats()
    ms = e0.elapsed_time(e1) / steps
    pairs = st["visible_pairs"]
    # the same call captured once in a CUDA graph and replayed (no launch gaps)
    op.set_timing(False)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(max(warmup, 1)):
        graph.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    graph_ms = e0.elapsed_time(e1) / steps
    # a few queries against the whole cache: the key stream (S x d elements,
    # plus the fp8 scales) is the algorithmic traffic of the filter kernel
    peaks, kind = measured_peaks()
    k_bytes = S * 128 * (1 if dtype == "fp8" else 2) + (S * 4 if dtype == "fp8" else 0)
    flop = 16384.0 * pairs                         # H * d * 2 per visible pair (one call)
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tflops = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    if dtype == "fp8":
        tflops *= FP8_OVER_BF16
    # the bound is whichever floor is higher: streaming the cache or the MMAs
    t_hbm = k_bytes / (hbm * 1e9)
    t_tc = flop / (tflops * 1e12)
    sec = st["ms_filter"] * 1e-3
    if t_hbm >= t_tc:
        bound, achieved, peak, unit = "hbm", k_bytes / sec / 1e9, hbm, "GB/s"
    else:
        bound, achieved, peak, unit = "tensor", flop / sec / 1e12, tflops, "TFLOP/s"
    line = {"metric": DECODE_METRIC, "value": world * pairs / (ms * 1e-3), "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded hot-key/topic generator)",
            "config": {"workload": f"decode: T={T} queries at positions {S - T}..{S - 1}, S={S}, H=64, "
                                   f"d=128, k=2048, previous-step sample; keys split over the GPU",
                       "engine": engine},
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                         "frac": achieved / peak,
                         "traffic": recorded_traffic(f"score_filter_decode_t{T}_{dtype}") if engine == "auto" else None,
                         "kernel": "filter stage (score_tc_kernel<filter>, keys split over the GPU)",
                         "peak_source": f"{kind} " + ("copy bandwidth" if bound == "hbm" else "bf16 sustained"),
                         "algorithmic_bytes_per_call": k_bytes, "algorithmic_flop_per_call": flop},
            "gpu_launches": st["launches"] - launches0,
            "stages_ms": {"sample": st["ms_sample"], "filter": st["ms_filter"], "select": st["ms_select"]},
            "candidates_per_query": st["cand_written"] / T, "n_overflow": st["n_overflow"],
            "graph": {"ms_per_step": graph_ms, "value": world * pairs / (graph_ms * 1e-3),
                      "how": "one call captured with torch.cuda.graph, replayed back to back"}}
    op.close()
    del graph, d, out, first, sample
    torch.cuda.empty_cache()
    return line


def run_decode(args):
    import torch
    rank, world, local = dist_env()
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    line = decode_record(args.queries or 1, args.dtype, args.engine, args.steps, args.warmup, dev,
                         rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def clock_normalised(achieved: float, peak: float, clocks, peaks) -> float | None:
    """achieved / (peak scaled to this run's SM clock): the measured tensor
    peak was taken at its own median SM clock under load, this run at
    another, and tensor throughput scales with the SM clock."""
    try:
        peak_mhz = float(peaks["clocks_under_load"]["sm_mhz_median"])
        run_mhz = float(clocks["sm_mhz"])
    except (KeyError, TypeError, ValueError):
        return None
    if peak_mhz <= 0 or run_mhz <= 0:
        return None
    return achieved / (peak * run_mhz / peak_mhz)


def device_uuid(torch, dev):
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        return None


def prefill_record(workload: str, dtype: str, steps: int, warmup: int, dev, *, rank: int = 0,
                   world: int = 1, queries: int = 0, e2e: bool = True, decoupled: bool = True,
                   dec_steps: int = 3, cpu: bool = False, cpu_queries: int = 64,
                   cpu_single_queries: int = 16, litedsa: bool = True) -> dict:
    """One prefill chunk (previous chunk first, its output is the sample): the
    timed fused path, its roofline, and optionally the end-to-end host-buffer
    call, the same-GPU decoupled baseline and the CPU oracle baseline."""
    import torch
    from indexer_topk_long_gb300 import IndexerTopK

    seed = 20260715 + rank        # each rank runs its own, independent chunk
    wl, inp, inp_prev = build_inputs(workload, dtype, seed, queries)
    d = to_dev(inp, torch, dev)
    dp = to_dev(inp_prev, torch, dev)
    k = wl.k
    op = IndexerTopK(max_T=wl.T, max_S=wl.S, k=k, dtype=dtype,
                     enable_decoupled=0, enable_host_io=1 if e2e else 0)
    stream = torch.cuda.current_stream()

    # previous chunk (its output provides the sample), outside the timed region
    S_prev = inp_prev.S
    prev_idx, _ = op(dp["q"], dp["w"], d["k_cache"][:S_prev], dp["positions"], k=k,
                     q_scale=dp["q_scale"], k_scale=None if dp["k_scale"] is None else d["k_scale"][:S_prev])
    out_idx = torch.empty((wl.T, k), dtype=torch.int32, device=dev)
    out_score = torch.empty((wl.T, k), dtype=torch.float32, device=dev)

    def step():
        sample = op.make_sample(prev_idx, wl.S, 3 * k)
        op(d["q"], d["w"], d["k_cache"], d["positions"], k=k, prev_topk=sample,
           q_scale=d["q_scale"], k_scale=d["k_scale"], out=(out_idx, out_score))

    for _ in range(max(warmup, 0)):
        step()
    torch.cuda.synchronize()
    warm = op.stats()
    if warm["device_status"] != 0:
        raise RuntimeError(f"device status {warm['device_status']}")

    clocks = ClockSampler(device_uuid(torch, dev))
    launches0 = op.stats()["launches"]
    op.set_timing(True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clock_info = clocks.stop()
    elapsed_ms = ev0.elapsed_time(ev1)
    st = op.stats()
    op.set_timing(False)
    launches = st["launches"] - launches0
    elapsed_ms = max_over_ranks(elapsed_ms, dev)
    pairs_step = st["visible_pairs"]
    assert pairs_step == wl.visible_pairs, (pairs_step, wl.visible_pairs)
    assert st["device_status"] == 0, st
    ms_per_step = elapsed_ms / steps
    value = whole_job_value(pairs_step, steps, world, elapsed_ms)

    peaks, peaks_kind = measured_peaks()
    bf16_peak = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    peak = bf16_peak * (FP8_OVER_BF16 if dtype == "fp8" else 1.0)
    achieved = FLOP_PER_PAIR * pairs_step / (st["ms_filter"] * 1e-3) / 1e12
    traffic = recorded_traffic(f"score_filter_{workload}_{dtype}")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "frac_clock_normalised": clock_normalised(achieved, peak, clock_info, peaks),
                "traffic": traffic,
                "kernel": "score_tc_kernel<filter> (fused score + bin + gate + write-back)",
                "peak_source": (f"{peaks_kind} bf16 sustained" +
                                (" x 2 (nominal fp8/bf16 ratio)" if dtype == "fp8" else "")),
                "clock_normalisation": ("peak x (this run's median SM MHz / the median SM MHz "
                                        "under load recorded with the measured peak)"),
                "algorithmic_flop_per_launch": FLOP_PER_PAIR * pairs_step}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": dtype,
        "data": "synthetic (seeded hot-key/topic generator; no dataset)",
        "config": {
            "workload": (f"{workload} prefill chunk: T={wl.T} queries at positions "
                         f"{wl.first_pos}..{wl.first_pos + wl.T - 1}, S={wl.S}, H={wl.H}, "
                         f"d={wl.d}, k={k}, {dtype} q/k, fp32 w, previous-chunk top-3k sample"),
            "l2": (f"inputs larger than L2 (key cache {wl.S * wl.d * (1 if dtype == 'fp8' else 2) / 2**20:.0f} MiB"
                   f" + queries {wl.T * wl.H * wl.d * (1 if dtype == 'fp8' else 2) / 2**20:.0f} MiB > 129 MB L2)"),
            "parallelism": f"replicas: {world} independent chunks, one per GPU",
            "visible_pairs_per_chunk": pairs_step,
        },
        "roofline": roofline,
        "gpu_launches": launches,
        "clocks": clock_info,
        "stages_ms": {"sample": st["ms_sample"], "filter": st["ms_filter"],
                      "select": st["ms_select"], "rescue": st["ms_rescue"],
                      "total_fused_call": st["ms_total"]},
        "candidates_per_query": st["cand_written"] / wl.T,
        "candidates_max": st["cand_max"],
        "n_overflow": st["n_overflow"],
        "bytes_written_per_query": {"fused": 8.0 * st["cand_written"] / wl.T + 8.0 * k,
                                    "decoupled": 4.0 * pairs_step / wl.T},
    }

    # ---- LiteDSA packing of the chunk's output (groups of 8 neighbouring queries)
    if litedsa:
        from indexer_topk_long_gb300 import litedsa_pack
        litedsa_pack(out_idx, 8)
        torch.cuda.synchronize()
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        _, lens, _ = litedsa_pack(out_idx, 8)
        l1.record(stream)
        torch.cuda.synchronize()
        line["litedsa"] = {"group": 8, "ms": l0.elapsed_time(l1),
                           "kv_rows_packed": int(lens.sum().item()), "kv_rows_per_query_lists": wl.T * k,
                           "kv_row_ratio": float(lens.sum().item()) / (wl.T * k)}

    # ---- end to end through the host-buffer C-ABI call
    if e2e:
        sample = op.make_sample(prev_idx, wl.S, 3 * k).cpu().pin_memory()
        host = {key: (v.cpu().pin_memory() if v is not None else None) for key, v in d.items()}
        hout = (torch.empty((wl.T, k), dtype=torch.int32, pin_memory=True),
                torch.empty((wl.T, k), dtype=torch.float32, pin_memory=True))
        def e2e_step():
            op.topk_host(host["q"], host["w"], host["k_cache"], host["positions"], k=k,
                         prev_topk=sample, q_scale=host["q_scale"], k_scale=host["k_scale"], out=hout)
        e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), dev)
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None) + \
            sample.numel() * 4
        d2h = sum(v.numel() * v.element_size() for v in hout)
        line["e2e"] = {"value": whole_job_value(pairs_step, steps, world, e_ms), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e_ms / steps,
                       "call": "ltk_indexer_topk_host (pinned host buffers, copies inside)"}
        ok = torch.equal(hout[0], out_idx.cpu())
        line["e2e"]["matches_device_call"] = bool(ok)
        del host

    # ---- same-GPU decoupled baseline (materialise fp32 scores, then select)
    op.close()
    if decoupled and world == 1:
        dec = IndexerTopK(max_T=wl.T, max_S=wl.S, k=k, dtype=dtype, enable_decoupled=1)
        di = torch.empty_like(out_idx)
        ds = torch.empty_like(out_score)
        def dec_step():
            dec.decoupled(d["q"], d["w"], d["k_cache"], d["positions"], k=k, q_scale=d["q_scale"],
                          k_scale=d["k_scale"], out=(di, ds))
        dec_step()
        torch.cuda.synchronize()
        dec.set_timing(True)
        n_dec = max(1, min(steps, dec_steps))
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_dec):
            dec_step()
        a1.record(stream)
        torch.cuda.synchronize()
        dst = dec.stats()
        dec_ms = a0.elapsed_time(a1) / n_dec
        line["decoupled"] = {"ms_per_step": dec_ms, "score_kernel_ms": dst["ms_filter"],
                             "select_ms": dst["ms_select"],
                             "score_matrix_bytes": 4 * wl.T * wl.S,
                             "fused_speedup": dec_ms / ms_per_step,
                             "identical_output": bool(torch.equal(di, out_idx) and torch.equal(ds, out_score))}
        dec.close()
        del dec, di, ds

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    if cpu and world == 1 and rank == 0:
        line["cpu_baseline"] = cpu_baseline_record(inp, k, cpu_single_queries, cpu_queries)

    del d, dp, out_idx, out_score, prev_idx
    torch.cuda.empty_cache()
    return line


def sub_record(line: dict) -> dict:
    """The keys of a sub-workload's record that the headline line nests."""
    keep = ("ms_per_step", "value", "unit", "dtype", "steps", "warmup", "config", "roofline",
            "stages_ms", "clocks", "candidates_per_query", "n_overflow", "decoupled", "graph",
            "gpu_launches")
    return {key: line[key] for key in keep if key in line}


def main():
    args = parse_args()
    if args.oracle_child:
        return oracle_child(args.oracle_child)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "retrieval":
        return run_retrieval(args)
    if args.workload == "decode":
        return run_decode(args)
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    line = prefill_record(args.workload, args.dtype, args.steps, args.warmup, dev, rank=rank,
                          world=world, queries=args.queries, e2e=not args.no_e2e,
                          decoupled=not args.no_decoupled, cpu=not args.no_cpu,
                          cpu_queries=args.cpu_queries, cpu_single_queries=args.cpu_single_queries)

    # ---- the other configurations, measured in the same run (one GPU only):
    # the 1M chunk in e4m3, the 256K chunk against its decoupled baseline
    # (the pages compare the two at 256K and 1M), decode at T = 1, and the
    # vector-retrieval workload (1024 queries x 8.4M rows, k = 1000)
    headline = (args.workload == "1m" and args.dtype == "bf16" and not args.queries)
    if headline and not args.no_extra and world == 1:
        extra_steps, extra_warm = max(1, min(args.steps, 5)), max(2, min(args.warmup, 3))
        line["fp8_1m"] = sub_record(prefill_record(
            "1m", "fp8", extra_steps, extra_warm, dev, e2e=False, decoupled=not args.no_decoupled,
            dec_steps=2, litedsa=False))
        line["prefill_256k"] = sub_record(prefill_record(
            "256k", "bf16", extra_steps, extra_warm, dev, e2e=False, decoupled=not args.no_decoupled,
            dec_steps=3, litedsa=False))
        line["decode_t1"] = sub_record(decode_record(1, "bf16", "auto", max(args.steps, 10),
                                                     extra_warm, dev))
        line["retrieval"] = sub_record(retrieval_record(dev, extra_steps, extra_warm, e2e=False,
                                                        decoupled=not args.no_decoupled, cpu=False))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
