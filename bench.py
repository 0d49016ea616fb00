#!/usr/bin/env python3
"""Benchmark of the verification hot path on GB300.

Workload (one "step"): chain speculative sampling with c* for R=64 requests,
gamma=7 draft positions, V=151936 bf16 logits, temperature 1 -- one
specv_verify_chain call over a batch resident in HBM (target [64, 8, V] +
draft [64, 7, V] = 291.7 MB of logits).  Metric: verified draft positions per
second (sum of l_r over the batch / step time), plus achieved HBM GB/s as a
fraction of the measured copy bandwidth.

`--impl reference` times the CPU oracle (the reference arm of this repo) on the
same workload, one bounded sample of requests per step.

`--workload` selects another row of the hot path for its own JSON line (the
default is the headline chain workload above):
  greedy    T = 0 chain verification, R=64, gamma=7, V=151936 (target rows only)
  tv        standalone c* (specv_tv_accept), R=64, gamma=7, V=151936, T = 1
  tree      greedy tree verification, R=16 trees of 60 nodes + root, V=151936
  markov    DSpark Markov head, R=512, gamma=7, V=129280, rank 256, T = 1,
            float32 logits written
  schedule  greedy scheduler, R=512, gamma=7, SPS table of 4096 entries
  dspark    the DSpark round: Markov drafting (R=512, gamma=7, V=129280, bf16
            logits), the scheduler's lengths, then chain verification with them

Multi-GPU (torchrun): every rank verifies its own batch (requests are
independent; no collective on the data path); value = all ranks' positions /
max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

R, GAMMA, V, TEMP = 64, 7, 151936, 1.0
METRIC = "verified draft positions/sec and achieved HBM GB/s (fraction of peak) at R=64,γ=7,V=151936"
UNIT = "positions/s"
WORKLOAD = "batched chain verify: R=64, gamma=7, V=151936 bf16, T=1.0, c* output"
ALGO_BYTES = R * (GAMMA + 1) * V * 2 + R * GAMMA * V * 2      # every logit read once
PROFILE = os.path.join(ROOT, "profiles", "chain_stats_batched_r64_g7_v151936.md")
KERNEL_SOURCES = [os.path.join(ROOT, "lossless_draft_verification_gb300", "csrc", f) for f in ("chain.cu", "common.cuh")]


def _peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _kernel_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _profile_traffic():
    """Per-launch DRAM traffic from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    try:
        txt = open(PROFILE).read()
    except OSError:
        return None
    m_h = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_h or not m_t or m_h.group(1) != _kernel_hash():
        return None
    return float(m_t.group(1))


class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum and the
    active clock-event reasons) for the GPU torch uses, matched by UUID."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device: int):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(torch_device).uuid)
            ok = self.lib.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(self.h)) == 0
        except Exception:
            ok = False
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(torch_device), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self) -> int:
        v = self.c.c_uint()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.c.byref(v))        # NVML_CLOCK_SM
        return v.value

    def sm_max_mhz(self) -> int:
        v = self.c.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.c.byref(v))
        return v.value

    def reasons(self) -> int:
        v = self.c.c_ulonglong()
        self.reasons_fn(self.h, self.c.byref(v))
        return v.value


class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled while the timed
    region runs: NVML polled every ~0.2 ms from a thread (a timed region of a
    few milliseconds still gets samples); nvidia-smi at 10 ms if NVML cannot
    be loaded."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.nvml = None
        self.thread = None
        self.samples = []
        self.stop_flag = False

    def start(self):
        try:
            self.nvml = _Nvml(self.gpu)
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            import threading

            def poll():
                while not self.stop_flag:
                    self.samples.append((self.nvml.sm_mhz(), self.nvml.reasons()))
                    time.sleep(0.0002)
            self.thread = threading.Thread(target=poll, daemon=True)
            self.thread.start()
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "10"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.nvml is not None:
            self.stop_flag = True
            self.thread.join()
            if not self.samples:                      # the region ended before the first poll returned
                self.samples.append((self.nvml.sm_mhz(), self.nvml.reasons()))
            sm = [a for a, _ in self.samples]
            reasons = sorted({n for _, b in self.samples for bit, n in _Nvml.REASONS.items() if b & bit})
            return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.nvml.sm_max_mhz(), "reasons": reasons,
                    "samples": len(sm), "source": "nvml"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
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
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


def cpu_info() -> dict:
    """Host CPU model and core count (the oracle baseline's machine)."""
    model = None
    try:
        for line in open("/proc/cpuinfo"):
            k = line.split(":")[0].strip().lower()
            if k in ("model name", "cpu model", "hardware"):
                model = line.split(":", 1)[1].strip()
                break
    except OSError:
        pass
    if model is None:
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "model": model}


def rank_seed(rank: int) -> int:
    """Seed of rank `rank`'s batch: ranks verify independent request batches."""
    return 3 + 1000 * rank


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time (ms) when running under torch.distributed, else `ms`."""
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, ms_max: float) -> float:
    """Units processed by all ranks per second, timed by the slowest rank."""
    return world * units_per_rank / (ms_max * 1e-3)


def _oracle_request(task):
    """One request through the oracle: widen its bf16 rows, verify.  A worker
    task of the all-core baseline (module level so spawned workers import it)."""
    import oracle
    import synth
    t_bits, d_bits, x, u, T = task
    t = synth.bf16_bits_to_f64(t_bits)[None]
    d = synth.bf16_bits_to_f64(d_bits)[None]
    return oracle.verify_chain(t, d, x[None], u[None], T)


def _tasks(case, idx):
    return [(case.target.raw[r], case.draft.raw[r], case.tokens[r], case.uniforms[r], case.temperature) for r in idx]


def _spawn_pool(n):
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"                     # one thread per worker
    # glibc keeps freed blocks instead of unmapping them and numpy asks for no
    # huge pages, so the workers' repeated large temporaries reuse memory
    # instead of faulting in fresh pages (read at the workers' start-up)
    os.environ["MALLOC_MMAP_MAX_"] = "0"
    os.environ["MALLOC_TRIM_THRESHOLD_"] = str(1 << 34)
    os.environ.setdefault("NUMPY_MADVISE_HUGEPAGE", "0")
    return ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))


def oracle_single_thread(case, budget_s: float):
    """The oracle request by request on one core until `budget_s` elapses
    (wrapping around the batch).  Returns (positions/s, requests done, seconds,
    {r: ChainResult} for the first pass over the batch)."""
    results = {}
    done = 0
    tasks = _tasks(case, range(case.R))
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        r = done % case.R
        res = _oracle_request(tasks[r])
        results.setdefault(r, res)
        done += 1
    el = time.perf_counter() - t0
    return done * case.gamma / el, done, el, results


def oracle_all_cores(case, budget_s: float, pool, n_workers: int):
    """The same oracle call spread over `n_workers` spawned processes, one
    request per task, whole batches until `budget_s` elapses."""
    tasks = _tasks(case, range(case.R))
    list(pool.map(_oracle_request, tasks[:n_workers]))            # workers started and warm
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        list(pool.map(_oracle_request, tasks))
        done += case.R
    el = time.perf_counter() - t0
    return done * case.gamma / el, done, el


def parity_counts(results, A, y, c, case, tol=1e-5):
    """Exact / flagged-threshold counts of the GPU's outputs against the oracle
    on the sampled requests.  A differing accept decision is flagged when its
    uniform lies within `tol` of min(1, q/p); a differing token with the same
    accepted length when the draw's uniform lies within `tol` of a boundary of
    the oracle's CDF bracket; anything else is a mismatch."""
    import numpy as np
    out = {"requests": 0, "exact": 0, "flagged_accept": 0, "flagged_sample": 0, "mismatch": 0,
           "max_abs_cstar_diff": 0.0}
    for r, res in sorted(results.items()):
        out["requests"] += 1
        Ag, yg, L = int(A[r]), int(y[r]), case.gamma
        ok = ~np.isnan(res.c_star[0])
        if ok.any():
            out["max_abs_cstar_diff"] = max(out["max_abs_cstar_diff"], float(np.abs(c[r][ok] - res.c_star[0][ok]).max()))
        if Ag == int(res.accepted[0]) and yg == int(res.token[0]):
            out["exact"] += 1
            continue
        u = case.uniforms[r]
        if Ag != int(res.accepted[0]):
            flagged = all(abs(float(u[k, 0]) - res.thr[0, k]) < tol
                          for k in range(min(L, max(Ag, int(res.accepted[0])) + 1))
                          if (k < Ag) != (float(u[k, 0]) < res.thr[0, k]))
            out["flagged_accept" if flagged else "mismatch"] += 1
            continue
        u1 = float(u[Ag, 1])
        near = abs(u1 - res.lo_at[0, Ag]) < tol or abs(u1 - res.hi_at[0, Ag]) < tol
        out["flagged_sample" if near else "mismatch"] += 1
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import synth
    case = synth.chain_batched(seed=3, R=R)
    n_workers = max(1, os.cpu_count() or 1)
    with _spawn_pool(n_workers) as pool:
        tasks = _tasks(case, range(R))
        list(pool.map(_oracle_request, tasks[:n_workers]))          # warm workers (untimed)
        t0 = time.perf_counter()
        list(pool.map(_oracle_request, tasks[:n_workers]))
        per_wave = time.perf_counter() - t0
        # size one step so that the whole run stays within ~2 minutes
        waves = int(max(1, min(-(-R // n_workers), 120.0 / max(1e-3, per_wave * (args.steps + args.warmup)))))
        n_req = min(R, waves * n_workers)

        def step(i):
            s = (i * n_req) % R
            list(pool.map(_oracle_request, [tasks[(s + j) % R] for j in range(n_req)]))
        for i in range(args.warmup):
            step(i)
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(args.warmup + i)
        el = time.perf_counter() - t0
    value = args.steps * n_req * GAMMA / el
    ci = cpu_info()
    sample = (f"{n_req} of {R} requests per step (gamma=7, V=151936) over {n_workers} worker processes, "
              f"float64 numpy oracle; host {ci['model']} ({ci['nproc']} cores)")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_workers, "kind": "oracle", "sample": sample,
                            "cpu": ci},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch

    import lossless_draft_verification_gb300 as specv
    from lossless_draft_verification_gb300 import build as _build
    import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    specv.load()

    case = synth.chain_batched(seed=rank_seed(rank), R=R)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    target = to_dev(case.target.raw.view(np.int16)).view(torch.bfloat16)
    draft = to_dev(case.draft.raw.view(np.int16)).view(torch.bfloat16)
    tokens = to_dev(case.tokens.astype(np.int32))
    uniforms = to_dev(case.uniforms.astype(np.float32))
    acc = torch.empty(R, dtype=torch.int32, device=dev)
    tok = torch.empty(R, dtype=torch.int32, device=dev)
    cst = torch.empty(R, GAMMA, dtype=torch.float32, device=dev)
    nbytes = specv.specv_verify_chain_workspace_size(R, GAMMA, V, specv.SPECV_BF16)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    ptrs = (target.data_ptr(), draft.data_ptr(), specv.SPECV_BF16, tokens.data_ptr(), None, uniforms.data_ptr(),
            R, GAMMA, V, TEMP, acc.data_ptr(), tok.data_ptr(), cst.data_ptr(), ws.data_ptr(), nbytes, sp)

    def call():
        st = specv.specv_verify_chain(*ptrs)
        if st != 0:
            raise specv.SpecvError(st, "specv_verify_chain")

    # The batch (291.7 MB) is 2.26x the L2, so by default steps run back to back
    # without a flush: the walk reads every row in the same order each step and
    # the L2 keeps only the last rows of the previous one, which the next step
    # reads last.  --flush-l2 writes a 2x-L2 buffer before every step instead.
    do_flush = args.flush_l2 or ALGO_BYTES < 2 * l2
    for _ in range(max(3, args.warmup)):
        if do_flush:
            flush.zero_()
        call()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        if do_flush:
            flush.zero_()
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if dist is not None:
        dist.barrier()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms_med, ms_mean = statistics.median(times), statistics.fmean(times)
    ms_max = max_over_ranks(ms_med, dist, dev)
    positions = R * GAMMA                   # lengths = gamma for every request
    value = whole_job_rate(positions, world, ms_max)
    A_gpu, y_gpu, c_gpu = acc.cpu().numpy(), tok.cpu().numpy(), cst.cpu().numpy()

    # end to end through the public API with pinned host buffers: requests in
    # four groups whose host-to-device copies (two copy streams) overlap the
    # previous group's kernels
    e2e = None
    if not args.no_e2e:
        h_t = torch.from_numpy(case.target.raw.view(np.int16)).view(torch.bfloat16).pin_memory()
        h_d = torch.from_numpy(case.draft.raw.view(np.int16)).view(torch.bfloat16).pin_memory()
        h_x = torch.from_numpy(case.tokens.astype(np.int32)).pin_memory()
        h_u = torch.from_numpy(case.uniforms.astype(np.float32)).pin_memory()
        n_e2e = max(3, min(args.steps, 30))
        chunks = 4
        for _ in range(3):
            specv.verify_chain(h_t, h_d, h_x, h_u, TEMP, chunks=chunks)
        torch.cuda.synchronize()
        e_times = []
        for _ in range(n_e2e):
            flush.zero_()
            s = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            s.record(stream)
            A_h, y_h, c_h = specv.verify_chain(h_t, h_d, h_x, h_u, TEMP, chunks=chunks)
            e.record(stream)
            torch.cuda.synchronize()
            e_times.append(s.elapsed_time(e))
        e_max = max_over_ranks(statistics.median(e_times), dist, dev)
        h2d = sum(t.numel() * t.element_size() for t in (h_t, h_d, h_x, h_u))
        d2h = sum(t.numel() * t.element_size() for t in (A_h, y_h, c_h))
        e2e = {"value": whole_job_rate(positions, world, e_max), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_max, "h2d_gbs": h2d / (e_max * 1e-3) / 1e9,
               "pipelining": f"{chunks} request groups, copies on two streams overlapping the previous group's kernels",
               "same_outputs_as_device_call": bool((A_h.numpy() == A_gpu).all() and (y_h.numpy() == y_gpu).all())}

    cpu = None
    parity = None
    if rank == 0 and not args.no_cpu_baseline:
        n_workers = max(1, os.cpu_count() or 1)
        ci = cpu_info()
        v1, n1, el1, results = oracle_single_thread(case, args.cpu_seconds / 2)
        with _spawn_pool(n_workers) as pool:
            vn, nn, eln = oracle_all_cores(case, args.cpu_seconds / 2, pool, n_workers)
        cpu = {"value": vn, "unit": UNIT, "cores": n_workers, "kind": "oracle",
               "sample": f"{nn} request verifications ({nn * GAMMA} positions) of this batch in {eln:.1f} s over "
                         f"{n_workers} worker processes (one request per task), float64 numpy oracle",
               "cpu": ci,
               "single_thread": {"value": v1, "unit": UNIT, "cores": 1,
                                 "sample": f"{n1} request verifications ({n1 * GAMMA} positions) in {el1:.1f} s"}}
        parity = parity_counts(results, A_gpu, y_gpu, c_gpu, case)
        parity["rule"] = ("GPU vs oracle on the sampled requests of the timed call: a differing decision is allowed "
                          "only where the uniform is within 1e-5 of its threshold (flagged)")

    peak, peak_kind = _peak_hbm()
    achieved = ALGO_BYTES / (ms_med * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": _profile_traffic(), "peak_source": peak_kind,
            "kernel": "chain_stats + chain_finish (whole specv_verify_chain call; a lower bound for chain_stats)",
            "algorithmic_bytes_per_launch": ALGO_BYTES}
    if dist is not None:
        dist.barrier()
    if rank == 0:
        out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": ms_max, "ms_mean": ms_mean, "ms_median": ms_med,
               "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": {"workload": WORKLOAD, "R": R, "gamma": GAMMA, "V": V, "temperature": TEMP,
                          "batch_per_gpu": R, "parallelism": f"independent requests x{world}",
                          "l2": ("flushed (2x L2 write) before every timed step" if do_flush else
                                 f"not flushed: inputs {ALGO_BYTES / 1e6:.1f} MB are {ALGO_BYTES / l2:.2f}x the L2 "
                                 f"({l2 / 1e6:.0f} MB)"), "wall_s": wall,
                          "timing": "median of the timed steps' CUDA-event times (mean beside it)"},
               "hbm_gbs": achieved, "hbm_frac": achieved / peak, "roofline": roof, "cpu_baseline": cpu,
               "parity_sample": parity, "e2e": e2e, "gpu_launches": 2 * args.steps, "clocks": clocks}
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def _timed(call, flush, steps, warmup, stream):
    """Median CUDA-event time (ms) of `steps` calls after `warmup` (at least 3),
    L2 flushed before each when `flush` is given; clocks sampled meanwhile."""
    import torch
    for _ in range(max(3, warmup)):
        if flush is not None:
            flush.zero_()
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(torch.cuda.current_device())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    sampler.start()
    for s_, e_ in ev:
        if flush is not None:
            flush.zero_()
        s_.record(stream)
        call()
        e_.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    times = [s_.elapsed_time(e_) for s_, e_ in ev]
    clocks["ms_mean"] = statistics.fmean(times)
    return statistics.median(times), clocks


def run_workload(args):
    """One JSON line for a non-headline row of the path (device-resident inputs)."""
    import numpy as np
    import torch

    import lossless_draft_verification_gb300 as specv
    from lossless_draft_verification_gb300 import build as _build
    import synth

    _build.build()
    specv.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    td = lambda a, kind=None: torch.from_numpy(np.ascontiguousarray(a if kind is None else a.astype(kind))).to(dev)
    bf = lambda lg: td(lg.raw.view(np.int16)).view(torch.bfloat16)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    peak, peak_kind = _peak_hbm()
    w = args.workload

    def check(st, name):
        if st != 0:
            raise specv.SpecvError(st, name)

    if w in ("greedy", "tv"):
        case = synth.chain_batched(seed=3, R=R, temperature=1.0)
        target, draft = bf(case.target), bf(case.draft)
        if w == "greedy":
            x = td(case.tokens, np.int32)
            acc = torch.empty(R, dtype=torch.int32, device=dev)
            tok = torch.empty(R, dtype=torch.int32, device=dev)
            nb = specv.specv_verify_chain_workspace_size(R, GAMMA, V, specv.SPECV_BF16)
            ws = torch.empty(nb, dtype=torch.uint8, device=dev)
            call = lambda: check(specv.specv_verify_chain(target.data_ptr(), None, specv.SPECV_BF16, x.data_ptr(), None,
                                                          None, R, GAMMA, V, 0.0, acc.data_ptr(), tok.data_ptr(), None,
                                                          ws.data_ptr(), nb, sp), "specv_verify_chain")
            algo = R * (GAMMA + 1) * V * 2
            units, unit, metric = R * GAMMA, "positions/s", "greedy chain verification: verified draft positions/sec"
            desc, launches = "greedy chain verify: R=64, gamma=7, V=151936 bf16, T=0 (target rows only)", 2
            kernel = "argmax tiles + greedy finish (whole call)"
        else:
            cst = torch.empty(R, GAMMA, dtype=torch.float32, device=dev)
            nb = specv.specv_tv_accept_workspace_size(R, GAMMA, V, specv.SPECV_BF16)
            ws = torch.empty(nb, dtype=torch.uint8, device=dev)
            call = lambda: check(specv.specv_tv_accept(target.data_ptr(), draft.data_ptr(), specv.SPECV_BF16, R, GAMMA,
                                                       GAMMA + 1, V, 1.0, cst.data_ptr(), ws.data_ptr(), nb, sp),
                                 "specv_tv_accept")
            algo = 2 * R * GAMMA * V * 2
            units, unit, metric = R * GAMMA, "positions/s", "analytic acceptance c*: (request, position) pairs/sec"
            desc, launches = "tv_accept: R=64, gamma=7, V=151936 bf16, T=1", 2
            kernel = "chain_stats + c* finish (whole call)"
        ms, clocks = _timed(call, flush, args.steps, args.warmup, stream)
        roof = {"bound": "hbm", "achieved": algo / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                "traffic": None, "peak_source": peak_kind, "kernel": kernel, "algorithmic_bytes_per_launch": algo}
    elif w == "tree":
        case = synth.tree_greedy(seed=4)
        Rt, N1, Vt = case.target.raw.shape
        target = bf(case.target)
        par, tks = td(case.parents, np.int32), td(case.tokens, np.int32)
        plen = torch.empty(Rt, dtype=torch.int32, device=dev)
        nodes = torch.empty(Rt, case.max_depth, dtype=torch.int32, device=dev)
        tok = torch.empty(Rt, dtype=torch.int32, device=dev)
        nb = specv.specv_verify_tree_greedy_workspace_size(Rt, N1 - 1, Vt, specv.SPECV_BF16)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        call = lambda: check(specv.specv_verify_tree_greedy(target.data_ptr(), specv.SPECV_BF16, par.data_ptr(),
                                                            tks.data_ptr(), Rt, N1 - 1, Vt, case.max_depth,
                                                            plen.data_ptr(), nodes.data_ptr(), tok.data_ptr(),
                                                            ws.data_ptr(), nb, sp), "specv_verify_tree_greedy")
        algo = Rt * N1 * Vt * 2
        units, unit, metric = Rt * (N1 - 1), "nodes/s", "greedy tree verification: candidate nodes verified/sec"
        desc, launches, kernel = "greedy tree: R=16 trees, 60 nodes + root, depth <= 8, V=151936 bf16", 1, "tree_walk"
        ms, clocks = _timed(call, flush, args.steps, args.warmup, stream)
        roof = {"bound": "hbm", "achieved": algo / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                "traffic": None, "peak_source": peak_kind, "kernel": kernel, "algorithmic_bytes_per_launch": algo}
    elif w in ("markov", "markov_tokens"):
        Rm, Gm, Vm, rank = 512, args.positions or 7, 129280, 256
        m = synth.markov(seed=5, R=Rm, gamma=Gm, V=Vm, rank=rank)
        U, W1, W2 = bf(m.U), bf(m.W1), bf(m.W2)
        anchor, u = td(m.anchor, np.int32), td(m.uniforms, np.float32)
        toks = torch.empty(Rm, Gm, dtype=torch.int32, device=dev)
        keep = w == "markov"
        logits = torch.empty(Rm, Gm, Vm, dtype=torch.float32, device=dev) if keep else None
        nb = specv.specv_markov_draft_workspace_size(Rm, Gm, Vm, rank)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        call = lambda: check(specv.specv_markov_draft(U.data_ptr(), W1.data_ptr(), W2.data_ptr(), anchor.data_ptr(),
                                                      u.data_ptr(), Rm, Gm, Vm, rank, 1.0, toks.data_ptr(),
                                                      logits.data_ptr() if keep else None, specv.SPECV_F32,
                                                      ws.data_ptr(), nb, sp),
                             "specv_markov_draft")
        if keep:
            algo = Gm * (Rm * Vm * 2 + rank * Vm * 2 + Rm * Vm * 4)
        else:
            algo = Gm * Rm * Vm * 2 + rank * Vm * 2     # U once per step, W2 once (it stays in L2 across steps)
        flops = Gm * 2 * Rm * rank * Vm
        units, unit, metric = Rm * Gm, "tokens/s", "Markov-head drafting: draft tokens/sec"
        desc = (f"DSpark Markov head: R=512, gamma={Gm}, V=129280, rank 256, T=1, "
                + ("float32 logits out" if keep else "tokens only (no logits kept)"))
        launches, kernel = 2 * Gm, "markov logits + sample (whole call)"
        ms, clocks = _timed(call, flush, args.steps, args.warmup, stream)
        roof = {"bound": "hbm", "achieved": algo / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                "traffic": None, "peak_source": peak_kind, "kernel": kernel, "algorithmic_bytes_per_launch": algo,
                "tensor_tflops": flops / (ms * 1e-3) / 1e12}
    elif w == "schedule":
        Rs, Gs = 512, 7
        conf = td(synth.confidences(5, Rs, Gs))
        sps = td(synth.sps_table(4096))
        lengths = torch.empty(Rs, dtype=torch.int32, device=dev)
        theta = torch.empty(1, dtype=torch.float64, device=dev)
        nb = specv.specv_schedule_workspace_size(Rs, Gs)
        ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=dev)
        call = lambda: check(specv.specv_schedule(conf.data_ptr(), sps.data_ptr(), Rs, Gs, 4096, lengths.data_ptr(),
                                                  theta.data_ptr(), ws.data_ptr(), ws.numel(), sp), "specv_schedule")
        ms, clocks = _timed(call, None, args.steps, args.warmup, stream)
        units, unit, metric = 1, "schedules/s", "greedy scheduler: schedules/sec (latency-bound)"
        desc, launches, kernel = "scheduler: R=512, gamma=7, SPS table 4096 entries", 1, "schedule"
        roof = {"bound": "latency", "achieved": None, "peak": None, "unit": None, "traffic": None, "kernel": kernel}
    elif w in ("schedule_global", "prune"):
        Rs, Gs = 512, 7
        conf = td(synth.confidences(5, Rs, Gs))
        lengths = torch.empty(Rs, dtype=torch.int32, device=dev)
        ws = torch.empty(256, dtype=torch.uint8, device=dev)
        if w == "schedule_global":
            stale = td(synth.confidences(6, Rs, Gs))
            sps = td(synth.sps_table(4096))
            theta = torch.empty(1, dtype=torch.float64, device=dev)
            call = lambda: check(specv.specv_schedule_global(conf.data_ptr(), stale.data_ptr(), sps.data_ptr(), Rs, Gs,
                                                             4096, lengths.data_ptr(), theta.data_ptr(), ws.data_ptr(),
                                                             ws.numel(), sp), "specv_schedule_global")
            units, unit, metric = 1, "schedules/s", "asynchronous global-search scheduler: schedules/sec (latency-bound)"
            desc, kernel = "global-search scheduler: R=512, gamma=7, stale and current confidences, SPS table 4096", "schedule"
        else:
            call = lambda: check(specv.specv_prune_threshold(conf.data_ptr(), Rs, Gs, 0.5, lengths.data_ptr(),
                                                             ws.data_ptr(), ws.numel(), sp), "specv_prune_threshold")
            units, unit, metric = 1, "prunings/s", "confidence-threshold pruning: calls/sec (latency-bound)"
            desc, kernel = "threshold pruning: R=512, gamma=7, threshold 0.5", "prune"
        ms, clocks = _timed(call, None, args.steps, args.warmup, stream)
        launches = 1
        roof = {"bound": "latency", "achieved": None, "peak": None, "unit": None, "traffic": None, "kernel": kernel}
    elif w == "dart":
        Rt, dt_, Vt, kt, wt, tht = 16, 8, 151936, 25, 20, 59
        xt = bf(synth.make_logits(3.0 * synth.normal(8, 1, (Rt, dt_, Vt)), "bf16"))
        par = torch.empty(Rt, tht + 1, dtype=torch.int32, device=dev)
        tokt = torch.empty(Rt, tht + 1, dtype=torch.int32, device=dev)
        nn = torch.empty(Rt, dtype=torch.int32, device=dev)
        nb = specv.specv_dart_tree_workspace_size(Rt, dt_, Vt, kt, wt, tht, specv.SPECV_BF16)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        call = lambda: check(specv.specv_dart_tree(xt.data_ptr(), specv.SPECV_BF16, Rt, dt_, Vt, 1.0, kt, wt, tht,
                                                   par.data_ptr(), tokt.data_ptr(), nn.data_ptr(), ws.data_ptr(), nb,
                                                   sp), "specv_dart_tree")
        ms, clocks = _timed(call, flush, args.steps, args.warmup, stream)
        algo = Rt * dt_ * Vt * 2
        units, unit, metric = Rt, "trees/s", "DART candidate-tree construction: trees/sec"
        desc, launches, kernel = ("DART tree: R=16, d=8 offsets, V=151936 bf16, top-25, beam 20, 59 nodes", 2,
                                  "whole specv_dart_tree call: dart_topk_tiles reads the logits once (HBM); "
                                  "dart_build, about 70 % of the call, is per-request latency")
        roof = {"bound": "hbm", "achieved": algo / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                "traffic": None, "peak_source": peak_kind, "kernel": kernel, "algorithmic_bytes_per_launch": algo}
    elif w == "confidence":
        Rc, Gc, Hc, Vc, rank = 512, 7, 4096, 129280, 256
        hc = bf(synth.make_logits(synth.normal(7, 1, (Rc, Gc, Hc)), "bf16"))
        W1c = bf(synth.make_logits(0.02 * synth.normal(7, 2, (Vc, rank)), "bf16"))
        wc = td((synth.normal(7, 3, (Hc + rank,)) / np.sqrt(Hc + rank)).astype(np.float32))
        anc = td((synth.uniform_u24(7, 4, (Rc,)) * Vc).astype(np.int32))
        tokc = td((synth.uniform_u24(7, 5, (Rc, Gc)) * Vc).astype(np.int32))
        confo = torch.empty(Rc, Gc, dtype=torch.float32, device=dev)
        ws = torch.empty(256, dtype=torch.uint8, device=dev)
        call = lambda: check(specv.specv_confidence_head(hc.data_ptr(), W1c.data_ptr(), wc.data_ptr(), 0.5, anc.data_ptr(),
                                                         tokc.data_ptr(), Rc, Gc, Hc, Vc, rank, confo.data_ptr(),
                                                         ws.data_ptr(), ws.numel(), sp), "specv_confidence_head")
        ms, clocks = _timed(call, flush, args.steps, args.warmup, stream)
        algo = Rc * Gc * (Hc + rank) * 2 + (Hc + rank) * 4 + Rc * Gc * 4
        units, unit, metric = Rc * Gc, "positions/s", "confidence head: draft positions scored/sec"
        desc, launches, kernel = "confidence head: R=512, gamma=7, H=4096, rank 256, V=129280 bf16", 1, "confidence"
        roof = {"bound": "hbm", "achieved": algo / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                "traffic": None, "peak_source": peak_kind, "kernel": kernel, "algorithmic_bytes_per_launch": algo}
    elif w == "dspark_recompute":
        Rm, Gm, Vm, rank = 512, 7, 129280, 256
        m = synth.markov(seed=5, R=Rm, gamma=Gm, V=Vm, rank=rank)
        tgt = synth.dspark_target(5, m.U)
        U, W1, W2, target = bf(m.U), bf(m.W1), bf(m.W2), bf(tgt)
        anchor, u_m = td(m.anchor, np.int32), td(m.uniforms, np.float32)
        conf = td(synth.confidences(5, Rm, Gm))
        sps = td(synth.sps_table(4096))
        u_v = td(synth.uniform_f32(5, 44, (Rm, Gm + 1, 2)))
        toks = torch.empty(Rm, Gm, dtype=torch.int32, device=dev)
        dlog = torch.empty(Rm, Gm, Vm, dtype=torch.bfloat16, device=dev)
        lengths = torch.empty(Rm, dtype=torch.int32, device=dev)
        theta = torch.empty(1, dtype=torch.float64, device=dev)
        acc = torch.empty(Rm, dtype=torch.int32, device=dev)
        out = torch.empty(Rm, dtype=torch.int32, device=dev)
        cst = torch.empty(Rm, Gm, dtype=torch.float32, device=dev)
        nb_m = specv.specv_markov_draft_workspace_size(Rm, Gm, Vm, rank)
        nb_r = specv.specv_markov_recompute_logits_workspace_size(Rm, Gm)
        nb_v = specv.specv_verify_chain_workspace_size(Rm, Gm, Vm, specv.SPECV_BF16)
        ws_m = torch.empty(nb_m, dtype=torch.uint8, device=dev)
        ws_s = torch.empty(256, dtype=torch.uint8, device=dev)
        ws_r = torch.empty(nb_r, dtype=torch.uint8, device=dev)
        ws_v = torch.empty(nb_v, dtype=torch.uint8, device=dev)

        def call():
            check(specv.specv_markov_draft(U.data_ptr(), W1.data_ptr(), W2.data_ptr(), anchor.data_ptr(),
                                           u_m.data_ptr(), Rm, Gm, Vm, rank, 1.0, toks.data_ptr(), None,
                                           specv.SPECV_BF16, ws_m.data_ptr(), nb_m, sp), "specv_markov_draft")
            check(specv.specv_schedule(conf.data_ptr(), sps.data_ptr(), Rm, Gm, 4096, lengths.data_ptr(),
                                       theta.data_ptr(), ws_s.data_ptr(), 256, sp), "specv_schedule")
            check(specv.specv_markov_recompute_logits(U.data_ptr(), W1.data_ptr(), W2.data_ptr(), anchor.data_ptr(),
                                                      toks.data_ptr(), lengths.data_ptr(), Rm, Gm, Vm, rank,
                                                      dlog.data_ptr(), ws_r.data_ptr(), nb_r, sp),
                  "specv_markov_recompute_logits")
            check(specv.specv_verify_chain(target.data_ptr(), dlog.data_ptr(), specv.SPECV_BF16, toks.data_ptr(),
                                           lengths.data_ptr(), u_v.data_ptr(), Rm, Gm, Vm, 1.0, acc.data_ptr(),
                                           out.data_ptr(), cst.data_ptr(), ws_v.data_ptr(), nb_v, sp),
                  "specv_verify_chain")
        ms, clocks = _timed(call, flush, args.steps, args.warmup, stream)
        ell = lengths.cpu().numpy().astype(np.int64)
        verified = int(ell.sum())
        live = int(ell.sum())
        # drafting: U once per step + W2 once; recompute: the live U rows + W2 + the live rows written;
        # verification: the live target rows + bonus rows and the live draft rows
        algo = (Gm * Rm * Vm * 2 + rank * Vm * 2) + (live * Vm * 2 + rank * Vm * 2 + live * Vm * 2) + \
            int(((ell + 1) * Vm * 2 + ell * Vm * 2).sum())
        units, unit, metric = verified, "positions/s", "DSpark round (draft, schedule, verify): verified draft positions/sec"
        desc = (f"DSpark round without kept draft logits: Markov head R=512, gamma=7, V=129280, rank 256 (tokens only, "
                f"bf16 draw precision); scheduler lengths (sum {verified}); the verified rows' draft logits recomputed; "
                f"chain verification T=1")
        launches, kernel = 2 * Gm + 1 + 2 + 2, "markov + schedule + recompute + verify (whole round)"
        roof = {"bound": "hbm", "achieved": algo / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                "traffic": None, "peak_source": peak_kind, "kernel": kernel, "algorithmic_bytes_per_launch": algo}
    elif w == "dspark":
        Rm, Gm, Vm, rank = 512, 7, 129280, 256
        m = synth.markov(seed=5, R=Rm, gamma=Gm, V=Vm, rank=rank)
        tgt = synth.dspark_target(5, m.U)
        U, W1, W2, target = bf(m.U), bf(m.W1), bf(m.W2), bf(tgt)
        anchor, u_m = td(m.anchor, np.int32), td(m.uniforms, np.float32)
        conf = td(synth.confidences(5, Rm, Gm))
        sps = td(synth.sps_table(4096))
        u_v = td(synth.uniform_f32(5, 44, (Rm, Gm + 1, 2)))
        toks = torch.empty(Rm, Gm, dtype=torch.int32, device=dev)
        dlog = torch.empty(Rm, Gm, Vm, dtype=torch.bfloat16, device=dev)
        lengths = torch.empty(Rm, dtype=torch.int32, device=dev)
        theta = torch.empty(1, dtype=torch.float64, device=dev)
        acc = torch.empty(Rm, dtype=torch.int32, device=dev)
        out = torch.empty(Rm, dtype=torch.int32, device=dev)
        cst = torch.empty(Rm, Gm, dtype=torch.float32, device=dev)
        nb_m = specv.specv_markov_draft_workspace_size(Rm, Gm, Vm, rank)
        nb_v = specv.specv_verify_chain_workspace_size(Rm, Gm, Vm, specv.SPECV_BF16)
        ws_m = torch.empty(nb_m, dtype=torch.uint8, device=dev)
        ws_s = torch.empty(256, dtype=torch.uint8, device=dev)
        ws_v = torch.empty(nb_v, dtype=torch.uint8, device=dev)

        def call():
            check(specv.specv_markov_draft(U.data_ptr(), W1.data_ptr(), W2.data_ptr(), anchor.data_ptr(),
                                           u_m.data_ptr(), Rm, Gm, Vm, rank, 1.0, toks.data_ptr(), dlog.data_ptr(),
                                           specv.SPECV_BF16, ws_m.data_ptr(), nb_m, sp), "specv_markov_draft")
            check(specv.specv_schedule(conf.data_ptr(), sps.data_ptr(), Rm, Gm, 4096, lengths.data_ptr(),
                                       theta.data_ptr(), ws_s.data_ptr(), 256, sp), "specv_schedule")
            check(specv.specv_verify_chain(target.data_ptr(), dlog.data_ptr(), specv.SPECV_BF16, toks.data_ptr(),
                                           lengths.data_ptr(), u_v.data_ptr(), Rm, Gm, Vm, 1.0, acc.data_ptr(),
                                           out.data_ptr(), cst.data_ptr(), ws_v.data_ptr(), nb_v, sp),
                  "specv_verify_chain")
        ms, clocks = _timed(call, flush, args.steps, args.warmup, stream)
        ell = lengths.cpu().numpy().astype(np.int64)
        verified = int(ell.sum())
        algo = Gm * (Rm * Vm * 2 + rank * Vm * 2 + Rm * Vm * 2) + int(((ell + 1) * Vm * 2 + ell * Vm * 2).sum())
        units, unit, metric = verified, "positions/s", "DSpark round (draft, schedule, verify): verified draft positions/sec"
        desc = (f"DSpark round: Markov head R=512, gamma=7, V=129280, rank 256, bf16 logits; scheduler lengths "
                f"(sum {verified}); chain verification T=1")
        launches, kernel = 2 * Gm + 1 + 2, "markov + schedule + verify (whole round)"
        roof = {"bound": "hbm", "achieved": algo / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                "traffic": None, "peak_source": peak_kind, "kernel": kernel, "algorithmic_bytes_per_launch": algo}
    else:
        raise SystemExit(f"unknown workload {w}")
    if roof.get("achieved") is not None:
        roof["frac"] = roof["achieved"] / roof["peak"]
    out = {"metric": metric, "value": units / (ms * 1e-3), "unit": unit, "n_gpus": 1, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16", "data": "synthetic",
           "config": {"workload": desc, "l2": "flushed (2x L2 write) before every timed step"
                      if w not in ("schedule", "schedule_global", "prune") else "inputs are a few KB (L2-resident)"},
           "roofline": roof, "gpu_launches": None if launches is None else launches * args.steps, "clocks": clocks}
    print(json.dumps(out), flush=True)
    return 0


def main():
    global R, ALGO_BYTES, WORKLOAD
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--flush-l2", action="store_true", help="headline: flush L2 before every timed step")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--requests", type=int, default=64, help="R (smaller for profiling captures)")
    ap.add_argument("--workload", default="chain",
                    choices=["chain", "greedy", "tv", "tree", "markov", "markov_tokens", "schedule", "schedule_global", "prune", "confidence", "dart", "dspark", "dspark_recompute"])
    ap.add_argument("--positions", type=int, default=0, help="Markov workload: draft positions (default 7)")
    args = ap.parse_args()
    world = os.environ.get("WORLD_SIZE")
    if args.gpus > 1 and world is None:
        # one process per GPU: relaunch this command under torchrun
        import socket
        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            port = so.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
        return subprocess.call(cmd)
    if world is not None and int(world) != args.gpus:
        sys.stderr.write(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}\n")
        return 2
    if args.requests != R:
        R = args.requests
        ALGO_BYTES = R * (GAMMA + 1) * V * 2 + R * GAMMA * V * 2
        WORKLOAD = WORKLOAD.replace("R=64", f"R={R}")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "chain":
        return run_workload(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
