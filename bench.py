#!/usr/bin/env python
"""Benchmark of the JoLT KV-cache encode/decode path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--configs A,B,...|none]

One step = the whole hot path over one batch of synthetic units: factor
(ST-HOSVD) -> sweep of the full (r_T, r_d, b) grid -> Lagrangian allocation ->
serialization of the chosen candidates, then decode of every unit back to
bf16.  `value` is encode GB/s: 16-bit-equivalent input bytes of all units /
encode time; decode GB/s is reported beside it.  Inputs are resident in HBM
when a timed step starts; L2 is flushed (a 256 MiB write) between steps,
outside the timed events.  `e2e` repeats the encode through the same public
calls from pinned host memory: host-to-device copy of X and signs, encode,
device-to-host copy of the blobs, all inside the timed region.

The line's workload is the largest single-GPU configuration, the LLaMA-2-13B
shaped cache (20 units of [160, 1024, 128] bf16).  `configs` adds one record
per other large configuration (Mistral-7B shaped at 1024 and 2048 tokens, and
the 4096-token FlashJoLT case with its decode of all 16 units back to bf16),
each timed the same way.

--impl reference times the float64 CPU oracle (oracle/) on a bounded sample
of the same workload: one token window of each of P units, P = min(units,
host cores), one single-threaded process per unit.

Under torchrun (N > 1) every rank runs an independent replica of the
workload (no data-path collective); the timed region is bracketed by
barriers and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import kvgen  # noqa: E402

METRIC = "KV encode GB/s (full (r_T,r_d,b) sweep+alloc) and decode GB/s, 1×B300"
L2_BYTES = 126 * 2 ** 20
MAIN_WORKLOAD = "llama_t1024"
EXTRA_CONFIGS = ("mistral_t1024", "mistral_t2048", "flash_t4096")
THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6400.0), "measured", d
    return 6400.0, "fallback", {}


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 50 ms; the summary keeps the samples that
    arrived between mark_start() and mark_end() (the timed region).  Entering
    waits (up to 5 s) for the first sample, so the sampler is live before the
    region starts."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.span = (0, None)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.perf_counter()
            while not self.lines and self.proc.poll() is None and time.perf_counter() - t0 < 5.0:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def mark_start(self):
        self.span = (len(self.lines), None)

    def mark_end(self):
        self.span = (self.span[0], len(self.lines))

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines[self.span[0]:self.span[1]]:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- dist
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(backend):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as tdist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        tdist.init_process_group(backend, rank=rank, world_size=ws)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as tdist
        tdist.barrier()


def max_over_ranks(ws, v: float, device=None) -> float:
    if ws <= 1:
        return v
    import torch
    import torch.distributed as tdist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- process pools
class single_threaded_children:
    """Environment for spawned children: one BLAS/OpenMP thread each (the
    variables are read when a child imports numpy)."""

    def __enter__(self):
        self.saved = {k: os.environ.get(k) for k in THREAD_VARS}
        for k in THREAD_VARS:
            os.environ[k] = "1"
        return self

    def __exit__(self, *a):
        for k, v in self.saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def workload(name, groups=0):
    """The named workload, or the same shapes and generator with only its
    first `groups` layer groups (a smaller batch of identical units, for
    profiling runs)."""
    if groups:
        return kvgen.custom_workload(name, n_groups=groups)
    return kvgen.WORKLOADS[name]


def _gen_unit(task):
    name, groups, u = task
    w = workload(name, groups)
    x = kvgen.make_unit(w, u)
    s = kvgen.make_signs(w, u)
    sk = kvgen.make_sketch(w, u) if w.token_mode == "randomized" else None
    return name, u, x, s, sk


def gen_inputs(names, procs=None, groups=0):
    """Host inputs of every unit of each named workload, generated by a pool
    of spawned processes (before any CUDA call of this process):
    {name: (list of stored unit arrays, signs [U][D], sketch [U][H][D][ell] or None)}."""
    nu = {n: workload(n, groups).n_units for n in names}
    tasks = [(n, groups, u) for n in names for u in range(nu[n])]
    procs = max(1, min(procs or (os.cpu_count() or 1), len(tasks)))
    out = {n: ([None] * nu[n], [None] * nu[n], [None] * nu[n]) for n in names}
    if procs == 1:
        results = map(_gen_unit, tasks)
    else:
        with single_threaded_children():
            pool = mp.get_context("spawn").Pool(procs)
        results = pool.imap_unordered(_gen_unit, tasks)
    for name, u, x, s, sk in results:
        out[name][0][u] = x
        out[name][1][u] = s
        out[name][2][u] = sk
    if procs > 1:
        pool.close()
        pool.join()
    res = {}
    for n, (xs, ss, sks) in out.items():
        res[n] = (xs, np.stack(ss), None if sks[0] is None else np.stack(sks))
    return res


# ----------------------------------------------------------------- CPU oracle
def oracle_window(w) -> int:
    """Tokens of the oracle's sample window: the whole unit up to 128 tokens,
    else 48 (above every truncated token rank of the grid)."""
    return w.T if w.T <= 128 else 48


def _oracle_unit(task):
    """One process of the CPU baseline: the float64 oracle, as it stands, on
    a token window of one unit (all heads and features).  Returns (input
    bytes, seconds, BLAS threads of this process)."""
    name, u = task
    from oracle import run as orun
    w = kvgen.WORKLOADS[name]
    tw = oracle_window(w)
    x = kvgen.unit_values_f64(w, kvgen.make_unit(w, u))[:, :tw, :].copy()
    s = kvgen.make_signs(w, u)
    sk = None
    if w.token_mode == "randomized":
        sk = [kvgen.make_sketch(w, u).astype(np.float64)]
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:
        threads = 1
    t = time.perf_counter()
    orun.encode_units([x], [s], w.rT, w.rd, w.bits, w.block, 10 ** 12, token_mode=w.token_mode,
                      sketches=sk, power_iters=w.power_iters, serialize=True)
    return x.size * 2, time.perf_counter() - t, int(threads)


class OraclePool:
    """P = min(units, host cores) spawned single-threaded processes; a sample
    runs the oracle on one token window of each of units 0 .. P-1 at once."""

    def __init__(self, name):
        self.name = name
        w = kvgen.WORKLOADS[name]
        self.P = max(1, min(w.n_units, os.cpu_count() or 1))
        with single_threaded_children():
            self.pool = mp.get_context("spawn").Pool(self.P)
        self.pool.map(int, range(self.P))      # the workers are up before timing

    def sample(self):
        t = time.perf_counter()
        res = self.pool.map(_oracle_unit, [(self.name, u) for u in range(self.P)], chunksize=1)
        wall = time.perf_counter() - t
        nbytes = sum(r[0] for r in res)
        threads = sum(r[2] for r in res)
        w = kvgen.WORKLOADS[self.name]
        desc = (f"oracle encode (factor, full grid, allocation, serialization) of a "
                f"{oracle_window(w)}-token window of units 0..{self.P - 1} "
                f"({w.H}x{oracle_window(w)}x{w.D} each, f64), one single-threaded process "
                f"per unit")
        return nbytes, wall, threads, desc

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline_record(name, samples=1):
    pool = OraclePool(name)
    try:
        tb, tt = 0, 0.0
        for _ in range(samples):
            b, dt, threads, desc = pool.sample()
            tb += b
            tt += dt
    finally:
        pool.close()
    return {"value": tb / tt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": desc, "host_cpu_count": os.cpu_count(), "cpu_model": cpu_model(),
            "processes": pool.P, "wall_s_per_sample": tt / samples}


def run_reference(args):
    ws, rank, _ = init_dist("gloo")
    if rank != 0:
        return
    pool = OraclePool(args.workload)
    try:
        for _ in range(args.warmup):
            pool.sample()
        tot_b, tot_t = 0, 0.0
        threads, sample = 1, ""
        for _ in range(args.steps):
            b, dt, threads, sample = pool.sample()
            tot_b += b
            tot_t += dt
    finally:
        pool.close()
    gbs = tot_b / tot_t / 1e9
    line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": args.workload, "sample": sample},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": sample, "host_cpu_count": os.cpu_count(),
                             "cpu_model": cpu_model()},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU path
STAGES = ("factor", "sweep", "allocate", "encode", "decode")


class Run:
    """The device state of one workload: inputs, encoder, output buffer."""

    def __init__(self, w, host):
        import torch
        from partial_tucker_rotated_st_b300 import codec
        self.w = w
        xs, signs, sk = host
        arr = np.ascontiguousarray(np.stack(xs))
        Xh = torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16) if w.dtype == "bf16" \
            else torch.from_numpy(arr)
        self.Xh = Xh.pin_memory()
        self.Sh = torch.from_numpy(signs).pin_memory()
        self.X = self.Xh.cuda()
        self.S = self.Sh.cuda()
        self.K = None if sk is None else torch.from_numpy(sk).cuda()
        self.cfg = codec.config_for(w)
        self.enc = codec.Encoder(self.cfg, w.n_units)
        self.xhat = torch.empty(w.n_units, w.H, w.T, w.D, dtype=torch.bfloat16, device="cuda")
        self.in_bytes = 2 * w.elems_per_unit * w.n_units      # 16-bit-equivalent bytes


def timed_steps(run, steps, warmup, flush, st, clk=None):
    """Warm-up, then `steps` timed steps; per-stage device time (CUDA events
    on the launching stream), the fused sweep kernel's own time (events the
    library records around its launch), the decoder's time, host wall time
    and library launches per step."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    enc, w = run.enc, run.w

    def step(timers=None):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
        kev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for e in kev:
            e.record(st)   # creates the CUDA event; the library records it again
        ev[0].record(st)
        enc.factor(run.X, run.K)
        ev[1].record(st)
        J.jolt_set_sweep_events(*kev)
        enc.sweep(run.X, run.S)
        J.jolt_set_sweep_events()
        ev[2].record(st)
        enc.allocate(w.budget_bytes, refine=True)
        ev[3].record(st)
        enc.choice_host.copy_(enc.choice, non_blocking=True)
        st.synchronize()
        desc = enc.serialize(run.X, run.S, enc.choice_host.tolist())
        ev[4].record(st)
        codec.decode(desc, enc.blob, enc.stride, J.BF16, out=run.xhat)
        ev[5].record(st)
        if timers is not None:
            timers.append((ev, kev))
        return desc

    for _ in range(warmup):
        step()
        flush.fill_(1)
    st0 = enc.status()
    if st0 != J.OK:
        raise SystemExit(f"{w.name}: device status {J.jolt_status_string(st0)}")
    timers = []
    torch.cuda.synchronize()
    n0 = J.jolt_launch_count()
    if clk is not None:
        clk.mark_start()
    t0 = time.perf_counter()
    desc = None
    for _ in range(steps):
        desc = step(timers)
        flush.fill_(1)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if clk is not None:
        clk.mark_end()
    launches = (J.jolt_launch_count() - n0) // max(steps, 1)
    per = {s: 0.0 for s in STAGES}
    sweep_k = 0.0
    for ev, kev in timers:
        for i, s in enumerate(STAGES):
            per[s] += ev[i].elapsed_time(ev[i + 1]) / 1e3
        sweep_k += kev[0].elapsed_time(kev[1]) / 1e3
    per = {s: v / steps for s, v in per.items()}
    st1 = enc.status()
    if st1 != J.OK:
        raise SystemExit(f"{w.name}: device status {J.jolt_status_string(st1)}")
    return {"per": per, "sweep_kernel_s": sweep_k / steps, "wall_s": wall / steps,
            "launches": int(launches), "desc": desc}


def factor_record(run, steps, flush, st, pk):
    """The factor step alone with its stage-boundary events: the feature
    stage (side stream), the whole-feature token solve (caller's stream),
    the truncated token solves after the join, the cores; its dense
    contractions' algorithmic flops against the sustained bf16 tensor peak
    (the step is a chain of small latency-bound solves, so the fraction is
    small by construction)."""
    import torch
    from partial_tucker_rotated_st_b300 import jolt as J
    w, enc = run.w, run.enc
    acc = {k: 0.0 for k in ("feature", "full_token_solve", "truncated_solves", "cores", "total")}
    for i in range(steps + 2):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        for e in ev:
            e.record(st)
        J.jolt_set_factor_events(ev)
        enc.factor(run.X, run.K)
        J.jolt_set_factor_events()
        torch.cuda.synchronize()
        flush.fill_(1)
        if i < 2:
            continue
        acc["feature"] += ev[0].elapsed_time(ev[1])
        acc["full_token_solve"] += ev[0].elapsed_time(ev[2])
        acc["truncated_solves"] += min(ev[1].elapsed_time(ev[3]), ev[2].elapsed_time(ev[3]))
        acc["cores"] += ev[3].elapsed_time(ev[4])
        acc["total"] += ev[0].elapsed_time(ev[4])
    ms = {k: v / steps for k, v in acc.items()}
    H, T, D, U = w.H, w.T, w.D, w.n_units
    RT = max(r for r in w.rT if r != kvgen.FULL)
    RD = max(r for r in w.rd if r != kvgen.FULL)
    N = H * T * D
    flops_unit = (2 * N * D                       # feature Gram
                  + 2 * N * RD                    # projection Y = X U_d
                  + 2 * T * T * H * RD            # truncated token Grams (prefix slabs)
                  + 2 * N * RT * len(w.rd))       # cores Z = X_h^T U_T of every rank
    if w.token_mode == "exact":
        flops_unit += 2 * T * T * H * D           # whole-feature token Gram
    else:
        # FlashJoLT: Z = A Omega, then q times A^T Q and A (A^T Q), and the
        # final A^T Q, each 2 H T r_d ell for every feature rank
        ell = RT + w.oversample
        rds = sum(w.D if r == kvgen.FULL else r for r in w.rd)
        flops_unit += (2 + 2 * w.power_iters) * 2 * H * T * rds * ell
    flops = flops_unit * U
    peak = pk.get("bf16_tflops_sustained", 1400.0)
    crit = "feature" if ms["feature"] >= ms["full_token_solve"] else "full_token_solve"
    return {"stages_ms": ms, "critical_path": [crit, "truncated_solves", "cores"],
            "dense_flops": int(flops),
            "dense_tflops_achieved": flops / (ms["total"] / 1e3) / 1e12,
            "peak_tflops": peak, "peak_kind": "measured bf16 sustained",
            "frac": flops / (ms["total"] / 1e3) / 1e12 / peak}


def blob_bytes_of(desc):
    return sum(int(d.bytes) for d in desc)


def decode_roofline(w, desc, dec_t, hbm):
    alg = blob_bytes_of(desc) + 2 * w.elems_per_unit * w.n_units
    return {"kernel": "decode_tc_kernel", "bound": "hbm", "achieved": alg / dec_t / 1e9,
            "peak": hbm, "unit": "GB/s", "frac": alg / dec_t / 1e9 / hbm,
            "bytes_algorithmic": int(alg), "traffic": decode_traffic(w)}


def e2e_pipelined(args, run, st):
    """Encode end to end through the public calls (Encoder.encode and
    blobs_to_host) from pinned host memory: every step copies its X and
    signs host to device and reads its serialized blobs back.  Two encoders
    and two input buffers alternate so that the copies run on two more
    streams (host to device, device to host: the link is full duplex) beside
    the neighbouring steps' compute (step i + 1's inputs go in, and step
    i - 1's blobs come out, while step i computes); each buffer is reused
    only after the copies and compute that read it are done.  The
    inputs (bigger than L2) change buffer every step, so no L2 flush is
    needed.  Returns the record (with the mean seconds per step under
    "_s_per_step") and the last step's result."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    w = run.w
    encs = [run.enc, codec.Encoder(run.cfg, w.n_units)]
    Xd = [run.X, torch.empty_like(run.X)]
    Sd = [run.S, torch.empty_like(run.S)]
    host = [torch.empty(w.n_units * e.stride, dtype=torch.uint8, pin_memory=True) for e in encs]
    cs = torch.cuda.Stream()               # host to device
    co = torch.cuda.Stream()               # device to host
    d2h = [0]
    last = [None]

    def pipeline(n):
        h2d_done = [torch.cuda.Event() for _ in range(n)]
        comp_done = [torch.cuda.Event() for _ in range(n)]
        d2h_done = [torch.cuda.Event() for _ in range(n)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)

        def h2d(i):
            b = i % 2
            with torch.cuda.stream(cs):
                if i >= 2:
                    cs.wait_event(comp_done[i - 2])     # the buffer's last reader is done
                Xd[b].copy_(run.Xh, non_blocking=True)
                Sd[b].copy_(run.Sh, non_blocking=True)
                h2d_done[i].record(cs)

        t0.record(cs)
        h2d(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                h2d(i + 1)
            st.wait_event(h2d_done[i])
            if i >= 2:
                st.wait_event(d2h_done[i - 2])          # this encoder's blobs are out
            r = encs[b].encode(Xd[b], Sd[b], w.budget_bytes, run.K)
            comp_done[i].record(st)
            co.wait_event(comp_done[i])
            d2h[0] = encs[b].blobs_to_host(r.desc, host[b], stream=co)
            d2h_done[i].record(co)
            last[0] = (r, encs[b])
        t1.record(co)
        t1.synchronize()
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / 1e3

    pipeline(max(args.warmup, 2))
    t = pipeline(args.steps)
    rec = {"unit": "GB/s",
           "h2d_bytes_per_step": int(run.Xh.numel() * run.Xh.element_size() + run.Sh.numel()),
           "d2h_bytes_per_step": int(d2h[0]),
           "pipelined": "two encoders; each step's H2D copy and blob read-back on two copy "
                        "streams, overlapping the neighbouring steps' compute; timed from the "
                        "first copy to the last read-back",
           "_s_per_step": t / args.steps}
    r, e = last[0]
    if e is not run.enc:
        run.enc, encs[1] = e, run.enc                   # the encoder holding the last blobs
        run.X, Xd[1] = Xd[1], run.X
        run.S, Sd[1] = Sd[1], run.S
    return rec, r


def config_record(run, res, hbm, kind, pk, sms, fac=None):
    """Per-configuration record: encode and decode GB/s, stage times, the
    factor step's stage breakdown, the fused sweep's and the decoder's
    rooflines."""
    w = run.w
    per = res["per"]
    enc_t = per["factor"] + per["sweep"] + per["allocate"] + per["encode"]
    return {"workload": w.name, "units": w.n_units, "unit_shape": [w.H, w.T, w.D],
            "token_mode": w.token_mode, "budget_bytes": w.budget_bytes,
            "encode_gbs": run.in_bytes / enc_t / 1e9,
            "decode_gbs": run.in_bytes / per["decode"] / 1e9,
            "decode_output": f"bf16 [{w.n_units}][{w.H}][{w.T}][{w.D}]",
            "stages_ms": {s: 1e3 * v for s, v in per.items()},
            "sweep_roofline": roofline(w, res["sweep_kernel_s"], hbm, kind, pk, sms),
            "decode_roofline": decode_roofline(w, res["desc"], per["decode"], hbm),
            "factor": fac,
            "gram_tensor": gram_tensor_record(w),
            "gpu_launches": res["launches"]}


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    names = [args.workload] + [c for c in args.configs if c != args.workload]
    host = gen_inputs(names, max(1, (os.cpu_count() or 1) // ws), args.groups)   # before any CUDA call
    ws, rank, local = init_dist("nccl")
    torch.cuda.set_device(local)
    from partial_tucker_rotated_st_b300 import build as jbuild
    jbuild.build()
    from partial_tucker_rotated_st_b300 import jolt as J

    sms = torch.cuda.get_device_properties(local).multi_processor_count
    hbm, kind, pk = peaks()
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()

    # ---- the line's workload
    w = workload(args.workload, args.groups)
    run = Run(w, host.pop(args.workload))
    torch.cuda.synchronize()
    barrier(ws)
    with ClockSampler(local) as clk:
        res = timed_steps(run, args.steps, args.warmup, flush, st, clk)
    barrier(ws)
    per = res["per"]
    enc_t = per["factor"] + per["sweep"] + per["allocate"] + per["encode"]
    enc_t = max_over_ranks(ws, enc_t, "cuda")
    dec_t = max_over_ranks(ws, per["decode"], "cuda")
    value = ws * run.in_bytes / enc_t / 1e9
    dec_gbs = ws * run.in_bytes / dec_t / 1e9
    desc = res["desc"]

    # end to end through the public calls, from pinned host memory
    e2e, r = e2e_pipelined(args, run, st)
    enc = run.enc                          # the encoder holding the last step's blobs
    e2e_t = max_over_ranks(ws, e2e.pop("_s_per_step"), "cuda")
    e2e["value"] = ws * run.in_bytes / e2e_t / 1e9

    fac = factor_record(run, args.steps, flush, st, pk)
    attn = attention_bench(args, w, r.desc, enc, flush, st, hbm, kind)
    adm = admission_bench(args, w, r.desc, enc, flush, st)
    modeled = modeled_allocator(args, w, enc, run.X, run.K, run.S, w.budget_bytes, run.in_bytes,
                                flush, st, ws)
    dom = max(("factor", "sweep", "encode", "decode"), key=lambda s: per[s])
    roof = roofline(w, res["sweep_kernel_s"], hbm, kind, pk, sms)
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * (enc_t + dec_t),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": args.workload, "units": w.n_units,
                       "unit_shape": [w.H, w.T, w.D],
                       "input": "bf16" if w.dtype == "bf16" else "f32",
                       "budget_bytes": w.budget_bytes, "token_mode": w.token_mode,
                       "allocator": "lambda bisection + greedy swaps",
                       "l2": "flushed between steps (256 MiB write)",
                       "parallelism": f"replicas{ws}",
                       **({"groups": args.groups} if args.groups else {})},
            "decode": {"value": dec_gbs, "unit": "GB/s",
                       "roofline": decode_roofline(w, desc, dec_t, hbm)},
            "stages_ms": {s: 1e3 * v for s, v in per.items()},
            "dominant_stage": dom,
            "factor": fac,
            "gram_tensor": gram_tensor_record(w),
            "wall_ms_per_step": 1e3 * res["wall_s"],
            "roofline": roof,
            "e2e": e2e,
            "modeled_allocator": modeled,
            "attention": attn,
            "admission": adm,
            "gpu_launches": res["launches"],
            "sm_count": sms,
            "clocks": clk.summary()}
    del run, r, enc
    torch.cuda.empty_cache()

    # ---- one record per other configuration, timed the same way
    recs = {}
    for name in args.configs:
        if name == args.workload:
            continue
        wx = workload(name, args.groups)
        rx = Run(wx, host.pop(name))
        resx = timed_steps(rx, args.steps, args.warmup, flush, st)
        facx = factor_record(rx, args.steps, flush, st, pk)
        recs[name] = config_record(rx, resx, hbm, kind, pk, sms, facx)
        del rx
        torch.cuda.empty_cache()
    line["configs"] = recs

    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_record(args.workload)
    if rank == 0:
        print(json.dumps(line), flush=True)


SWEEP_SRC = os.path.join(ROOT, "partial_tucker_rotated_st_b300", "csrc", "sweep_tc.cu")


def attention_bench(args, w, desc, enc, flush, st, hbm, hbm_kind, nq=4):
    """Attention of nq queries per head over every group's compressed K and V
    (the blobs of the last encode), through jolt_attend, against
    materializing the cache (jolt_decode to bf16) and running torch's
    scaled_dot_product_attention on it.  L2 is flushed before every call.
    Algorithmic bytes: the sections of every blob (U_T, U_d, G, scales,
    codes) plus the queries and the outputs."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    G, H, T, D = len(desc) // 2, w.H, w.T, w.D
    rng = np.random.default_rng(20260102)
    q = torch.from_numpy(rng.standard_normal((G, H, nq, D)).astype(np.float32)).cuda()
    scale = 1.0 / float(np.sqrt(D))
    aws = torch.empty(J.jolt_attend_workspace_size(G, H, T, D, nq), dtype=torch.uint8,
                      device="cuda")
    out = torch.empty_like(q)
    xhat = torch.empty(2 * G, H, T, D, dtype=torch.bfloat16, device="cuda")
    qb = q.to(torch.bfloat16)

    def fused():
        codec.attend(desc, enc.blob, enc.stride, q, scale, out=out, ws=aws)

    def materialize():
        codec.decode(desc, enc.blob, enc.stride, J.BF16, out=xhat)
        torch.nn.functional.scaled_dot_product_attention(qb, xhat[0::2], xhat[1::2], scale=scale)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
            flush.fill_(1)
        tot = 0.0
        for _ in range(args.steps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            e1.synchronize()
            tot += e0.elapsed_time(e1) / 1e3
            flush.fill_(1)
        return tot / args.steps

    n0 = J.jolt_launch_count()
    t = timed(fused)
    launches = (J.jolt_launch_count() - n0) // (args.warmup + args.steps)
    tm = timed(materialize)
    sec = 0
    for d in desc:
        sec += (2 * T * d.rT if d.rT < T else 0) + (2 * D * d.rd if d.rd < D else 0)
        sec += 2 * H * d.rT * d.rd
        if d.b > 0:
            sec += 2 * H * T + H * T * D * d.b // 8
    alg = sec + 2 * q.numel() * 4
    return {"ms": 1e3 * t, "queries_per_call": G * H * nq, "tokens": T, "nq_per_head": nq,
            "launches_per_call": int(launches),
            "roofline": {"kernel": "attend_prep + attend_chunk + attend_merge (one call)",
                         "bound": "hbm", "achieved": alg / t / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": alg / t / 1e9 / hbm, "traffic": attend_traffic(w),
                         "bytes_algorithmic": int(alg), "peak_kind": hbm_kind},
            "materialize_then_sdpa_ms": 1e3 * tm,
            "speedup_vs_materialize": tm / t}


def admission_bench(args, w, desc, enc, flush, st, tau=128):
    """Admission of tau new tokens into every unit of the last encode
    (jolt_admit: fold-in under the fixed factors, residual coded), timed
    like the main step; GB/s of 16-bit-equivalent new-token input."""
    import torch
    from partial_tucker_rotated_st_b300 import codec
    from partial_tucker_rotated_st_b300 import jolt as J
    U = len(desc)
    rng = np.random.default_rng(20260103)
    xn = kvgen.round_to_bf16(rng.standard_normal((U, w.H, tau, w.D)).astype(np.float32))
    X = torch.from_numpy(xn.view(np.int16)).view(torch.bfloat16).cuda()
    sout = codec.admit_stride(enc.stride, w.H, tau, w.D)
    out = torch.empty(U, sout, dtype=torch.uint8, device="cuda")
    aws = torch.empty(J.jolt_admit_workspace_size(U, w.H, tau, w.D), dtype=torch.uint8,
                      device="cuda")

    def call():
        codec.admit(desc, enc.blob, enc.stride, X, out=out, ws=aws)

    for _ in range(args.warmup):
        call()
        flush.fill_(1)
    n0 = J.jolt_launch_count()
    tot = 0.0
    for _ in range(args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        call()
        e1.record(st)
        e1.synchronize()
        tot += e0.elapsed_time(e1) / 1e3
        flush.fill_(1)
    t = tot / args.steps
    nbytes = U * w.H * tau * w.D * 2
    return {"ms": 1e3 * t, "new_tokens": tau, "units": U, "unit": "GB/s",
            "value": nbytes / t / 1e9,
            "launches_per_call": int((J.jolt_launch_count() - n0) // max(args.steps, 1))}


def modeled_allocator(args, w, enc, X, K, S, budget, in_bytes, flush, st, ws):
    """The modeled-error allocation path (no sweep): factor -> modeled table
    from the spectra -> bisection -> serialize, timed like the main step; and
    the measured distortion of its choice against the measured-table choice
    (both from the last main step's tables, same budget)."""
    import torch
    from partial_tucker_rotated_st_b300 import jolt as J
    rng = np.random.default_rng(20260101)
    rows = torch.from_numpy(rng.standard_normal((8192, w.D)).astype(np.float32)).cuda()
    scratch = torch.zeros(8, dtype=torch.float64, device="cuda")
    eps2 = torch.zeros(len(w.bits), dtype=torch.float64, device="cuda")
    J.jolt_calibrate_eps2(rows, list(w.bits), scratch, eps2)
    eps2_h = eps2.cpu().tolist()
    U = enc.U
    md = torch.zeros(U, enc.ncand, dtype=torch.float64, device="cuda")
    ch = torch.zeros(U, dtype=torch.int32, device="cuda")
    lam = torch.zeros(1, dtype=torch.float64, device="cuda")
    stt = torch.zeros(1, dtype=torch.int32, device="cuda")
    ch_host = torch.empty(U, dtype=torch.int32, pin_memory=True)
    dist_meas = enc.dist.clone()
    cost = enc.cost.clone()
    choice_meas = enc.choice.clone()

    def step():
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        enc.factor(X, K)
        J.jolt_model_candidates(enc.cfg, U, enc.ws, eps2_h, md)
        J.jolt_allocate(U, enc.ncand, md, cost, budget, enc.cfg.align, ch, lam, stt)
        ch_host.copy_(ch, non_blocking=True)
        st.synchronize()
        enc.serialize(X, S, ch_host.tolist())
        e1.record(st)
        return e0, e1

    for _ in range(args.warmup):
        step()
        flush.fill_(1)
    tot = 0.0
    for _ in range(args.steps):
        e0, e1 = step()
        e1.synchronize()
        tot += e0.elapsed_time(e1) / 1e3
        flush.fill_(1)
    t = max_over_ranks(ws, tot / args.steps, "cuda")
    dm, cm, zm = dist_meas.cpu().numpy(), cost.cpu().numpy(), choice_meas.cpu().numpy()
    zmod = ch.cpu().numpy()
    idx = np.arange(U)
    return {"encode_gbs": ws * in_bytes / t / 1e9, "unit": "GB/s",
            "eps2": eps2_h,
            "measured_dist_sum_of_model_choice": float(dm[idx, zmod].sum()),
            "measured_dist_sum_of_measured_choice": float(dm[idx, zm].sum()),
            "bytes_model_choice": int(cm[idx, zmod].sum()),
            "bytes_measured_choice": int(cm[idx, zm].sum())}


ATTEND_SRC = os.path.join(ROOT, "partial_tucker_rotated_st_b300", "csrc", "attend.cu")
DECODE_SRC = os.path.join(ROOT, "partial_tucker_rotated_st_b300", "csrc", "decode_tc.cu")
GRAM_SRC = os.path.join(ROOT, "partial_tucker_rotated_st_b300", "csrc", "gram_tc.cu")
PROFILES = os.path.join(ROOT, "profiles")


def _sha(path):
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def profile_records(kind, src_path, workload, profiles_dir=PROFILES):
    """The `<kind>:` JSON lines of the committed ncu summaries under profiles/
    for this workload whose `src_sha256` still matches the kernel source
    (counters of another source or workload are not this kernel's)."""
    try:
        src = _sha(src_path)
        files = sorted(glob.glob(os.path.join(profiles_dir, "*.md")))
    except OSError:
        return []
    out = []
    for f in files:
        for line in open(f).read().splitlines():
            if not line.startswith(kind + ":"):
                continue
            rec = json.loads(line.split(":", 1)[1])
            if rec.get("src_sha256") == src and rec.get("workload") == workload:
                rec["source"] = os.path.relpath(f, os.path.dirname(profiles_dir))
                out.append(rec)
    return out


def traffic_record(kernel, src_path, bytes_key, w, profiles_dir=PROFILES):
    """DRAM bytes per launch of `kernel` on workload w from a committed ncu
    capture: the figure as recorded when the capture ran all w.n_units units,
    else scaled by the units processed (the kernels read each unit's data a
    fixed number of times, so traffic grows in proportion); None if no
    capture of the current source exists."""
    for rec in profile_records("traffic_record", src_path, w.name, profiles_dir):
        if rec.get("kernel") != kernel:
            continue
        units = int(rec.get("units", w.n_units))
        return int(round(int(rec[bytes_key]) * w.n_units / units))
    return None


def decode_traffic(w):
    """DRAM bytes of one decoder launch."""
    return traffic_record("decode_tc_kernel", DECODE_SRC, "dram_bytes_per_launch", w)


def attend_traffic(w):
    """DRAM bytes of one jolt_attend call (its three kernels)."""
    return traffic_record("attend", ATTEND_SRC, "dram_bytes_per_call", w)


def sweep_traffic(w):
    """DRAM bytes of one sweep-kernel launch."""
    return traffic_record("sweep_tc_kernel", SWEEP_SRC, "dram_bytes_per_launch", w)


def gram_tensor_record(w):
    """Tensor-pipe activity of the factor step's tcgen05 products (the feature
    and token Grams, the subspace-iteration product, the projection and the
    cores) from a committed ncu capture of the current sources, keyed by
    kernel; {} when none matches."""
    out = {}
    csrc = os.path.join(ROOT, "partial_tucker_rotated_st_b300", "csrc")
    for src in (GRAM_SRC, os.path.join(csrc, "proj_tc.cu"), os.path.join(csrc, "flash_tc.cu")):
        for rec in profile_records("tensor_record", src, w.name):
            out[rec["kernel"]] = {k: v for k, v in rec.items()
                                  if k not in ("kernel", "workload", "src_sha256")}
    return out


def roofline(w, kernel_s, hbm, kind, pk, sms=148):
    """Roofline of the fused sweep kernel.  Its dense products (the rotation
    of X and every rank checkpoint's reconstruction) run on the tensor cores;
    what bounds it is the FP32 scoring of every candidate, counted per element
    and rank pair as: the residual y (1 FMA), |y| max (1), y^2 for b = 0
    (1 FMA), and per b > 0 the scaled rounding (1 FMA + 1 add), the residual
    (1 FMA) and its square (1 FMA), FMA = 2 flops: 26 flops per pair per
    element.  `kernel_s` is the kernel's own average duration (CUDA events
    around its launch); `sms` the device's multiprocessor count.  The HBM
    fraction of the same launch (X read once, 2 bytes per element) is
    reported beside it, and so are the launch's algorithmic bytes: X, and the
    chains' operands each read once (the fp16 token coefficients Y16 and U_T16,
    the fp32 rotated factor rows W of every feature rank, Q U_d and the sign
    matrix), against which the measured DRAM traffic is compared."""
    U, N = w.n_units, w.elems_per_unit
    RT = max(r for r in w.rT if r != kvgen.FULL)
    RD = max(r for r in w.rd if r != kvgen.FULL)
    nd, nT, nb = len(w.rd), len(w.rT), len(w.bits)
    nbq = sum(1 for b in w.bits if b > 0)
    pairs = nT * nd
    flops_el = pairs * (2 + 1 + 2 * (nb - nbq) + 7 * nbq)
    tensor_el = 2 * w.D + 2 * 2 * (nd * RT + RD)   # rotation; chains with the hi/lo split
    flops = flops_el * N * U
    sm_max = pk.get("sm_max_mhz", 2032.0)
    peak = sms * 128 * 2 * sm_max * 1e6 / 1e12
    ach = flops / kernel_s / 1e12
    hbm_ach = 2.0 * N * U / kernel_s / 1e9
    has_full_t = kvgen.FULL in w.rT
    alg = U * (2 * N                                        # X
               + (2 * w.H * w.T * RD if has_full_t else 0)  # Y16 (the r_T = T chains)
               + 2 * nd * w.T * RT                          # U_T16 of every feature rank
               + 4 * nd * w.H * RT * w.D                    # W rows of every feature rank
               + 4 * RD * w.D + 2 * w.D * w.D)              # Q U_d, diag(sigma) H
    traffic = sweep_traffic(w)
    return {"kernel": "sweep_tc_kernel", "bound": "alu", "achieved": ach, "peak": peak,
            "unit": "TFLOP/s", "frac": ach / peak, "traffic": traffic,
            "bytes_algorithmic": int(alg),
            "traffic_over_algorithmic": None if traffic is None else traffic / alg,
            "kernel_ms": 1e3 * kernel_s,
            "peak_source": f"derived: FP32 pipe, {sms} SMs (device) x 128 lanes x 2 flop x "
                           f"max SM clock",
            "flops_per_element": flops_el, "tensor_flops_per_element": tensor_el,
            "bytes_per_element_algorithmic": 2,
            "hbm_achieved_gbs": hbm_ach, "hbm_frac": hbm_ach / hbm,
            "hbm_peak_gbs": hbm, "hbm_peak_kind": kind}


def parse_configs(s):
    if s in ("", "none"):
        return []
    out = [c.strip() for c in s.split(",") if c.strip()]
    for c in out:
        if c not in kvgen.WORKLOADS:
            raise SystemExit(f"unknown workload {c}")
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--workload", default=MAIN_WORKLOAD, choices=sorted(kvgen.WORKLOADS))
    ap.add_argument("--configs", default=",".join(EXTRA_CONFIGS),
                    help="comma-separated workloads with a record of their own, or 'none'")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--groups", type=int, default=0,
                    help="run only the first N layer groups of each workload (profiling runs)")
    args = ap.parse_args()
    args.configs = parse_configs(args.configs)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
