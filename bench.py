"""Benchmark of the Muon optimizer step on GB300 (one JSON line on stdout).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME]

A step is one muon_step over every parameter of the workload (momentum,
normalisation, 5 Newton-Schulz steps, weight-decay update).  The default
workload is the largest single-GPU one: the parameter matrices of 24 dense
transformer layers, 4 x [4096, 4096], [11008, 4096] and 2 x [4096, 11008]
bf16 per layer (168 slices in three groups, 4.86 G parameters).  Other
workloads (--workload): 74 separate bf16 [24, 10240] parameters grouped into
one [74, 24, 10240] batch (the small-parameter case of the HyperParallel FSDP
Muon RFC, section 3), 3-D stacks plus expert tensors, a synthetic MoE model.
Inputs are seeded synthetic tensors generated on the device.  L2 is flushed
(512 MB write) before every timed step; each step is timed with CUDA events
on the launching stream and ms_per_step is their mean, max over ranks.

--impl reference times the fp64 CPU oracle on the host cores on the same
workload (per step a bounded sample of every group, extrapolated to the
whole workload by the Newton-Schulz flop count where a whole slice does not
fit the step's time budget) and prints the same line with
"impl": "reference".  Under torchrun only rank 0 runs it.

With N > 1 (torchrun) each rank runs its own replica of the workload on its
own GPU: slices are independent, there is no data-path collective
("scaling": "weak"); a barrier brackets the timed region and the time is the
max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "muon_step_matrices_per_s"
UNIT = "matrices/s"
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, device) -> float:
    """Max of a per-rank time over all ranks (identity without a process
    group).  Works with NCCL on GPUs and with gloo on CPU tensors."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


SLOWDOWN_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clock_rejected(clocks: dict, device) -> bool:
    """True on any rank whose clock record shows a hardware or thermal
    slowdown, or (over at least three samples) a median SM clock below 70%
    of its maximum with no reason reported."""
    bad = any(r in clocks.get("reasons", ()) for r in SLOWDOWN_REASONS)
    mhz, top = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if mhz and top and mhz < 0.7 * top and not clocks.get("reasons") and \
            clocks.get("samples", 0) >= 3:
        bad = True
    return max_over_ranks(1.0 if bad else 0.0, device) > 0.0


def weak_scaling_value(slices_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank updates its own replica of the
    workload, so the job processes slices_per_rank * world matrices in the
    slowest rank's step time."""
    return slices_per_rank * world / (ms_max * 1e-3)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], tc=d["bf16_tflops"], tc_sustained=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sustained=1700.0, src="fallback")


def workload_work(w):
    """Algorithmic bytes (optimizer state touched once) and Newton-Schulz
    flops per step: the standard count T (4 m^2 n + 2 m^3) per slice and the
    symmetric-aware count T (3 m^2 n + m^3) (X X^T and b A + c A A are
    symmetric: half of each suffices), which the tensor roofline uses so the
    symmetric tiles the dense path skips do not inflate it."""
    es = 2 if w.dtype == torch.bfloat16 else 4
    per_el = es + 8 + 2 * es            # G read, M read+write, W read+write
    nbytes = 0
    flops = 0
    flops_sym = 0
    skinny_bytes = 0
    for s in w.shapes:
        E, M, N = (s if len(s) == 3 else (1,) + tuple(s))
        m, n = min(M, N), max(M, N)
        nbytes += E * M * N * per_el
        flops += E * w.ns_steps * (4 * m * m * n + 2 * m ** 3)
        flops_sym += E * w.ns_steps * (3 * m * m * n + m ** 3)
        if m <= 64:
            skinny_bytes += E * M * N * per_el
    return nbytes, flops, flops_sym, skinny_bytes, per_el


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.t0 = time.time()
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def wait_first(self, timeout=5.0):
        t = time.time()
        while self.p is not None and time.time() - t < timeout:
            self.f.flush()
            if os.path.getsize(self.f.name) > 0:
                return
            time.sleep(0.05)

    def stop(self):
        if self.p is not None:
            time.sleep(0.25)
            self.p.terminate()
            try:
                self.p.wait(2)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        for r in rows:
            for name, col in (("hw_slowdown", 5), ("hw_thermal_slowdown", 6),
                              ("sw_thermal_slowdown", 7), ("sw_power_cap", 8)):
                if r[col].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(rows[0][2]), "reasons": sorted(reasons), "samples": len(rows)}


def _code_text(path: str) -> str:
    import re
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_digest(path: str) -> str:
    """sha256 of a C/C++/CUDA source with its comments and blank space
    removed, so that an edit of comments alone keeps a profile valid while
    any change of code invalidates it."""
    return hashlib.sha256(_code_text(path).encode()).hexdigest()


def sources_digest(names) -> str:
    """source_digest over several sources of the library (csrc/ names)."""
    texts = [_code_text(os.path.join(ROOT, "newton_schulz_05_gb300", "csrc", n)) for n in names]
    return hashlib.sha256("\n".join(texts).encode()).hexdigest()


def profile_value(profile: str, sources, key: str):
    """A number from a committed ncu summary, valid only while the kernel
    sources it was captured from are unchanged (by their digest)."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    names = [sources] if isinstance(sources, str) else list(sources)
    kv = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source digest") != sources_digest(names) or key not in kv:
        return None
    return float(kv[key].split()[0])


def skinny_traffic(per_launch_units):
    """DRAM bytes of one fused-kernel launch of the 74 x [24, 10240] workload
    from the committed ncu summary, while skinny.cu is unchanged."""
    return profile_value("skinny_kernel_74x24x10240.txt", "skinny.cu", "dram bytes per launch")


# ---------------------------------------------------------------- oracle leg
def _ns_flops(m, n, T):
    return T * (4 * m * m * n + 2 * m ** 3)


class OracleSampler:
    """The fp64 oracle timed on a bounded sample of a workload, extrapolated
    to the whole workload.

    Per bucket of equal (M, N) one slice is drawn with the workload's seeded
    recipe.  When the oracle's whole step on that slice fits the bucket's
    share of the time budget, whole slices are timed (as many as the host
    threads run side by side); otherwise the oracle's whole step runs on the
    first r working rows of the slice (columns when M > N), r chosen to fit
    the budget, and its time is scaled to the full slice by the standard
    Newton-Schulz flop count T (4 m^2 n + 2 m^3), which dominates the step
    for such slices.  Bucket times are scaled by the bucket's slice count."""

    def __init__(self, w, threads: int):
        import oracle

        oracle.build()
        self.oracle = oracle
        self.w = w
        self.threads = threads
        self.buckets = {}
        for i, s in enumerate(w.shapes):
            E, M, N = (s if len(s) == 3 else (1,) + tuple(s))
            self.buckets.setdefault((M, N), [0, i])[0] += E
        self.total_slices = sum(c for c, _ in self.buckets.values())
        self.inputs = {}
        for (M, N), (_, pidx) in self.buckets.items():
            W = synth.draw((M, N), w.param_std, synth.param_seed(1, pidx), w.dtype)
            G = synth.draw((M, N), w.grad_std, synth.param_seed(0, pidx), w.dtype)
            self.inputs[(M, N)] = (W, G, torch.zeros((M, N), dtype=torch.float32))
        self.rate = None   # oracle flops/s, from the first sample

    def _run(self, W, G, Mo, k):
        """k copies of one slice: side by side on the host threads, or one
        slice with its products' rows spread over them."""
        w = self.w
        if k == 1:
            self.oracle.muon_slice(W, G, Mo, w.lr, w.beta, w.wd, w.nesterov, T=w.ns_steps,
                                   coeffs=w.coeffs, threads=self.threads)
            return
        self.oracle.muon_slices([W] * k, [G] * k, [Mo] * k, w.lr, w.beta, w.wd, w.nesterov,
                                T=w.ns_steps, coeffs=w.coeffs, threads=self.threads,
                                want_O=False)

    def sample(self, budget_s: float):
        """Time one sample of every bucket; returns (extrapolated seconds for
        one step of the whole workload, sample description)."""
        T = self.w.ns_steps
        share = budget_s / len(self.buckets)
        total, notes = 0.0, []
        for (M, N), (count, _) in self.buckets.items():
            W, G, Mo = self.inputs[(M, N)]
            m, n = min(M, N), max(M, N)
            full = max(_ns_flops(m, n, T), 1)
            if self.rate is None:
                # calibration: a small sub-block (or the whole slice if small)
                r = min(m, 64)
                t0 = time.perf_counter()
                self._sub(W, G, Mo, M, N, r)
                dt = time.perf_counter() - t0
                self.rate = max(_ns_flops(r, n, T), 1) / max(dt, 1e-6)
            if full / self.rate <= share:
                k = max(1, min(count, self.threads))
                t0 = time.perf_counter()
                self._run(W, G, Mo, k)
                dt = time.perf_counter() - t0
                total += dt / k * count
                notes.append("[%d,%d]: %d whole slice%s" % (M, N, k, "s" if k > 1 else ""))
                self.rate = k * full / max(dt, 1e-9)
            else:
                r = int((share * self.rate / (T * (4 * n + 2 * m) + 1e-9)) ** 0.5)
                r = max(8, min(m, r // 8 * 8))
                # solve 4 r^2 n + 2 r^3 ~ share * rate more exactly
                while r > 8 and _ns_flops(r, n, T) > share * self.rate:
                    r -= 8
                t0 = time.perf_counter()
                self._sub(W, G, Mo, M, N, r)
                dt = time.perf_counter() - t0
                sub = max(_ns_flops(r, n, T), 1)
                total += dt * full / sub * count
                notes.append("[%d,%d]: first %d of %d working rows, scaled by flops" % (M, N, r, m))
                self.rate = sub / max(dt, 1e-9)
        return total, "; ".join(notes)

    def _sub(self, W, G, Mo, M, N, r):
        if M <= N:
            self._run(W[:r].contiguous(), G[:r].contiguous(), Mo[:r].contiguous(), 1)
        else:
            self._run(W[:, :r].contiguous(), G[:, :r].contiguous(), Mo[:, :r].contiguous(), 1)


def oracle_rate(w, budget_s: float, threads: int):
    """The oracle's throughput on the workload (matrices/s), from about
    budget_s seconds of samples.  Returns (rate, sample text, seconds used)."""
    t_start = time.time()
    smp = OracleSampler(w, threads)
    smp.sample(min(2.0, budget_s / 4))        # warm-up and rate calibration
    t_step, notes = smp.sample(budget_s)
    rate = smp.total_slices / t_step
    extra = "" if "whole" in notes and "scaled" not in notes else "; extrapolated"
    return rate, notes + extra, time.time() - t_start


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    smp = OracleSampler(w, threads)
    # every step: one bounded sample of the workload, sized so that the whole
    # --steps K --warmup W run takes about 150 s of host time
    budget_per_step = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    smp.sample(min(2.0, budget_per_step))   # rate calibration
    times = []
    notes = ""
    for it in range(args.warmup + args.steps):
        t_step, notes = smp.sample(budget_per_step)
        if it >= args.warmup:
            times.append(t_step)
    t = sum(times) / len(times)
    rate = smp.total_slices / t
    extrapolated = "scaled" in notes or any(
        c > min(c, threads) for c, _ in smp.buckets.values())
    sample = "per step, fp64 oracle on %d threads: %s%s" % (
        threads, notes, "; extrapolated to all %d slices" % smp.total_slices if extrapolated else "")
    out = {"impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": w.name, "slices": smp.total_slices},
           "cpu_baseline": {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


# ---------------------------------------------------------------- our arm
def run_ours(args, w):
    import newton_schulz_05_gb300 as mu
    from newton_schulz_05_gb300 import build as mb

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        mb.build()
    if ws_n > 1:
        dist.barrier()
    mb.build()
    mu.load()

    shapes = list(w.shapes)
    # host-side planning (grouping by trailing dims), timed apart from the step
    plan_t = []
    for _ in range(5):
        t0 = time.perf_counter()
        plan = mu.Plan(list(zip(shapes, [w.dtype] * len(shapes))))
        plan_t.append((time.perf_counter() - t0) * 1e3)
    W = synth.make_params(w, device=dev)
    G = synth.make_grads(w, 0, device=dev)
    M = synth.make_momentum(w, device=dev)
    wsp = mu.alloc_workspace(plan, dev)
    stream = torch.cuda.current_stream(dev)
    hp = dict(lr=w.lr, beta=w.beta, wd=w.wd, nesterov=w.nesterov, ns_steps=w.ns_steps,
              coeffs=w.coeffs)
    step = mu.PreparedStep(plan, W, G, M, workspace=wsp, stream=stream, **hp)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    launches_per_step = plan.launches(w.ns_steps)
    n_slices = plan.num_slices

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    assert mu.workspace_error(wsp, stream) == 0

    def timed_region():
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        sampler = ClockSampler(local)
        sampler.wait_first()
        if ws_n > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.time()
        for k in range(args.steps):
            flush.zero_()
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.time() - t0
        if ws_n > 1:
            dist.barrier()
        return [a.elapsed_time(b) for a, b in ev], t1, sampler.stop()

    per, t_wall, clocks = timed_region()
    # a region that saw a thermal or hardware slowdown, or SM clocks far below
    # their maximum with no reason given (a clock lock left by someone
    # else), is timed once more; every rank takes the same decision
    if clock_rejected(clocks, dev):
        first = {k: clocks[k] for k in ("sm_mhz", "reasons")}
        per, t_wall, clocks = timed_region()
        clocks["remeasured_after"] = first
    ms = max_over_ranks(sum(per) / len(per), dev)
    err = mu.workspace_error(wsp, stream)

    # ---- the step with the write-back of its dirty L2 lines.  A read-only
    # sweep over a buffer larger than L2 evicts every line and writes back
    # the dirty ones without leaving new dirty lines.  Per iteration: flush
    # and sweep (L2 clean, none of the step's data cached), then the step,
    # then a sweep (which writes back what the step left dirty), then a
    # second sweep (nothing left to write back); the step with its
    # write-back is step + first sweep - second sweep.
    sweep_buf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    n_wb = max(1, min(args.steps, 20))
    marks = []
    for _ in range(n_wb):
        flush.zero_()
        sweep_buf.sum()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        step()
        e[1].record(stream)
        sweep_buf.sum()
        e[2].record(stream)
        sweep_buf.sum()
        e[3].record(stream)
        marks.append(e)
    torch.cuda.synchronize(dev)
    ms_wb = max_over_ranks(statistics.mean(
        e[0].elapsed_time(e[1]) + e[1].elapsed_time(e[2]) - e[2].elapsed_time(e[3])
        for e in marks), dev)
    del sweep_buf

    # ---- per-kernel device time: the same step through muon_step_timed, a
    # CUDA event on the launching stream before every launch (a second timed
    # region right after the first, L2 flushed before each step)
    n_timed = max(1, min(args.steps, 5))
    acc = {k: [0.0, 0] for k in mu.KERNEL_CLASSES}
    for _ in range(n_timed):
        flush.zero_()
        for k, (kms, kn) in step.timed().items():
            acc[k][0] += kms
            acc[k][1] += kn
    kernels = {k: {"ms_per_step": v[0] / n_timed, "launches_per_step": v[1] / n_timed}
               for k, v in acc.items() if v[1]}

    # ---- end to end through the public API with HOST buffers: the optimizer
    # state (parameters, gradients, momenta) in page-locked host memory, one
    # muon_step_host call per step, which copies each unit of slices in,
    # steps it and copies its parameters and momenta back, copies
    # overlapping the kernels.  Each kind of state lives in one flat host
    # buffer from muon_host_alloc (page-locked, on transparent huge pages),
    # the parameters being views into it (the layout of a flat-parameter
    # data-parallel trainer).
    def flat(ts):
        buf = mu.alloc_host(sum(x.numel() for x in ts), ts[0].dtype)
        views, off = [], 0
        for x in ts:
            views.append(buf[off:off + x.numel()].view(x.shape))
            off += x.numel()
        return buf, views

    hW, Wh = flat(W)
    hG, Gh = flat(G)
    hM, Mh = flat(M)
    for d, h in zip(W + G + M, Wh + Gh + Mh):
        h.copy_(d)
    h2d = sum(x.numel() * x.element_size() for x in (hW, hG, hM))
    d2h = sum(x.numel() * x.element_size() for x in (hW, hM))
    # args.host_bufs staging buffers of args.host_unit_gb each (at least one
    # slice, at most an eighth of the state)
    part = max(plan.host_unit_bytes, min(int(args.host_unit_gb * (1 << 30)), h2d // 8))
    staging = torch.empty(args.host_bufs * part, dtype=torch.uint8, device=dev)
    del W, G, M, step   # the device copies are not needed any more
    host_step = mu.PreparedHostStep(plan, Wh, Gh, Mh, workspace=wsp, staging=staging,
                                    unit_bytes=part, stream=stream, **hp)

    for _ in range(min(args.warmup, 3)):
        host_step()
    torch.cuda.synchronize(dev)
    # the plain copy bandwidth of this host memory right now, for reference:
    # each buffer read once into the staging (in pieces of its size), and the
    # gradients' first piece copied back out over itself
    def h2d_gbs(h):
        src = h.view(torch.uint8).view(-1)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for o in range(0, src.numel(), staging.numel()):
            k = min(staging.numel(), src.numel() - o)
            staging[:k].copy_(src[o:o + k], non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize(dev)
        return src.numel() / 1e9 / (c0.elapsed_time(c1) * 1e-3)
    copy_gbs = {"h2d_params": h2d_gbs(hW), "h2d_grads": h2d_gbs(hG), "h2d_momenta": h2d_gbs(hM)}
    g8 = hG.view(torch.uint8).view(-1)
    k = min(staging.numel(), g8.numel())
    staging[:k].copy_(g8[:k])
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    g8[:k].copy_(staging[:k], non_blocking=True)
    c1.record(stream)
    torch.cuda.synchronize(dev)
    copy_gbs["d2h"] = k / 1e9 / (c0.elapsed_time(c1) * 1e-3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_steps = max(1, min(args.steps, 50))
    e0.record(stream)
    for _ in range(e_steps):
        host_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / e_steps, dev)
    assert mu.workspace_error(wsp, stream) == 0

    nbytes, flops, flops_sym, skinny_bytes, per_el = workload_work(w)
    pk = peaks()
    kinds = {g["kernel"] for g in plan.groups()}
    if kinds == {mu.KERNEL_SKINNY} and launches_per_step == 1:
        # one fused launch per step: its duration is the step's event time
        achieved = nbytes / (ms * 1e-3) / 1e9
        traffic = skinny_traffic(n_slices)
        roof = {"bound": "hbm", "kernel": "skinny_kernel", "achieved": achieved,
                "peak": pk["hbm"], "unit": "GB/s", "frac": achieved / pk["hbm"],
                "traffic": traffic,
                "frac_with_writeback": nbytes / (ms_wb * 1e-3) / 1e9 / pk["hbm"],
                "note": "algorithmic bytes %d B/element x %d elements per launch; peak %s" % (
                    per_el, w.num_elements, "of measured" if pk["src"] == "measured" else "of fallback")}
    else:
        # the dominant kernel is the tcgen05 GEMM of the dense groups: its
        # algorithmic flops (symmetric-aware, T(3m^2n+m^3) per dense slice)
        # over its device time per step from the per-launch events.  A timed
        # region of a second or more runs under the power cap: the sustained
        # peak applies, the burst peak to shorter ones
        sustained = ms * args.steps >= 1000.0
        peak = pk["tc_sustained"] if sustained else pk["tc"]
        dense_sym = dense_std = 0
        for g in plan.groups():
            if g["kernel"] == mu.KERNEL_DENSE:
                m_, n_ = g["m"], g["n"]
                dense_sym += g["count"] * w.ns_steps * (3 * m_ * m_ * n_ + m_ ** 3)
                dense_std += g["count"] * w.ns_steps * (4 * m_ * m_ * n_ + 2 * m_ ** 3)
        g_ms = kernels.get("gemm", {}).get("ms_per_step", 0.0)
        g_n = kernels.get("gemm", {}).get("launches_per_step", 0)
        achieved = dense_sym / (g_ms * 1e-3) / 1e12 if g_ms > 0 else 0.0
        step_achieved = flops_sym / (ms * 1e-3) / 1e12
        traffic = None
        if w.name == "dense_24L":
            traffic = profile_value("tc_gemm_traffic_dense.txt", ["tc_gemm.cu", "dense.cu"],
                                    "dram bytes per launch (dense_24L, scaled)")
        roof = {"bound": "tensor", "kernel": "tc_gemm (Newton-Schulz products)",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic,
                "launch_ms": g_ms / g_n if g_n else None,
                "flops_per_launch": dense_sym / g_n if g_n else None,
                "achieved_standard_count": dense_std / (g_ms * 1e-3) / 1e12 if g_ms > 0 else 0.0,
                "step_achieved": step_achieved, "step_frac": step_achieved / peak,
                "note": "symmetric-aware NS flops T(3m^2n+m^3) of the dense slices per step over "
                        "the GEMM's device time per step (CUDA events around each launch on its "
                        "stream); standard count T(4m^2n+2m^3) in achieved_standard_count; "
                        "step_achieved: all NS flops over the whole step time; peak bf16 %s %s" % (
                    "sustained" if sustained else "burst",
                    "of measured" if pk["src"] == "measured" else "of fallback")}

    # operand types of the tensor-core products: the fused skinny kernel takes
    # bf16 V and bf16 Q (fp32 m x m recursion), the dense path fp16 iterates
    if kinds == {mu.KERNEL_SKINNY}:
        arith, mode = "bf16", "bf16 tensor-core operands, fp32 accumulate, fp32 m x m recursion"
    elif mu.KERNEL_SKINNY in kinds:
        arith, mode = "f16", ("fp16 tensor-core operands (dense groups), bf16 (skinny groups), "
                              "fp32 accumulate")
    else:
        arith, mode = "f16", "fp16 tensor-core operands, fp32 accumulate"
    out = {"metric": METRIC, "value": weak_scaling_value(n_slices, ws_n, ms), "unit": UNIT,
           "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "ms_per_step_median": statistics.median(per), "ms_per_step_min": min(per),
           "ms_per_step_with_writeback": ms_wb,
           "plan_ms": statistics.median(plan_t),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": arith, "data": "synthetic",
           "config": {"workload": w.name, "slices": n_slices, "param_dtype": str(w.dtype),
                      "ns_steps": w.ns_steps, "l2": "flushed (512 MB write) before each timed step",
                      "parallelism": "replica per GPU" if ws_n > 1 else "single GPU",
                      "mode": mode},
           "roofline": roof, "kernels": kernels,
           "e2e": {"value": weak_scaling_value(n_slices, ws_n, ms_e2e), "unit": UNIT,
                   "ms_per_step": ms_e2e, "unit_bytes": part, "buffers": args.host_bufs,
                   "plain_copy_GBps": copy_gbs,
                   "call": "muon_step_host: parameters, gradients and momenta in page-locked "
                           "host memory from muon_host_alloc (transparent huge pages); per "
                           "step every unit of slices is copied in, stepped "
                           "and its parameters and momenta copied back, the copies of one unit "
                           "overlapping the kernels of its neighbours",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
           "clocks": clocks, "gpu_launches": launches_per_step * args.steps,
           "wall_s_timed": t_wall, "device_error": err}
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        rate, sample, used = oracle_rate(w, budget_s=15.0, threads=os.cpu_count() or 1)
        out["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": os.cpu_count() or 1,
                               "kind": "oracle", "sample": sample + " (%.1f s)" % used}
    if rank == 0:
        print(json.dumps(out))
    if ws_n > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dense_24L", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--host-unit-gb", type=float, default=2.0,
                    help="end-to-end leg: staging bytes of one unit of slices (GiB)")
    ap.add_argument("--host-bufs", type=int, default=4,
                    help="end-to-end leg: staging buffers in rotation")
    ap.add_argument("--ns-steps", type=int, default=None,
                    help="Newton-Schulz steps T (default: the workload's, 5); T = 0 times "
                         "the step without the iteration, for its share of the step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = synth.workload(args.workload)
    if args.ns_steps is not None:
        w = dataclasses.replace(w, ns_steps=args.ns_steps)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
