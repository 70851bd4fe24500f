"""Benchmark of the verify + realign hot path (one step = one speculative round).

    python bench.py [--gpus N] [--steps K] [--warmup W]
                    [--workload glm4_9b|vicuna7b|qwen3_8b|tiny|exspec_pool|exspec_serving|exspec_sweep|
                                read_floor]
                    [--impl specdec|reference] [--ping-pong] [--no-all-configs]

A step is one round: verification of the round's D drafts per row against the target's scores
(greedy, or speculative rejection sampling for the GLM-4-9B-shaped workload), then realignment
of the left-padded batch (every layer's surviving K/V columns move to their new place in the one
cache buffer -- rows that do not shift stay -- or, with --ping-pong, to the other of two buffers;
ids/mask/position IDs are rebuilt).  Inputs are synthetic, seeded and resident on the device
before the timed region; every round streams gigabytes of K/V, far more than L2.  The default
workload is the GLM-4-9B-shaped sampled round (the largest); the line's ``all_configs`` block
then times every other workload the same way (tiny, Vicuna-7B- and Qwen3-8B-shaped rounds, the
EXSPEC pool, the batch-size sweep B = 1..64), each with its own steps and ms_per_step.
With --gpus N (under torchrun) every rank runs an independent replica of the workload (the path
has no exchange step); ``value`` is the rounds of all ranks over the slowest rank's time.

--impl reference times the CPU oracle (plain numpy, float64) on this host: W untimed and K timed
whole rounds of the same workload, one round per step; it is the deliberately slow baseline, not
a target.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify+realign rounds/s"


L2_BYTES = 129e6  # GB300 L2


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=40)
    p.add_argument("--warmup", type=int, default=4)
    p.add_argument("--workload", default="glm4_9b")
    p.add_argument("--impl", default="specdec", choices=["specdec", "reference"])
    p.add_argument("--copy-engine", type=int, default=0)
    p.add_argument("--top-k", type=int, default=0,
                   help="sampled workloads: top-k sampling setting (0: off)")
    p.add_argument("--top-p", type=float, default=1.0,
                   help="sampled workloads: top-p sampling setting (1: off)")
    p.add_argument("--launch", default="graph+pdl", choices=["stream", "pdl", "graph", "graph+pdl"],
                   help="how the timed rounds are launched: plain stream launches; each "
                        "realignment as a programmatic dependent of its verification (pdl); the "
                        "timed rounds captured once into a CUDA graph and replayed (graph)")
    p.add_argument("--philox", action="store_true",
                   help="sampled workloads: draw the uniforms in-kernel (Philox) instead of "
                        "reading them from HBM")
    p.add_argument("--window", type=int, default=0,
                   help="exspec_serving: length window of a batch (0: exact length)")
    p.add_argument("--ping-pong", action="store_true",
                   help="two K/V caches, realigned from one into the other (default: one cache "
                        "realigned in place)")
    p.add_argument("--realign-schedule", default="counter", choices=["counter", "fixed"],
                   help="realignment work distribution: CTAs take work items from a counter "
                        "(default), or every CTA moves one fixed share")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-depth", type=int, default=0,
                   help="e2e: device staging sets for the host-fed rounds' inputs (0: as many as "
                        "fit 1 GiB, from 2 to 8)")
    p.add_argument("--layers", type=int, default=0,
                   help="override the workload's layer count (smaller cache, e.g. for ncu)")
    p.add_argument("--no-all-configs", action="store_true",
                   help="time the selected workload only (no all_configs block)")
    p.add_argument("--no-cpu-baseline", action="store_true",
                   help="skip timing the oracle (cpu_baseline: null), e.g. under a profiler")
    return p.parse_args()


# ------------------------------------------------------------------------------ distributed

def dist_setup(gpus):
    import torch
    import torch.distributed as dist
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, ws, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    """Largest value of ``x`` over all ranks (the slowest rank's time)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------ clocks

class NvmlClocks:
    """Read-only NVML queries through ctypes (SM clock, its maximum, clock-event reasons) for the
    device with the given UUID; ``ok`` is False when NVML cannot be used."""
    # clock-event reason bits of NVML's nvmlClocksEventReasons
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}

    def __init__(self, uuid):
        import ctypes
        self.ok = False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if uuid is None or self.lib.nvmlDeviceGetHandleByUUID(
                    uuid.encode(), ctypes.byref(self.handle)) != 0:
                return
            self.u = ctypes.c_uint()
            self.ull = ctypes.c_ulonglong()
            self.ctypes = ctypes
            self.ok = self.max_sm() is not None
        except (OSError, AttributeError):
            self.ok = False

    def sm(self):
        return (self.u.value if self.lib.nvmlDeviceGetClockInfo(
            self.handle, 1, self.ctypes.byref(self.u)) == 0 else None)  # 1: NVML_CLOCK_SM

    def max_sm(self):
        return (self.u.value if self.lib.nvmlDeviceGetMaxClockInfo(
            self.handle, 1, self.ctypes.byref(self.u)) == 0 else None)

    def reasons(self):
        f = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        if f(self.handle, self.ctypes.byref(self.ull)) != 0:
            return set()
        return {name for name, bit in self.BITS.items() if self.ull.value & bit}


def bind_local_cpus(index):
    """Restrict this process's threads to the CPU cores NVML reports as local to the GPU, so that
    pinned host buffers (allocated and touched by these threads) land on the GPU's NUMA node.
    Returns (cores now allowed, whether the set was narrowed); a no-op where NVML cannot say."""
    import ctypes
    import torch
    allowed = os.sched_getaffinity(0)
    if not torch.cuda.is_available():
        return len(allowed), False
    try:
        uuid = str(torch.cuda.get_device_properties(index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        nv = NvmlClocks(uuid)
        if not nv.ok:
            return len(allowed), False
        words = (ctypes.c_ulong * 64)()
        if nv.lib.nvmlDeviceGetCpuAffinity(nv.handle, 64, words) != 0:
            return len(allowed), False
    except (AttributeError, RuntimeError, OSError):
        return len(allowed), False
    bits = ctypes.sizeof(ctypes.c_ulong) * 8
    local = {w * bits + b for w in range(64) for b in range(bits) if (words[w] >> b) & 1}
    keep = local & allowed
    if not keep or keep == allowed:
        return len(allowed), False
    os.sched_setaffinity(0, keep)
    return len(keep), True


class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed region runs: an NVML thread polling
    back to back (timed regions can be a few ms long), else nvidia-smi every 10 ms (started
    before the region, which begins once its first sample is in)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.nv_samples = []
        self.nv_max = None
        self.nv = None

    def _poll(self):  # back to back: each NVML query already takes on the order of 1 ms
        while not self.stop.is_set():
            mhz = self.nv.sm()
            if mhz is not None:
                self.nv_samples.append((mhz, self.nv.reasons()))

    def __enter__(self):
        import threading
        import torch
        try:
            uuid = str(torch.cuda.get_device_properties(self.index).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except (AttributeError, RuntimeError):
            uuid = None
        self.nv = NvmlClocks(uuid)
        if self.nv.ok:
            self.nv_max = self.nv.max_sm()
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self.proc.stdout.readline()  # the region starts once sampling runs
            if first.strip():
                self.lines.append(first)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.nv is not None and self.nv.ok:
            self.stop.set()
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines += [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if self.nv_samples:
            sm = [m for m, _ in self.nv_samples]
            reasons = set().union(*(r for _, r in self.nv_samples))
            return {"sm_mhz": statistics.median(sm), "sm_max_mhz": self.nv_max,
                    "reasons": sorted(reasons), "samples": len(sm), "source": "nvml"}
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


def captured_traffic(kernel: str, algorithmic_bytes: float):
    """DRAM traffic per launch from the committed ncu capture of ``kernel``, scaled to this
    launch's algorithmic bytes; None when the kernel source changed since the capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f)[kernel]
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != rec["source_sha256"]:
                return None
        ratio = (rec["dram_read_bytes"] + rec["dram_write_bytes"]) / rec["algorithmic_bytes"]
        return round(ratio * algorithmic_bytes)
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ------------------------------------------------------------------------------ GPU arm

def workload(args):
    import dataclasses
    from speculative_decoding_specdec_gb300 import synth
    w = synth.WORKLOADS["exspec_pool" if args.workload in ("exspec_sweep", "exspec_serving",
                                                           "read_floor")
                        else args.workload]
    return dataclasses.replace(w, layers=args.layers) if args.layers else w


def accept_histogram(n_hist, first, last, D):
    """Accept lengths of rounds [first, last) from the per-round committed lengths (row r holds
    N_b at the start of round r, so a_b = N'_b - N_b - 1): the count of each a in 0..D over all
    rows and rounds -- a < D is also the position of the first rejected draft -- and their mean."""
    import numpy as np
    n = np.asarray(n_hist, dtype=np.int64)
    a = (n[first + 1:last + 1] - n[first:last] - 1).reshape(-1)
    if a.size and (a.min() < 0 or a.max() > D):
        raise RuntimeError("accept length outside [0, D]")
    hist = np.bincount(a, minlength=D + 1)[:D + 1]
    return {"accept_len_hist": [int(x) for x in hist],
            "mean_accept_len": float(a.mean()) if a.size else 0.0}


def run_specdec(args, rank, ws, local):
    import numpy as np
    import torch
    from speculative_decoding_specdec_gb300 import synth
    from speculative_decoding_specdec_gb300.engine import EqspecBatch

    w = workload(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    K, Wm = args.steps, args.warmup
    R = K + Wm
    gen_cpu = synth.make_gen(w.seed * 1000 + rank)
    n0 = w.prompt_lengths(gen_cpu)
    prompts = [torch.randint(0, w.V, (int(n),), generator=gen_cpu).tolist() for n in n0]
    cap = w.capacity(int(n0.max()), rounds=R)
    eng = EqspecBatch(w.layers, w.heads, w.head_dim, w.kv_dtype, w.B, w.D, cap, R, device=dev,
                      in_place=not args.ping_pong, scheduled=args.realign_schedule == "counter")
    g = torch.Generator(device=dev).manual_seed(w.seed * 7919 + rank)
    for k in eng.kv:
        k.normal_(generator=g)
    # all rounds' inputs, generated before any timed region
    logits, drafts, draft_logits, uniforms = [], [], [], []
    for _ in range(R):
        if w.mode == "greedy":
            lg, d = synth.greedy_round(g, w.B, w.D, w.V, w.alpha, dtype=w.logit_dtype, device=dev)
        else:
            lg, dl, d, u = synth.sampled_round(g, w.B, w.D, w.V, w.temperature,
                                               dtype=w.logit_dtype, device=dev,
                                               draft_candidates=args.top_k)
            draft_logits.append(dl)
            uniforms.append(u)
        logits.append(lg)
        drafts.append(d)
    stream = torch.cuda.current_stream()

    def verify(r, lg=None, d=None):
        lg = logits[r] if lg is None else lg
        d = drafts[r] if d is None else d
        if w.mode == "greedy":
            eng.verify_greedy(lg, d)
        elif args.philox:
            eng.verify_sample(lg, draft_logits[r], d, None, w.temperature,
                              top_k=args.top_k, top_p=args.top_p, seed=w.seed)
        else:
            eng.verify_sample(lg, draft_logits[r], d, uniforms[r], w.temperature,
                              top_k=args.top_k, top_p=args.top_p)

    # ---------------- device-resident timing
    # With --pdl each realignment is launched as a programmatic dependent of the verification
    # ahead of it; with --graph the K timed rounds are captured once into a CUDA graph and the
    # timed region is one replay.  Either way the timed rounds carry no events between their
    # kernels (an event would serialise them), and a second pass over the same rounds, with
    # events, gives the per-kernel times.
    use_pdl = "pdl" in args.launch
    eng.pdl = use_pdl
    fused = args.launch != "stream"
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]

    def warm():
        eng.start(prompts)
        for r in range(Wm):
            verify(r)
            eng.realign(drafts[r], copy_engine=args.copy_engine)
        torch.cuda.synchronize()

    def rounds(inner):
        for i in range(K):
            r = Wm + i
            if inner:
                # a short device sleep ahead of the first event, so that on an idle GPU the
                # events time the kernels, not the host's launch of them
                torch.cuda._sleep(100_000)
                ev[i][0].record(stream)
            verify(r)
            if inner:
                ev[i][1].record(stream)
            eng.realign(drafts[r], copy_engine=args.copy_engine)
            if inner:
                ev[i][2].record(stream)

    warm()
    graph = None
    launch_used = args.launch
    if args.launch.startswith("graph"):
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                rounds(False)
            torch.cuda.synchronize()
        except Exception as exc:  # capture refused: time the same rounds as stream launches
            print(f"graph capture failed ({exc}); timing stream launches", file=sys.stderr)
            graph = None
            launch_used = "pdl" if use_pdl else "stream"
            warm()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            rounds(not fused)
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    ms = t0.elapsed_time(t1)
    status = int(eng.status.item())
    if status:
        raise RuntimeError(f"device status {status} during the timed rounds")
    if fused:  # the per-kernel breakdown, from a pass with events
        eng.pdl = False
        warm()
        rounds(True)
        torch.cuda.synchronize()
        eng.pdl = use_pdl
    t_verify = sum(e[0].elapsed_time(e[1]) for e in ev) / K
    t_realign = sum(e[1].elapsed_time(e[2]) for e in ev) / K
    n_hist = eng.n_hist.cpu().numpy().astype(np.int64)
    acc = [(n_hist[r + 1] - n_hist[r] - 1) for r in range(Wm, R)]
    w_hist = eng.w_hist[:, 0].cpu().numpy().astype(np.int64)
    moved_cols = 0  # N'_b - 1 per row; in place, rows whose columns do not shift move nothing
    for r in range(Wm, R):
        cols = n_hist[r + 1] - 1
        if not args.ping_pong:
            shift = (w_hist[r + 1] - n_hist[r + 1]) - (w_hist[r] - n_hist[r])
            cols = cols[shift != 0]
        moved_cols += int(cols.sum())
    realign_bytes = 2.0 * moved_cols * w.token_bytes / K
    es = torch.tensor([], dtype=w.logit_dtype).element_size()
    filtered = w.mode == "sampled" and (args.top_k or args.top_p < 1.0)  # + the filter kernel
    verify_bytes = (w.B * (w.D + 1) * w.V * es + (w.B * w.D * w.V * es if w.mode == "sampled" else 0)
                    + w.B * w.D * 4 + w.B * 8)
    committed = float(sum(int(a.sum()) + len(a) for a in acc)) / K

    # ---------------- end to end through the public API with host buffers
    # HostRounds copies each round's inputs from pinned host memory on a copy stream, overlapping
    # the round before, and reads each round's results back into pinned host memory.
    e2e = None
    if not args.no_e2e:
        from speculative_decoding_specdec_gb300.engine import HostRounds
        host = []
        for r in range(R):
            h = {"logits": logits[r], "draft": drafts[r]}
            if w.mode == "sampled":
                h["draft_logits"] = draft_logits[r]
                if not args.philox:
                    h["uniforms"] = uniforms[r]
            host.append({k: v.cpu().pin_memory() for k, v in h.items()})
        # Every pinned input buffer is read by the device once before the timed region, into a
        # scratch buffer the rounds never read: on these hosts the first device read of freshly
        # pinned pages can take ~10x longer than every later read of them (a one-time mapping
        # cost that a serving process pays once for the staging buffers it reuses).  The timed
        # rounds still copy all their inputs from host memory; the first reads are reported.
        scratch = {k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in host[0].items()}
        first_read = []
        for h in host:
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for name, t in h.items():
                scratch[name].copy_(t, non_blocking=True)
            f1.record(stream)
            torch.cuda.synchronize()
            first_read.append(f0.elapsed_time(f1))
        del scratch
        round_bytes = sum(v.numel() * v.element_size() for v in host[0].values())
        depth = args.e2e_depth or max(2, min(8, (1 << 30) // max(1, round_bytes)))
        feed = HostRounds(eng, host[0], stream, timed=True, depth=depth)
        out = torch.empty((R, 3 * w.B + 1), dtype=torch.int32).pin_memory()
        # the host link's rate for one round's inputs alone, copied again and again from the
        # same pinned buffers
        link = []
        for rep in range(5):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for name, t in host[0].items():
                feed.slots[0][name].copy_(t, non_blocking=True)
            c1.record(stream)
            torch.cuda.synchronize()
            if rep:
                link.append(c0.elapsed_time(c1))
        h2d_gbs = feed.h2d_bytes / (statistics.median(link) / 1e3) / 1e9

        def step(d):
            if w.mode == "greedy":
                eng.verify_greedy(d["logits"], d["draft"])
            elif args.philox:
                eng.verify_sample(d["logits"], d["draft_logits"], d["draft"], None, w.temperature,
                                  top_k=args.top_k, top_p=args.top_p, seed=w.seed)
            else:
                eng.verify_sample(d["logits"], d["draft_logits"], d["draft"], d["uniforms"],
                                  w.temperature, top_k=args.top_k, top_p=args.top_p)

        eng.start(prompts)
        feed.run(host[:Wm], step, out)
        torch.cuda.synchronize()
        barrier(ws)
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        feed.run(host[Wm:], step, out)
        s1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ms = max_over_ranks(s0.elapsed_time(s1), ws)
        copy_ms = feed.copy_ms()[-K:]  # the timed rounds' input copies
        if int(eng.status.item()):
            raise RuntimeError("device status set during the end-to-end rounds")
        n_e2e = out[:K, 2 * w.B:3 * w.B].numpy().astype(np.int64)
        if not (n_e2e == n_hist[Wm + 1:R + 1]).all():
            raise RuntimeError("end-to-end rounds committed other lengths than the device rounds")
        e2e = {"value": K * ws / (e2e_ms / 1e3), "unit": "rounds/s",
               "h2d_bytes_per_step": feed.h2d_bytes, "d2h_bytes_per_step": feed.d2h_bytes,
               "copies": "H2D on a copy stream up to staging_depth - 1 rounds ahead of the "
                         "compute stream; D2H after each round",
               "staging_depth": depth,
               "first_read_ms": {"median": round(statistics.median(first_read), 3),
                                 "max": round(max(first_read), 3),
                                 "note": "each round's pinned buffers read once by the device "
                                         "before the timed region (a one-time cost of fresh "
                                         "pinned pages on these hosts); not in the timed "
                                         "region"},
               "h2d_gbs_repeated": round(h2d_gbs, 1),
               "h2d_ms_per_round": {"median": round(statistics.median(copy_ms), 3),
                                    "max": round(max(copy_ms), 3)},
               "copy_bound_rounds_per_s": round(h2d_gbs * 1e9 / feed.h2d_bytes, 1)}

    ms_max = max_over_ranks(ms, ws)
    rounds_all = sum_over_ranks(float(K), ws)
    peak, peak_kind = measured_peaks()
    achieved = realign_bytes / (t_realign / 1e3) / 1e9
    verify_gbs = verify_bytes / (t_verify / 1e3) / 1e9
    sfu = None
    if w.mode == "sampled" and not filtered:
        # the second roof of sampled verification: one exp2 per score of the 2D+1 rows, then two
        # per vocabulary entry of the residual row pair (one for a bonus row), against the MUFU's
        # nominal 16 exp2 per clock per SM at the SM clock sampled during the timed region
        acc_hist = accept_histogram(n_hist, Wm, R, w.D)["accept_len_hist"]
        rows_resid = sum(acc_hist[:w.D]) / K
        rows_bonus = acc_hist[w.D] / K
        exps = w.B * (2 * w.D + 1) * w.V + (2 * rows_resid + rows_bonus) * w.V
        props = torch.cuda.get_device_properties(dev)
        sm_mhz = clk.summary().get("sm_mhz") or 2070
        mufu = 16 * props.multi_processor_count * sm_mhz * 1e6
        sfu = {"exps_per_launch": round(exps), "exps_per_s": round(exps / (t_verify / 1e3)),
               "peak_exps_per_s": round(mufu), "frac": round(exps / (t_verify / 1e3) / mufu, 4),
               "peak_source": "16 exp2/clock/SM (nominal) x SMs x sampled SM clock"}
    return {
        "value": rounds_all / (ms_max / 1e3),
        "ms_per_step": ms_max / K,
        "launch": launch_used,
        "clocks": clk.summary(),
        "e2e": e2e,
        "roofline": {"bound": "hbm", "kernel": "realign", "achieved": round(achieved, 1),
                     "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": captured_traffic("realign_kernel", realign_bytes),
                     "bytes_per_launch": realign_bytes, "ms_per_launch": t_realign},
        "verify": {"kernel": "greedy_kernel" if w.mode == "greedy" else
                   ("filter_kernel + sample_kernel" if filtered else "sample_kernel"),
                   "ms_per_launch": t_verify, "bytes_per_launch": verify_bytes,
                   "achieved_gbs": round(verify_gbs, 1), "frac": round(verify_gbs / peak, 4),
                   "traffic": None if filtered else
                   captured_traffic("greedy_kernel" if w.mode == "greedy" else "sample_kernel",
                                    verify_bytes),
                   **({"sfu": sfu} if sfu else {})},
        "committed_slots_per_s": committed / (ms_max / K / 1e3),
        "committed_per_round": committed,
        "acceptance": accept_histogram(n_hist, Wm, R, w.D),
        "cap_cols": cap,
        "bytes_per_round": realign_bytes + verify_bytes,
    }


# ------------------------------------------------------------------------------ EXSPEC pool

def run_pool(args, rank, ws):
    """EXSPEC SequencePool rounds: grouping by length, one greedy verification over the pool,
    then per batch an in-place commit (uniform batch) or gather + append (mixed leftovers).  The
    verification pass that would write the new K/V columns between gather and append belongs to
    the model and is not run; the copies move the same bytes either way."""
    import numpy as np
    import torch
    from speculative_decoding_specdec_gb300 import synth
    from speculative_decoding_specdec_gb300.engine import ExspecPool

    w = workload(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    K, Wm = args.steps, args.warmup
    R = K + Wm
    gen = synth.make_gen(w.seed * 1000 + rank)
    n0 = w.prompt_lengths(gen)
    alpha = torch.rand(w.B, generator=gen) * 0.4 + 0.5          # per-sequence acceptance U[0.5, 0.9]
    prompts = [torch.randint(0, w.V, (int(n),), generator=gen).tolist() for n in n0]
    need = (int(n0.sum()) + w.B * (R * (w.D + 1) + w.D + 1)) * w.token_bytes
    free, _ = torch.cuda.mem_get_info()
    if need > 0.85 * free:
        raise SystemExit(f"pool arena needs {need / 1e9:.0f} GB, {free / 1e9:.0f} GB free: "
                         f"fewer rounds (--steps/--warmup)")
    pool = ExspecPool(w.layers, w.heads, w.head_dim, w.kv_dtype, prompts, w.D, R, device=dev,
                      scheduled=args.realign_schedule == "counter")
    g = torch.Generator(device=dev).manual_seed(w.seed)
    logits, drafts = [], []
    for _ in range(R):
        lg, d = synth.greedy_round(g, w.B, w.D, w.V, alpha.to(dev), dtype=w.logit_dtype, device=dev)
        logits.append(lg)
        drafts.append(d)
    stream = torch.cuda.current_stream()
    moved, uniform_frac, mixed_rows, kern = [], [], [], []

    def one_round(r, timed):
        n_before = pool.slot_len.cpu().numpy() if timed else None
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)] if timed else None
        batches = pool.schedule()
        if timed:
            # the schedule's readback left the device idle: queue the verification behind a
            # ~0.1 ms device sleep so that its events time the kernel, not the host's launch
            torch.cuda._sleep(200_000)
            ev[0].record(stream)
        pool.verify_greedy(logits[r], drafts[r])
        if timed:
            ev[1].record(stream)
        for off, k, uni in batches:
            pool.gather(off, k, uni)
            pool.append(off, k, uni, drafts[r])
        if timed:
            ev[2].record(stream)
            kern.append(ev)
            perm = pool.perm.cpu().numpy()
            n_after = pool.slot_len.cpu().numpy()
            cols = 0
            for off, k, uni in batches:
                if not uni:
                    rows = perm[off:off + k]
                    cols += int((n_before[rows] - 1).sum() + (n_after[rows] - n_before[rows]).sum())
            moved.append(2 * cols * w.token_bytes)
            nu = sum(k for _, k, uni in batches if uni)
            uniform_frac.append(nu / w.B)
            mixed_rows.append(w.B - nu)

    for r in range(Wm):
        one_round(r, False)
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    for i in range(K):
        one_round(Wm + i, True)
    torch.cuda.synchronize()
    wall = max_over_ranks(time.perf_counter() - t0, ws)
    if int(pool.status.item()):
        raise RuntimeError(f"device status {int(pool.status.item())}")
    verify_ms = [e[0].elapsed_time(e[1]) for e in kern]
    kern_ms = [e[1].elapsed_time(e[2]) for e in kern]
    peak, peak_kind = measured_peaks()
    gbs = sum(moved) / (sum(kern_ms) / 1e3) / 1e9
    # one greedy verification over every slot: scores [S][D+1][V], drafts, two outputs per slot
    es = torch.tensor([], dtype=w.logit_dtype).element_size()
    verify_bytes = w.B * (w.D + 1) * w.V * es + w.B * w.D * 4 + w.B * 8
    t_verify = float(np.mean(verify_ms))
    verify_gbs = verify_bytes / (t_verify / 1e3) / 1e9
    return {"value": sum_over_ranks(float(K), ws) / wall, "ms_per_step": wall / K * 1e3,
            "kernel_ms_per_round": float(np.mean(kern_ms)) + t_verify,
            "realign_gbs": round(gbs, 1), "realign_frac": round(gbs / peak, 4),
            "verify": {"kernel": "greedy_kernel", "ms_per_launch": t_verify,
                       "bytes_per_launch": verify_bytes, "achieved_gbs": round(verify_gbs, 1),
                       "frac": round(verify_gbs / peak, 4),
                       "traffic": captured_traffic("greedy_kernel", verify_bytes)},
            "peak": peak, "peak_source": peak_kind,
            "uniform_row_fraction_per_round": [round(x, 3) for x in uniform_frac],
            "mixed_rows_per_round": mixed_rows}


# ------------------------------------------------------------------------------ serving pool

def run_serving(args, rank, ws):
    """The SequencePool lifecycle under a closed loop of requests on the pool workload's cache
    (Vicuna-7B-shaped, 256 slots, D=5, V=32000): prompts from the 8 discrete lengths, each
    generating U[32, 128] tokens (length limit) with end-of-sequence token 2.  A round is
    schedule (+ one readback) -> admission of waiting requests into the freed slots and arena runs
    -> greedy verification of every slot -> per batch gather / append with retirement.  The
    prompts' K/V (the target's prefill) and the verification pass's K/V belong to the model and
    are not written; the copies move the same bytes either way."""
    import numpy as np
    import torch
    from speculative_decoding_specdec_gb300 import synth
    from speculative_decoding_specdec_gb300.engine import SequencePool

    w = workload(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    K, Wm = args.steps, args.warmup
    R = K + Wm
    S, D = w.B, w.D
    gen = synth.make_gen(w.seed * 1000 + 17 + rank)
    nreq = 6 * S
    plen = synth.lengths_discrete(gen, nreq, w.prompt[1]).tolist()
    limits = [int(n) + int(x) for n, x in zip(plen, torch.randint(32, 129, (nreq,), generator=gen))]
    prompts = [torch.randint(0, w.V, (int(n),), generator=gen).tolist() for n in plen]
    max_len = max(limits)
    mean_need = float(np.mean(limits)) + D - 1
    arena_cols = int(1.15 * mean_need * S)
    free, _ = torch.cuda.mem_get_info()
    need = (arena_cols + 8 * (max_len + D + 1)) * w.token_bytes + R * S * (D + 1) * w.V * 2
    if need > 0.85 * free:
        raise SystemExit(f"serving pool needs {need / 1e9:.0f} GB, {free / 1e9:.0f} GB free")
    pool = SequencePool(w.layers, w.heads, w.head_dim, w.kv_dtype, S, arena_cols, D, max_len,
                        batch_size=8, window=args.window, eos_id=2, device=dev,
                        scheduled=args.realign_schedule == "counter")
    alpha = (torch.rand(S, generator=gen) * 0.4 + 0.5).to(dev)    # acceptance U[0.5, 0.9] per slot
    g = torch.Generator(device=dev).manual_seed(w.seed)
    logits, drafts = [], []
    for _ in range(R):
        lg, d = synth.greedy_round(g, S, D, w.V, alpha, dtype=w.logit_dtype, device=dev)
        logits.append(lg)
        drafts.append(d)
    nxt = 0

    def admit():
        nonlocal nxt
        got = pool.admit(prompts[nxt:nxt + S], limits[nxt:nxt + S])
        nxt += len(got)
        return len(got)

    pool.schedule()
    admit()
    stream = torch.cuda.current_stream()
    stats = {"committed": 0, "finished": 0, "admitted": 0, "active": 0, "batches": 0,
             "uniform_rows": 0, "rows": 0, "moved": 0, "pad": 0, "cols": 0}
    dev_ms = []

    def one_round(r, timed):
        before = list(pool.host_len)
        batches, fin = pool.schedule()
        after = pool.host_len
        prev = getattr(one_round, "prev_rows", [])
        prev_mixed = getattr(one_round, "prev_mixed", [])
        if timed:
            stats["committed"] += sum(after[s] - before[s] for s in prev)
            stats["finished"] += len(fin)
            # append of the last round's gathered rows: a + 1 columns each (retirement may cut a
            # sequence shorter, so this slightly undercounts)
            stats["moved"] += 2 * sum(after[s] - before[s] for s in prev_mixed) * w.token_bytes
        n_adm = admit()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(stream)
        pool.verify_greedy(logits[r], drafts[r])
        for off, k, uni in batches:
            pool.gather(off, k, uni)
            pool.append(off, k, uni, drafts[r])
        ev[1].record(stream)
        rows = pool.host_perm
        mixed = [s for off, k, uni in batches if not uni for s in rows[off:off + k]]
        one_round.prev_rows = rows
        one_round.prev_mixed = mixed
        if timed:
            stats["moved"] += 2 * sum(after[s] - 1 for s in mixed) * w.token_bytes   # gather
            for off, k, _ in batches:
                lens = [after[s] for s in rows[off:off + k]]
                stats["pad"] += sum(max(lens) - x for x in lens)
                stats["cols"] += max(lens) * len(lens)
            dev_ms.append(ev)
            stats["admitted"] += n_adm
            stats["active"] += len(rows)
            stats["batches"] += len(batches)
            stats["uniform_rows"] += sum(k for _, k, uni in batches if uni)
            stats["rows"] += len(rows)

    for r in range(Wm):
        one_round(r, False)
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    for i in range(K):
        one_round(Wm + i, True)
    torch.cuda.synchronize()
    wall = max_over_ranks(time.perf_counter() - t0, ws)
    if int(pool.status.item()):
        raise RuntimeError(f"device status {int(pool.status.item())}")
    # the schedule kernel alone, on the final pool state (no finished slots left to report)
    pool.schedule()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    from speculative_decoding_specdec_gb300 import specdec as sd
    args_s = (pool.slot_state, pool.slot_len, pool.bs, pool.window, pool.perm, pool.offsets,
              pool.uniform, pool.finished, pool.reason, pool.counts, pool.status)
    for _ in range(5):
        sd.pool_schedule(*args_s)
    e0.record(stream)
    for _ in range(50):
        sd.pool_schedule(*args_s)
    e1.record(stream)
    torch.cuda.synchronize()
    sched_us = e0.elapsed_time(e1) / 50 * 1e3
    dev_total_s = sum(e[0].elapsed_time(e[1]) for e in dev_ms) / 1e3
    peak, peak_kind = measured_peaks()
    gbs = stats["moved"] / dev_total_s / 1e9
    return {"value": sum_over_ranks(float(K), ws) / wall, "ms_per_step": wall / K * 1e3,
            "device_ms_per_round": float(np.mean([e[0].elapsed_time(e[1]) for e in dev_ms])),
            "committed_tokens_per_s": sum_over_ranks(float(stats["committed"]), ws) / wall,
            "finished_per_round": stats["finished"] / K, "admitted_per_round": stats["admitted"] / K,
            "active_rows_per_round": stats["active"] / K,
            "batches_per_round": stats["batches"] / K,
            "uniform_row_fraction": round(stats["uniform_rows"] / max(1, stats["rows"]), 3),
            "pad_fraction": round(stats["pad"] / max(1, stats["cols"]), 4),
            "moved_gb_per_round": round(stats["moved"] / K / 1e9, 2),
            "gather_append_gbs": round(gbs, 1), "gather_append_frac": round(gbs / peak, 4),
            "peak": peak, "peak_source": peak_kind,
            "schedule_kernel_us": round(sched_us, 2), "slots": S, "arena_cols": arena_cols,
            "window": args.window, "requests_admitted_total": nxt}


# ------------------------------------------------------------------------------ batch sweep

def run_sweep(args, rank, ws):
    """EQSPEC rounds on the contiguous layout for B = 1..64 (Vicuna-7B-shaped cache, pool length
    distribution): per B the realignment time, the bytes it moves (surviving columns only) and
    the bytes a padded-row copy would move (2 * B * W' * P_tok), whose growth with B is the
    superlinear term."""
    import numpy as np
    import torch
    from speculative_decoding_specdec_gb300 import synth
    from speculative_decoding_specdec_gb300.engine import EqspecBatch

    base = synth.WORKLOADS["exspec_pool"]
    dev = torch.device("cuda", torch.cuda.current_device())
    K, Wm = args.steps, args.warmup
    R = K + Wm
    peak, peak_kind = measured_peaks()
    out = []
    for B in (1, 2, 4, 8, 16, 32, 64):
        gen = synth.make_gen(base.seed * 100 + B)
        n0 = synth.lengths_discrete(gen, B, base.prompt[1])
        prompts = [torch.randint(0, base.V, (int(n),), generator=gen).tolist() for n in n0]
        cap = int(n0.max()) + R * (base.D + 1) + base.D + 1
        eng = EqspecBatch(base.layers, base.heads, base.head_dim, base.kv_dtype, B, base.D, cap, R,
                          device=dev, in_place=not args.ping_pong,
                          scheduled=args.realign_schedule == "counter")
        g = torch.Generator(device=dev).manual_seed(B)
        rounds = [synth.greedy_round(g, B, base.D, base.V, 0.7, dtype=base.logit_dtype, device=dev)
                  for _ in range(R)]
        eng.start(prompts)
        stream = torch.cuda.current_stream()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(R)]
        for r, (lg, d) in enumerate(rounds):
            if B == 1:  # nothing moves, so the device idles: keep the host's launch out of the events
                torch.cuda._sleep(200_000)
            ev[r][2].record(stream)
            eng.verify_greedy(lg, d)
            ev[r][0].record(stream)
            eng.realign(d)
            ev[r][1].record(stream)
        torch.cuda.synchronize()
        ms = [ev[r][0].elapsed_time(ev[r][1]) for r in range(Wm, R)]
        vms = [ev[r][2].elapsed_time(ev[r][0]) for r in range(Wm, R)]
        es = torch.tensor([], dtype=base.logit_dtype).element_size()
        vbytes = B * (base.D + 1) * base.V * es + B * base.D * 4 + B * 8
        nh = eng.n_hist.cpu().numpy().astype(np.int64)
        wh = eng.w_hist.cpu().numpy().astype(np.int64)[:, 0]
        def moved(r):  # N'_b - 1 columns per row; in place, rows that do not shift move nothing
            cols = nh[r + 1] - 1
            if not args.ping_pong:
                cols = cols[(wh[r + 1] - nh[r + 1]) - (wh[r] - nh[r]) != 0]
            return cols.sum()
        alg = [2.0 * moved(r) * base.token_bytes for r in range(Wm, R)]
        committed = float(np.mean([(nh[r + 1] - nh[r]).sum() for r in range(Wm, R)]))
        padded = [2.0 * B * (wh[r + 1] - 1) * base.token_bytes for r in range(Wm, R)]
        gbs = sum(alg) / (sum(ms) / 1e3) / 1e9
        out.append({"B": B, "realign_ms_per_round": round(float(np.mean(ms)), 4),
                    "realign_gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                    "moved_gb_per_round": round(float(np.mean(alg)) / 1e9, 3),
                    "padded_copy_gb_per_round": round(float(np.mean(padded)) / 1e9, 3),
                    "mean_width": round(float(np.mean(wh[Wm + 1:R + 1])), 1),
                    "verify_ms_per_round": round(float(np.mean(vms)), 4),
                    "round_ms": round(float(np.mean(ms)) + float(np.mean(vms)), 4),
                    "committed_per_round": committed,
                    "verify_frac": round(vbytes / (float(np.mean(vms)) / 1e3) / 1e9 / peak, 4)})
        del eng, rounds
        torch.cuda.empty_cache()
    return {"sweep": out, "peak": peak, "peak_source": peak_kind}


# ------------------------------------------------------------------------------ CPU oracle

def host_memory_available():
    """Bytes this process can still allocate on the host: MemAvailable, capped by the cgroup's
    memory limit where one is set."""
    avail = None
    try:
        with open("/proc/meminfo") as f:
            for ln in f:
                if ln.startswith("MemAvailable:"):
                    avail = int(ln.split()[1]) * 1024
    except OSError:
        pass
    try:
        with open("/sys/fs/cgroup/memory.max") as f:
            lim = f.read().strip()
        with open("/sys/fs/cgroup/memory.current") as f:
            cur = int(f.read().strip())
        if lim != "max":
            room = int(lim) - cur
            avail = room if avail is None else min(avail, room)
    except (OSError, ValueError):
        pass
    return avail if avail is not None else 1 << 62


def oracle_rounds(wname, rounds, layers=None, seed=0):
    """Full rounds of the workload for the oracle: greedy or sampled verification of every row,
    then the realignment of the whole cache (``layers``: all of them by default), two buffers of
    the workload's geometry and capacity for ``rounds`` rounds.  The caches are filled with a
    constant (the oracle only moves values).  Returns (workload, layers used, one_round), where
    one_round() generates the next round's inputs (untimed) and returns the seconds spent in the
    oracle's verification and realignment."""
    import numpy as np
    import torch
    from oracle import specdec_oracle as O
    from speculative_decoding_specdec_gb300 import synth

    w = synth.WORKLOADS[wname]
    if w.mode not in ("greedy", "sampled"):
        raise ValueError(f"{wname}: no oracle round for this workload")
    gen = synth.make_gen(w.seed * 1000 + seed)
    n = w.prompt_lengths(gen).numpy().astype(np.int64)
    prompts = [torch.randint(0, w.V, (int(k),), generator=gen).tolist() for k in n]
    W = int(n.max())
    cap = w.capacity(W, rounds=rounds)
    Ls = w.layers if layers is None else min(layers, w.layers)
    dt = np.int16 if w.kv_dtype == torch.bfloat16 else np.int32  # same bytes as the K/V dtype
    kv = [np.full((Ls, 2, w.B, w.heads, cap, w.head_dim), 7, dtype=dt) for _ in range(2)]
    ids = np.zeros((w.B, cap), np.int32)
    for b, pr in enumerate(prompts):
        ids[b, W - len(pr):W] = pr
    state = {"n": n, "W": W, "ids": ids, "cur": 0}

    def one_round():
        if w.mode == "greedy":
            lg, d = synth.greedy_round(gen, w.B, w.D, w.V, w.alpha, dtype=w.logit_dtype)
            lg64 = lg.double().numpy()
            t0 = time.perf_counter()
            a, y = O.verify_greedy(lg64, d.numpy())
        else:
            lg, dl, d, u = synth.sampled_round(gen, w.B, w.D, w.V, w.temperature,
                                               dtype=w.logit_dtype)
            lg64, dl64, u64 = lg.double().numpy(), dl.double().numpy(), u.double().numpy()
            t0 = time.perf_counter()
            a, y, _, _ = O.verify_sample(lg64, dl64, d.numpy(), u64, w.temperature)
        t1 = time.perf_counter()
        c = state["cur"]
        out, ids2, _, _, n2, W2 = O.realign(kv[c], kv[1 - c], state["n"], state["W"], a, y,
                                            d.numpy(), state["ids"], 0)
        t2 = time.perf_counter()
        kv[1 - c] = out
        state.update(n=n2.astype(np.int64), W=W2, ids=ids2, cur=1 - c)
        return t1 - t0, t2 - t1

    return w, Ls, one_round


def oracle_bytes(wname, rounds):
    """Host bytes the oracle's full rounds hold at once: two caches and the one a realignment
    returns."""
    import torch
    from speculative_decoding_specdec_gb300 import synth
    w = synth.WORKLOADS[wname]
    gen = synth.make_gen(w.seed * 1000)
    cap = w.capacity(int(w.prompt_lengths(gen).max()), rounds=rounds)
    es = torch.tensor([], dtype=w.kv_dtype).element_size()
    return 3 * w.layers * 2 * w.B * w.heads * cap * w.head_dim * es


def oracle_layers(wname, rounds):
    """None (realign every layer) when the host can hold the oracle's caches for ``rounds``
    rounds, else the number of layers that fits (the caller scales that sample and says so)."""
    from speculative_decoding_specdec_gb300 import synth
    w = synth.WORKLOADS[wname]
    need, avail = oracle_bytes(wname, rounds), host_memory_available()
    return None if need <= 0.6 * avail else max(1, int(w.layers * 0.6 * avail / need))


def time_oracle(wname, budget_s=15.0, max_rounds=60):
    """Rounds/s of the oracle over whole rounds (every layer realigned unless the host cannot
    hold them: then a layer sample scaled to all layers), as many as fit the budget (at least
    one).  Returns (rounds/s, rounds timed, layers realigned, workload)."""
    w, Ls, one_round = oracle_rounds(wname, max_rounds, layers=oracle_layers(wname, max_rounds))
    total, rounds = 0.0, 0
    start = time.perf_counter()
    while True:
        t_verify, t_realign = one_round()
        total += t_verify + t_realign * (w.layers / Ls)
        rounds += 1
        if time.perf_counter() - start > budget_s or rounds >= max_rounds:
            break
    return rounds / total, rounds, Ls, w


def time_cpu_parallel(wname, budget_s=8.0, max_rounds=60, layers_sample=None):
    """Rounds/s of the row-parallel C++ baseline (oracle/specdec_cpu_parallel.cpp, one
    std::thread per host core) on whole rounds of the workload: verification of every row
    (greedy or sampled) and realignment of every layer, unless ``layers_sample`` is given or the
    host cannot hold two caches (then that many layers, scaled to all layers, and said so)."""
    import numpy as np
    import torch
    from oracle import _build_cpu
    from speculative_decoding_specdec_gb300 import synth

    w = synth.WORKLOADS[wname]
    lib = _build_cpu.load()
    threads = len(os.sched_getaffinity(0)) or 1  # the cores this process may run on
    gen = synth.make_gen(w.seed * 1000)
    n = w.prompt_lengths(gen).numpy().astype(np.int32)
    W = int(n.max())
    cap = w.capacity(W, rounds=max_rounds)
    es = 2 if w.kv_dtype == torch.bfloat16 else 4
    if layers_sample is None:  # two caches of every layer, if they fit in 60 % of free memory
        per_layer = 2 * 2 * w.B * w.heads * cap * w.head_dim * es
        layers_sample = max(1, min(w.layers, int(0.6 * host_memory_available() // per_layer)))
    Ls = min(layers_sample, w.layers)
    # K/V contents do not matter to a copy: a constant fill touches every page quickly
    kv = [np.full((Ls, 2, w.B, w.heads, cap, w.head_dim * es // 2), 7, dtype=np.int16)
          for _ in range(2)]
    ids = [np.zeros((w.B, cap), np.int32) for _ in range(2)]
    mask = np.zeros((w.B, cap), np.uint8)
    pos = np.zeros((w.B, cap), np.int32)
    n_out = np.zeros(w.B, np.int32)
    w_out = np.zeros(1, np.int32)
    a = np.zeros(w.B, np.int32)
    y = np.zeros(w.B, np.int32)
    dt = 1 if w.logit_dtype == torch.bfloat16 else 0
    cur, total, rounds = 0, 0.0, 0
    start = time.perf_counter()
    while True:
        host = lambda t: np.ascontiguousarray((t.view(torch.int16) if dt else t).numpy())  # noqa: E731
        if w.mode == "greedy":
            lg, d = synth.greedy_round(gen, w.B, w.D, w.V, w.alpha, dtype=w.logit_dtype)
            raw = host(lg)
            dd = np.ascontiguousarray(d.numpy().astype(np.int32))
            t0 = time.perf_counter()
            rc = lib.cpu_verify_greedy(raw.ctypes.data, dt, w.B, w.D, w.V, dd.ctypes.data,
                                       a.ctypes.data, y.ctypes.data, threads)
        else:
            lg, dl, d, u = synth.sampled_round(gen, w.B, w.D, w.V, w.temperature,
                                               dtype=w.logit_dtype)
            raw, rawd = host(lg), host(dl)
            dd = np.ascontiguousarray(d.numpy().astype(np.int32))
            uu = np.ascontiguousarray(u.numpy().astype(np.float32))
            t0 = time.perf_counter()
            rc = lib.cpu_verify_sample(raw.ctypes.data, rawd.ctypes.data, dt, w.B, w.D, w.V,
                                       dd.ctypes.data, uu.ctypes.data, float(w.temperature),
                                       a.ctypes.data, y.ctypes.data, threads)
        t1 = time.perf_counter()
        rc |= lib.cpu_realign(kv[cur].ctypes.data, kv[1 - cur].ctypes.data, Ls, w.B, w.heads, cap,
                              cap, w.head_dim * es, w.D, n.ctypes.data, W, a.ctypes.data,
                              y.ctypes.data, dd.ctypes.data, ids[cur].ctypes.data,
                              ids[1 - cur].ctypes.data, mask.ctypes.data, pos.ctypes.data,
                              n_out.ctypes.data, w_out.ctypes.data, 0, threads)
        t2 = time.perf_counter()
        if rc:
            raise RuntimeError(f"CPU baseline error {rc}")
        n, W, cur = n_out.copy(), int(w_out[0]), 1 - cur
        total += (t1 - t0) + (t2 - t1) * (w.layers / Ls)
        rounds += 1
        if time.perf_counter() - start > budget_s or rounds >= max_rounds:
            break
    return {"value": rounds / total, "unit": "rounds/s", "cores": threads,
            "kind": "row-parallel C++ baseline (std::thread over score rows and K/V runs)",
            "sample": f"{rounds} whole rounds: {w.mode} verification of all rows, realignment of "
                      f"all {w.layers} layers" if Ls == w.layers else
                      f"{rounds} rounds: {w.mode} verification of all rows, realignment of {Ls} of "
                      f"{w.layers} layers scaled x{w.layers / Ls:g} (host memory)"}


def run_reference(args, rank, ws):
    """The reference arm: the oracle, as it stands, on this host's cores.  W untimed and then K
    timed whole rounds of the workload (verification of every row, realignment of every layer),
    one round per step.  Only where the host cannot hold the oracle's caches does it realign a
    sample of the layers, scaled to all of them, and the line says so (``extrapolated``)."""
    if rank != 0:
        return None
    from speculative_decoding_specdec_gb300 import synth
    R = args.warmup + args.steps
    need, avail = oracle_bytes(args.workload, R), host_memory_available()
    w, Ls, one_round = oracle_rounds(args.workload, R, layers=oracle_layers(args.workload, R))
    for _ in range(args.warmup):
        one_round()
    tv, tr = 0.0, 0.0
    for _ in range(args.steps):
        a, b = one_round()
        tv, tr = tv + a, tr + b
    scale = w.layers / Ls
    out = {"value": args.steps / (tv + tr * scale), "ms_per_step": (tv + tr) / args.steps * 1e3}
    if Ls < w.layers:
        out["extrapolated"] = {"layers_timed": Ls, "scale": scale,
                               "why": f"host memory: {need / 1e9:.0f} GB needed for every layer, "
                                      f"{avail / 1e9:.0f} GB available"}
        sample = (f"{args.steps} rounds of {w.name} after {args.warmup} untimed: verification of "
                  f"all {w.B} rows, realignment of {Ls} of {w.layers} layers scaled x{scale:g}")
    else:
        sample = (f"{args.steps} whole rounds of {w.name} after {args.warmup} untimed: "
                  f"verification of all {w.B} rows, realignment of all {w.layers} layers")
    out["cpu_baseline"] = {"value": out["value"], "unit": "rounds/s", "cores": 1,
                           "kind": "oracle", "sample": sample}
    return out


# ------------------------------------------------------------------------------ read floor

def run_floor(args):
    """How long a plain streaming read of each verification input takes on this GPU, beside the
    verification kernel on the same bytes: CUDA events around one launch queued behind a device
    sleep, after (a) a 2 GB device copy that leaves L2 full of dirty lines (as a realignment does
    before the next round's verification) and (b) a 512 MB read that leaves it clean.  The plain
    reads are torch's amax over the bf16 scores and torch's sum over the same bytes viewed as
    fp32 (its fastest plain read here: 6.4 TB/s over 4 GB); each is one library reduction kernel
    that reads every byte once.
    The inputs are the workloads' own score shapes: Vicuna-7B 3.07 MB, Qwen3-8B 24.3 MB, the
    EXSPEC pool 98.3 MB (greedy) and GLM-4-9B 126.1 MB (sampled, target and draft rows)."""
    import statistics
    import torch
    from speculative_decoding_specdec_gb300 import specdec as sd
    from speculative_decoding_specdec_gb300 import synth

    dev = torch.device("cuda", torch.cuda.current_device())
    s = torch.cuda.current_stream()
    clean = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    big_a = torch.empty(1 << 31, dtype=torch.uint8, device=dev)
    big_b = torch.empty_like(big_a)
    reps = max(5, args.steps)
    out = []
    for name in ("vicuna7b", "qwen3_8b", "exspec_pool", "glm4_9b"):
        w = synth.WORKLOADS[name]
        g = torch.Generator(device=dev).manual_seed(w.seed)
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        a = torch.empty(w.B, dtype=torch.int32, device=dev)
        y = torch.empty(w.B, dtype=torch.int32, device=dev)
        if w.mode == "sampled":
            tl, dl, d, u = synth.sampled_round(g, w.B, w.D, w.V, w.temperature, device=dev)
            parts = (tl, dl)

            def verify():
                sd.verify_sample(tl, dl, d, u, w.temperature, a, y, st)
        else:
            lg, d = synth.greedy_round(g, w.B, w.D, w.V, 0.7, device=dev)
            parts = (lg,)
            ws = torch.zeros(sd.greedy_workspace_bytes(w.B, w.D), dtype=torch.uint8, device=dev)

            def verify():
                sd.verify_greedy(lg, d, a, y, st, ws)
        nbytes = sum(x.numel() * x.element_size() for x in parts)
        flat = torch.cat([x.reshape(-1) for x in parts])  # the same bytes in one tensor
        red = torch.empty((), dtype=flat.dtype, device=dev)

        words = flat.view(torch.float32)  # the same bytes as fp32 words
        red32 = torch.empty((), dtype=torch.float32, device=dev)

        def read():
            torch.amax(flat, dim=0, out=red)

        def sum_read():
            torch.sum(words, dim=0, out=red32)
        timed = [("read_us", read), ("sum_read_us", sum_read), ("verify_us", verify)]
        if w.mode == "sampled":
            # the same bytes through this library's bulk-copy streaming kernel: greedy
            # verification of the 2D+1 rows per batch row as one score tensor
            rows = flat.view(w.B, 2 * w.D + 1, w.V)
            d2 = torch.randint(0, w.V, (w.B, 2 * w.D), generator=g, device=dev, dtype=torch.int32)
            ws2 = torch.zeros(sd.greedy_workspace_bytes(w.B, 2 * w.D), dtype=torch.uint8,
                              device=dev)

            def ring_read():
                sd.verify_greedy(rows, d2, a, y, st, ws2)
            timed.append(("ring_read_us", ring_read))
        row = {"workload": name, "verify": w.mode, "mb": round(nbytes / 1e6, 2)}
        for cond in ("dirty", "clean"):
            for what, fn in timed:
                fn()
                t = []
                for _ in range(reps):
                    if cond == "dirty":
                        big_b.copy_(big_a)
                    else:
                        torch.amax(clean, dim=0)
                    torch.cuda._sleep(100_000)
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(s)
                    fn()
                    e1.record(s)
                    torch.cuda.synchronize()
                    t.append(e0.elapsed_time(e1) * 1e3)
                row[f"{what}_{cond}"] = round(statistics.median(t), 2)
        if int(st.item()):
            raise RuntimeError(f"device status {int(st.item())}")
        peak, _ = measured_peaks()
        for cond in ("dirty", "clean"):
            for what, _ in timed:
                key = what[:-3]
                row[f"{key}_frac_{cond}"] = round(
                    nbytes / (row[f"{what}_{cond}"] * 1e-6) / 1e9 / peak, 4)
        out.append(row)
        del flat, parts, timed
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------------------ all configs

def _sub_args(args, name):
    import argparse
    sub = argparse.Namespace(**vars(args))
    sub.workload, sub.no_e2e, sub.top_k, sub.top_p, sub.philox = name, True, 0, 1.0, False
    sub.layers = 0
    return sub


def _release():
    import gc
    import torch
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def specdec_summary(name, res, K, Wm):
    """One workload's entry of the all_configs block."""
    from speculative_decoding_specdec_gb300 import synth
    w = synth.WORKLOADS[name]
    rf, vf = res["roofline"], res["verify"]
    return {"workload": f"{w.name}: L={w.layers} KV heads={w.heads} head_dim={w.head_dim} B={w.B} "
                        f"D={w.D} V={w.V} {w.mode} verify",
            "steps": K, "warmup": Wm, "ms_per_step": res["ms_per_step"],
            "rounds_per_s": res["value"],
            "committed_token_slots_per_s": res["committed_slots_per_s"],
            "mean_accept_len": res["acceptance"]["mean_accept_len"],
            "realign": {"ms_per_launch": rf["ms_per_launch"], "bytes_per_launch": rf["bytes_per_launch"],
                        "gbs": rf["achieved"], "frac": rf["frac"]},
            "verify": {"kernel": vf["kernel"], "us_per_launch": vf["ms_per_launch"] * 1e3,
                       "bytes_per_launch": vf["bytes_per_launch"], "gbs": vf["achieved_gbs"],
                       "frac": vf["frac"]},
            "launch": res["launch"], "clocks": res["clocks"]}


def run_all_configs(args, rank, ws, headline=None):
    """Every other workload at the same steps and warm-up, one after another on this GPU, each
    with its own caches (freed before the next): the model-shaped EQSPEC rounds, the tiny
    correctness-sized round, the GLM-4-9B-shaped round under top-k 50 and under top-p 0.9, the
    EXSPEC pool, and the EQSPEC batch-size sweep B = 1..64."""
    out = {}
    if headline is not None:
        out[args.workload] = headline
    K, Wm = args.steps, args.warmup
    for name in ("tiny", "vicuna7b", "qwen3_8b", "glm4_9b"):
        if name == args.workload:
            continue
        _release()
        out[name] = specdec_summary(name, run_specdec(_sub_args(args, name), rank, ws, 0), K, Wm)
    # the sampled workload under the sampling settings (keep bounds, then masked verification)
    for key, top_k, top_p in (("glm4_9b_top_k50", 50, 1.0), ("glm4_9b_top_p0.9", 0, 0.9)):
        _release()
        sub = _sub_args(args, "glm4_9b")
        sub.top_k, sub.top_p = top_k, top_p
        entry = specdec_summary("glm4_9b", run_specdec(sub, rank, ws, 0), K, Wm)
        entry["workload"] += (f", top-k {top_k} (drafts from the draft model's top {top_k})"
                              if top_k else f", top-p {top_p}")
        out[key] = entry
    _release()
    pool = run_pool(_sub_args(args, "exspec_pool"), rank, ws)
    out["exspec_pool"] = {
        "workload": "exspec_pool: 256 sequences, L=32 KV heads=32 head_dim=128, D=5, V=32000, "
                    "prompts from {256,...,2048}, acceptance U[0.5,0.9] per sequence, batches of "
                    "8, greedy verify",
        "steps": K, "warmup": Wm, "ms_per_step": pool["ms_per_step"],
        "pool_rounds_per_s": pool["value"],
        "gather_append": {"gbs": pool["realign_gbs"], "frac": pool["realign_frac"]},
        "verify": {"kernel": "greedy_kernel", "us_per_launch": pool["verify"]["ms_per_launch"] * 1e3,
                   "bytes_per_launch": pool["verify"]["bytes_per_launch"],
                   "gbs": pool["verify"]["achieved_gbs"], "frac": pool["verify"]["frac"]},
        "mixed_rows_per_round": round(sum(pool["mixed_rows_per_round"]) /
                                      max(1, len(pool["mixed_rows_per_round"])), 1)}
    _release()
    sweep = run_sweep(_sub_args(args, "exspec_sweep"), rank, ws)
    out["batch_sweep"] = {
        "workload": "EQSPEC verify+realign on the contiguous layout, Vicuna-7B-shaped cache, "
                    "prompts from {256,...,2048}, D=5, V=32000, greedy, B in 1..64, in place",
        "steps": K, "warmup": Wm, "points": sweep["sweep"]}
    _release()
    return out


# ------------------------------------------------------------------------------ main

def workload_config(args, w, ws):
    """The ``config`` both arms print: what the workload is (geometry, batch, drafts, vocabulary,
    cache capacity, how its inputs relate to L2), nothing about how it is run."""
    import torch
    from speculative_decoding_specdec_gb300 import synth
    filtered = w.mode == "sampled" and (args.top_k > 0 or args.top_p < 1.0)
    R = args.steps + args.warmup
    cap = w.capacity(int(w.prompt_lengths(synth.make_gen(w.seed * 1000)).max()), rounds=R)
    les = torch.tensor([], dtype=w.logit_dtype).element_size()
    score_bytes = w.B * (w.D + 1) * w.V * les + (w.B * w.D * w.V * les if w.mode == "sampled" else 0)
    cache_bytes = w.token_bytes * w.B * cap
    if score_bytes + cache_bytes > 2 * L2_BYTES:
        l2 = (f"inputs larger than L2: a {cache_bytes / 1e9:.1f} GB K/V cache whose surviving "
              f"columns every round moves, and {score_bytes / 1e6:.1f} MB of score rows per round, "
              f"all rounds' rows distinct and generated before the timed region")
    else:
        l2 = (f"inputs smaller than L2 ({(cache_bytes + score_bytes) / 1e6:.3f} MB) and L2 not "
              f"flushed: a latency-bound correctness-sized workload, not a bandwidth figure")
    return {"workload": f"{w.name}: L={w.layers} KV heads={w.heads} head_dim={w.head_dim} "
                        f"B={w.B} D={w.D} V={w.V} {w.mode} verify",
            "B": w.B, "D": w.D, "V": w.V, "layers": w.layers, "kv_heads": w.heads,
            "head_dim": w.head_dim, "verify": w.mode,
            **({"top_k": args.top_k, "top_p": args.top_p} if filtered else {}),
            "parallelism": f"replicas x{ws}", "cap_cols": cap, "l2": l2}


def main():
    args = parse()
    rank, ws, local = dist_setup(args.gpus)
    w = workload(args)
    filtered = w.mode == "sampled" and (args.top_k > 0 or args.top_p < 1.0)  # + the filter kernel
    # the arithmetic the path computes in: greedy verification orders the scores as they are
    # stored (bf16 or fp32, exactly), sampled verification sums fp32 exponentials; the
    # realignment only moves bytes
    import torch
    dtype = "f32" if (w.mode == "sampled" or w.logit_dtype == torch.float32) else "bf16"
    line = {"metric": METRIC, "unit": "rounds/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic"}
    if args.workload in ("exspec_pool", "exspec_serving", "exspec_sweep", "read_floor"):
        config = {"workload": args.workload, "parallelism": f"replicas x{ws}",
                  "l2": "inputs larger than L2: every pool round moves tens of GB of K/V; all "
                        "rounds' score rows are distinct and generated before the timed region"}
    else:
        config = workload_config(args, w, ws)
    line["config"] = config
    if args.impl == "reference":
        if args.workload not in ("tiny", "vicuna7b", "qwen3_8b", "glm4_9b"):
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable":
                                  f"no oracle round for the {args.workload} workload"}))
            return
        res = run_reference(args, rank, ws)
        if rank == 0:
            line.update(impl="reference", value=res["value"], ms_per_step=res["ms_per_step"],
                        cpu_baseline=res["cpu_baseline"], dtype="f64",
                        e2e={"value": res["value"], "unit": "rounds/s",
                             "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0})
            if "extrapolated" in res:
                line["extrapolated"] = res["extrapolated"]
            print(json.dumps(line))
        return
    if args.workload == "exspec_pool":
        res = run_pool(args, rank, ws)
        if rank == 0:
            config["workload"] = (f"exspec_pool: {w.B} sequences, L={w.layers} KV heads={w.heads} "
                                  f"head_dim={w.head_dim}, D={w.D}, V={w.V}, prompts from "
                                  f"{{256,...,2048}}, acceptance U[0.5,0.9] per sequence, "
                                  f"batches of 8, greedy verify")
            line.update(value=res.pop("value"), ms_per_step=res.pop("ms_per_step"), pool=res,
                        unit="pool rounds/s", metric="EXSPEC pool rounds/s")
            print(json.dumps(line))
        return
    if args.workload == "exspec_serving":
        res = run_serving(args, rank, ws)
        if rank == 0:
            config["workload"] = (f"exspec_serving: {w.B} slots, L={w.layers} KV heads={w.heads} "
                                  f"head_dim={w.head_dim}, D={w.D}, V={w.V}, prompts from "
                                  f"{{256,...,2048}} generating U[32,128] tokens, acceptance "
                                  f"U[0.5,0.9] per slot, batches of 8, window {args.window}, "
                                  f"greedy verify")
            line.update(value=res.pop("value"), ms_per_step=res.pop("ms_per_step"), pool=res,
                        unit="rounds/s", metric="EXSPEC serving pool rounds/s")
            print(json.dumps(line))
        return
    if args.workload == "read_floor":
        if rank == 0:
            peak, kind = measured_peaks()
            line.update(metric="verification launch vs plain streaming read", unit="us",
                        value=None, higher_is_better=False, peak_gbs=peak, peak_source=kind,
                        floor=run_floor(args))
            line["config"] = {"workload": "read_floor: the verification inputs of vicuna7b, "
                                          "qwen3_8b, exspec_pool and glm4_9b"}
            print(json.dumps(line))
        return
    if args.workload == "exspec_sweep":
        res = run_sweep(args, rank, ws)
        if rank == 0:
            config["workload"] = ("exspec_sweep: EQSPEC verify+realign on the contiguous layout, "
                                  "Vicuna-7B-shaped cache, prompts from {256,...,2048}, D=5, "
                                  "V=32000, B in 1..64")
            line.update(metric="EQSPEC realign batch sweep", unit="ms/round", value=None,
                        higher_is_better=False, **res)
            print(json.dumps(line))
        return
    cores, narrowed = bind_local_cpus(local if ws > 1 else 0)
    res = run_specdec(args, rank, ws, local)
    every = None
    if ws == 1 and not args.no_all_configs:
        every = run_all_configs(args, rank, ws,
                                headline=specdec_summary(args.workload, res, args.steps,
                                                         args.warmup))
    if rank == 0:
        cpu = None
        if ws == 1 and not args.no_cpu_baseline:
            rps, rounds, Ls, _ = time_oracle(args.workload, budget_s=12.0,
                                             max_rounds=args.steps + args.warmup)
            cpu = {"value": rps, "unit": "rounds/s", "cores": 1, "kind": "oracle",
                   "sample": f"{rounds} whole rounds: verification of all {w.B} rows, "
                             f"realignment of all {w.layers} layers" if Ls == w.layers else
                             f"{rounds} rounds: verification of all {w.B} rows, realignment of "
                             f"{Ls} of {w.layers} layers scaled x{w.layers / Ls:g} (host memory)"}
        par = None
        if ws == 1 and not args.no_cpu_baseline:
            par = time_cpu_parallel(args.workload)
        line.update(value=res["value"], ms_per_step=res["ms_per_step"], clocks=res["clocks"],
                    e2e=res["e2e"], roofline=res["roofline"], verify=res["verify"],
                    committed_token_slots_per_s=res["committed_slots_per_s"],
                    committed_per_round=res["committed_per_round"],
                    acceptance=res.get("acceptance"),
                    gpu_launches=(3 if filtered else 2) * args.steps,
                    cpu_baseline=cpu, cpu_parallel=par)
        line["run"] = {"launch": res["launch"], "kv_buffers": 2 if args.ping_pong else 1,
                       "realign_schedule": args.realign_schedule,
                       "host_cpus": f"{cores} cores" + (" local to the GPU (NVML affinity)"
                                                        if narrowed else ""),
                       **({"uniforms": "in-kernel Philox4x32-10"}
                          if args.philox and w.mode == "sampled" else {})}
        if every is not None:
            line["all_configs"] = every
        print(json.dumps(line))


if __name__ == "__main__":
    main()
