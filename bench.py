"""Benchmark: varlen attention forward TFLOP/s and paged GQA decode HBM GB/s on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload longtail|packed|cross-d64|cross-d256|tiny|tiny-causal]
                    [--configs a,b,...]

One step is one pass of the whole hot path on one batch of synthetic input:
the varlen forward (device tile scheduler + prefill kernel) over the headline
workload -- by default the long-tail batch, the largest single-GPU one
(32768 tokens, one 8192-token sequence, H=32, D=128, causal) -- then a full
paged-decode pass (init, every 32-block tile step, finalize) over the decode
workload (64 sequences, context U{128..8192}, 32 q / 8 kv heads, D=128,
block size 16), captured as one CUDA graph.  `value` is the forward's
algorithmic TFLOP/s (4 * H * D * attended pairs); decode is reported under
"decode" in GB/s of algorithmic bytes.

Every prefill workload (long-tail, packed, cross-attention at D=64 and
D=256, tiny) is also timed on its own under "configs": the forward, the
varlen backward and the FP8 q / k forward where the library supports the
head_dim, each with its roofline and the CPU oracle's rate on a sample of
that workload.  L2 is flushed (a 256 MiB write) before each timed call;
device times come from CUDA events on the launching stream, reduced by the
median.  The end-to-end leg ("e2e") times the headline forward through the
public API from pinned host buffers, next to the measured host <-> device
link bandwidth.  Under torchrun each rank runs its own replica (the path has
no exchange step), so scaling is weak.

--impl reference times the fp64 CPU oracle (the only other implementation:
the pages publish no code that runs and no numbers) on a bounded sample of
the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "varlen attn fwd TFLOP/s & % of bf16 tensor peak; paged decode HBM GB/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def _file_hash(path):
    import hashlib
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _traffic(kernel_key):
    """Per-launch DRAM bytes from the committed ncu summary, if its kernel source is unchanged."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[kernel_key]
        src = os.path.join(ROOT, t["source"])
        if _file_hash(src) != t["source_sha256_16"]:
            return None
        return t["dram_bytes_per_launch"]
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t_start = time.time()
        else:
            self.t_stop = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            if self.t_start is not None and not (self.t_start - 0.1 <= t <= self.t_stop + 0.25):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[2]), max=float(parts[3]), power=float(parts[4]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(r["power"] for r in rows)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, world: int, device):
    """Per-rank timings -> their element-wise maximum over all ranks (the slowest rank
    sets the job's time).  With world == 1 the values come back unchanged."""
    vals = [float(v) for v in values]
    if world <= 1:
        return vals
    import torch
    import torch.distributed as dist
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def _oracle_rows_sample(case, n_rows, rng):
    import numpy as np
    H = case.num_heads
    rows = np.stack([rng.integers(0, case.total_q, n_rows), rng.integers(0, H, n_rows)], 1)
    return rows.astype(np.int64)


def _row_flops(case, rows):
    """Algorithmic flops of the sampled rows: 4 * D * visible keys per row."""
    import numpy as np
    cq = case.cu_seqlens_q
    b = np.searchsorted(cq, rows[:, 0], side="right") - 1
    i = rows[:, 0] - cq[b]
    lk = np.asarray(case.lengths_k)[b]
    vis = np.minimum(i + 1, lk) if case.causal else lk
    return int(4 * case.head_dim * vis.sum())


def cpu_oracle_rate(case, seconds: float, seed: int = 0):
    """Time the oracle (as it stands) on random rows of `case` for about `seconds`:
    batches of rows, each sized from the previous batch's rate, until the time is spent."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    n, flops, spent, rows_done, threads = 256, 0, 0.0, 0, 0
    cap = case.total_q * case.num_heads
    while spent < seconds:
        rows = _oracle_rows_sample(case, min(n, cap), rng)
        t0 = time.perf_counter()
        _, _, threads = oracle.varlen_fwd_rows(case.q, case.k, case.v, case.cu_seqlens_q,
                                               case.cu_seqlens_k, case.num_heads,
                                               case.head_dim, case.softmax_scale, case.causal,
                                               rows)
        dt = max(time.perf_counter() - t0, 1e-4)
        flops += _row_flops(case, rows)
        spent += dt
        rows_done += len(rows)
        left = seconds - spent
        # next batch: about half the remaining time (at least 1 s of work), at this rate
        n = int(max(256, len(rows) / dt * max(1.0, 0.5 * left)))
    return flops / spent / 1e12, threads, rows_done, spent


def run_reference(args):
    """The oracle as the reference arm: CPU, bounded sample per step."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np
    import oracle
    from variable_length_flashattention_gb300 import workloads as W
    oracle.build()
    case = W.VARLEN_WORKLOADS[args.workload](args.seed)
    budget = 120.0 / max(1, args.steps + args.warmup)          # seconds of CPU per step
    rng = np.random.default_rng(args.seed)
    rate, threads, _, _ = cpu_oracle_rate(case, min(2.0, budget), args.seed)
    # rows a step's budget covers at that rate, at the workload's average work per row
    from variable_length_flashattention_gb300 import accounting as A
    flops_per_row = A.varlen_flops(case) / max(1, case.total_q * case.num_heads)
    rows_per_step = max(1, int(budget * rate * 1e12 / max(1.0, flops_per_row)))
    rows_per_step = min(rows_per_step, case.total_q * case.num_heads)
    flops_total, t_total = 0, 0.0
    for step in range(args.warmup + args.steps):
        rows = _oracle_rows_sample(case, rows_per_step, rng)
        t0 = time.perf_counter()
        oracle.varlen_fwd_rows(case.q, case.k, case.v, case.cu_seqlens_q, case.cu_seqlens_k,
                               case.num_heads, case.head_dim, case.softmax_scale, case.causal,
                               rows)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            flops_total += _row_flops(case, rows)
            t_total += dt
    value = flops_total / t_total / 1e12
    sample = f"{rows_per_step} random (token, head) rows of the {args.workload} workload per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * t_total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "seed": args.seed},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
        "note": "fp64 CPU oracle; the pages publish no runnable implementation and no numbers",
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm

PREFILL_CONFIGS = ("longtail", "packed", "cross-d64", "cross-d256", "tiny", "tiny-causal")


def _median(xs):
    return float(statistics.median(xs)) if xs else None


class PrefillLeg:
    """One varlen workload resident in HBM, with its forward, backward and FP8
    forward calls (the latter two where the library supports the head_dim)."""

    def __init__(self, name, seed, dev, want_bwd=True, want_fp8=True):
        import torch
        from variable_length_flashattention_gb300 import accounting as A
        from variable_length_flashattention_gb300 import vfa, workloads as W
        self.name = name
        case = W.VARLEN_WORKLOADS[name](seed)
        self.case = case
        self.q, self.k, self.v = case.q.to(dev), case.k.to(dev), case.v.to(dev)
        self.cuq = torch.from_numpy(case.cu_seqlens_q).to(dev)
        self.cuk = torch.from_numpy(case.cu_seqlens_k).to(dev)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(case.total_q, case.num_heads, dtype=torch.float32, device=dev)
        self.ws = vfa.alloc_workspace(case.batch, case.total_q, case.total_k, case.num_heads,
                                      case.head_dim, device=dev)
        self.flops = A.varlen_flops(case)
        self.bwd_flops = A.varlen_bwd_flops(case)
        self.ctx_bytes = A.varlen_context_bytes(case)
        self.bwd = self.fp8 = None
        L = vfa.lib()
        self.fwd()
        if want_bwd and L.vfa_varlen_bwd_workspace_bytes(case.batch, case.total_q,
                                                         case.num_heads, case.head_dim) > 0:
            self.g = W.upstream_grad(case, seed).to(dev)
            self.dq = torch.empty_like(self.q)
            self.dk, self.dv = torch.empty_like(self.k), torch.empty_like(self.v)
            self.bws = vfa.alloc_bwd_workspace(case.batch, case.total_q, case.num_heads,
                                               case.head_dim, device=dev)
            self.bwd = self._bwd
        if want_fp8:
            f8 = W.fp8_qk(case)
            self.f8 = f8
            self.q8, self.k8 = f8.q8.to(dev), f8.k8.to(dev)
            self.out8 = torch.empty_like(self.q)
            self.lse8 = torch.empty_like(self.lse)
            try:
                self._fp8()
                self.fp8 = self._fp8
            except vfa.VfaError as e:
                if e.status != vfa.VFA_ERR_UNSUPPORTED:
                    raise
        torch.cuda.synchronize()
        self.check()

    def fwd(self, stream=None):
        from variable_length_flashattention_gb300 import vfa
        c = self.case
        vfa.varlen_fwd(self.q, self.k, self.v, self.cuq, self.cuk, c.max_seqlen_q,
                       c.softmax_scale, c.causal, out=self.out, lse=self.lse, workspace=self.ws,
                       stream=stream)

    def _bwd(self):
        from variable_length_flashattention_gb300 import vfa
        c = self.case
        vfa.varlen_bwd(self.q, self.k, self.v, self.out, self.g, self.lse, self.cuq, self.cuk,
                       c.softmax_scale, c.causal, dq=self.dq, dk=self.dk, dv=self.dv,
                       workspace=self.bws)

    def _fp8(self):
        from variable_length_flashattention_gb300 import vfa
        c = self.case
        vfa.varlen_fwd_fp8(self.q8, self.k8, self.v, self.cuq, self.cuk, c.max_seqlen_q,
                           c.softmax_scale, self.f8.descale_q, self.f8.descale_k, c.causal,
                           out=self.out8, lse=self.lse8, workspace=self.ws)

    def check(self):
        from variable_length_flashattention_gb300 import vfa
        if vfa.read_status(self.ws) != 0:
            raise RuntimeError(f"{self.name}: forward device status not OK")
        if self.bwd is not None:
            self.bwd()
            if vfa.read_status(self.bws) != 0:
                raise RuntimeError(f"{self.name}: backward device status not OK")


class DecodeLeg:
    """The paged-decode workload resident in HBM; one pass (init, every tile
    step, finalize) captured as a CUDA graph."""

    def __init__(self, seed, dev):
        import torch
        from variable_length_flashattention_gb300 import accounting as A
        from variable_length_flashattention_gb300 import vfa, workloads as W
        case = W.decode(seed)
        self.case = case
        S, Hq, D = case.num_seqs, case.num_q_heads, case.head_dim
        self.q, self.kp, self.vp = case.q.to(dev), case.k_pool.to(dev), case.v_pool.to(dev)
        self.tiles = []
        for t in range(case.num_steps):
            tb, tc = case.tile(t)
            self.tiles.append((torch.from_numpy(tb).to(dev), torch.from_numpy(tc).to(dev)))
        self.m = torch.empty(S, Hq, device=dev)
        self.l = torch.empty(S, Hq, device=dev)
        self.o = torch.empty(S, Hq, D, device=dev)
        self.out = torch.empty(S, Hq, D, dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.bytes = A.decode_bytes(case)
        self.launches = 2 + len(self.tiles)
        self.run_pass()
        torch.cuda.synchronize()
        if vfa.read_status(self.status) != 0:
            raise RuntimeError("decode device status not OK in warm-up")
        stream = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            self.run_pass()
        stream.wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.run_pass()
        torch.cuda.synchronize()

    def run_pass(self):
        from variable_length_flashattention_gb300 import vfa
        vfa.decode_init(self.m, self.l, self.o, self.status)
        for tb, tc in self.tiles:
            vfa.decode_step(self.q, self.kp, self.vp, tb, tc, self.m, self.l, self.o,
                            self.status)
        vfa.decode_finalize(self.l, self.o, out=self.out)


class DecodeLongLeg:
    """A few long contexts (49k-64k tokens), one tile step each, run as the
    split step (each (sequence, kv head) tile cut into runs over the SMs);
    init, split step and finalize captured as one CUDA graph."""

    def __init__(self, seed, dev):
        import torch
        from variable_length_flashattention_gb300 import accounting as A
        from variable_length_flashattention_gb300 import vfa, workloads as W
        case = W.decode_long(seed)
        self.case = case
        S, Hq, Hkv, D = case.num_seqs, case.num_q_heads, case.num_kv_heads, case.head_dim
        self.q, self.kp, self.vp = case.q.to(dev), case.k_pool.to(dev), case.v_pool.to(dev)
        tb, tc = case.tile(0)
        self.tb, self.tc = torch.from_numpy(tb).to(dev), torch.from_numpy(tc).to(dev)
        self.splits = vfa.decode_split_count(S, Hkv, case.tile_capacity)
        self.ws = vfa.alloc_decode_split_workspace(S, Hq, Hkv, D, self.splits, device=dev)
        self.m = torch.empty(S, Hq, device=dev)
        self.l = torch.empty(S, Hq, device=dev)
        self.o = torch.empty(S, Hq, D, device=dev)
        self.out = torch.empty(S, Hq, D, dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.bytes = A.decode_bytes(case)
        self.launches = 3
        self.run_pass()
        torch.cuda.synchronize()
        if vfa.read_status(self.status) != 0:
            raise RuntimeError("split decode device status not OK in warm-up")
        stream = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            self.run_pass()
        stream.wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.run_pass()
        torch.cuda.synchronize()

    def run_pass(self):
        from variable_length_flashattention_gb300 import vfa
        vfa.decode_init(self.m, self.l, self.o, self.status)
        vfa.decode_step_split(self.q, self.kp, self.vp, self.tb, self.tc, self.m, self.l, self.o,
                              self.splits, self.ws, self.status)
        vfa.decode_finalize(self.l, self.o, out=self.out)


def time_loop(fn, n, flush, stream, warmup=3):
    """CUDA-event times (ms) of n calls of fn, each after an L2 flush."""
    import torch
    for i in range(warmup):
        flush.fill_(float(i))
        fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    torch.cuda.synchronize()
    for i in range(n):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def tensor_roofline(flops, ms, peak, peak_source, traffic, kernel):
    ach = flops / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
            "frac": ach / peak, "traffic": traffic, "kernel": kernel,
            "peak_source": peak_source}


def link_bandwidth(nbytes, dev, reps=5):
    """Pinned host <-> device copy bandwidth (GB/s) over nbytes, one copy per
    direction per repetition (the best of reps), on a stream of its own."""
    import torch
    n = max(1, nbytes // 4)
    h = torch.empty(n, dtype=torch.float32).pin_memory()
    d = torch.empty(n, dtype=torch.float32, device=dev)
    s = torch.cuda.Stream()
    best = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        times = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                a.record(s)
                dst.copy_(src, non_blocking=True)
                b.record(s)
            s.synchronize()
            times.append(a.elapsed_time(b))
        best[name] = 4 * n / (min(times) * 1e-3) / 1e9
    return best


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist
    from variable_length_flashattention_gb300 import build as cuda_build
    from variable_length_flashattention_gb300 import vfa

    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world > 1:
        cuda_build.build()
    if world > 1:
        dist.barrier()
    vfa.lib()
    peaks = _peaks()
    seed = args.seed + rank                   # each replica its own batch
    head_name = args.workload
    names = [head_name] + [w for w in (args.configs.split(",") if args.configs else
                                       PREFILL_CONFIGS) if w and w != head_name]

    # ---------------- inputs (resident in HBM before timing)
    legs = {}
    for w in names:
        legs[w] = PrefillLeg(w, seed, dev, want_bwd=not args.no_backward,
                             want_fp8=not args.no_fp8)
    head = legs[head_name]
    dec = DecodeLeg(seed, dev)
    dlong = None if args.no_decode_long else DecodeLongLeg(seed, dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    if args.profile:
        part = {"prefill": head.fwd, "decode": dec.graph.replay, "backward": head.bwd,
                "fp8": head.fp8,
                "decode-long": dlong.graph.replay if dlong else None}[args.profile]
        if part is None:
            raise SystemExit(f"{args.profile} is not available for {head_name}")
        for i in range(args.warmup + args.steps):
            flush.fill_(float(i))
            part()
        torch.cuda.synchronize()
        print(f"profile run: {args.profile} on {head_name} x {args.warmup + args.steps}",
              flush=True)
        return

    # ---------------- the step: forward on the headline workload + one decode pass
    for i in range(args.warmup):
        flush.fill_(1.0)
        head.fwd()
        flush.fill_(2.0)
        dec.graph.replay()
    torch.cuda.synchronize()
    n_ev = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_ev)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.5)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark("start")
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        head.fwd()
        ev[i][1].record(stream)
        flush.fill_(float(-i))
        ev[i][2].record(stream)
        dec.graph.replay()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t0
    launches = args.steps * (2 + dec.launches)
    pre_ms = _median([e[0].elapsed_time(e[1]) for e in ev])
    dec_ms = _median([e[2].elapsed_time(e[3]) for e in ev])
    if vfa.read_status(head.ws) != 0 or vfa.read_status(dec.status) != 0:
        raise RuntimeError("device status not OK after timing")

    # ---------------- every config's forward, backward and FP8 forward: own timed loops
    n_x = max(5, min(args.steps, 200))
    per = {}
    for w, leg in legs.items():
        r = {}
        if w != head_name:
            r["fwd"] = _median(time_loop(leg.fwd, n_x, flush, stream))
            launches += 2 * n_x
        if leg.bwd is not None:
            r["bwd"] = _median(time_loop(leg.bwd, n_x, flush, stream))
            launches += 4 * n_x
        if leg.fp8 is not None:
            r["fp8"] = _median(time_loop(leg.fp8, n_x, flush, stream))
            launches += 2 * n_x
        leg.check()
        per[w] = r
    if dlong is not None:
        per["decode-long"] = {"pass": _median(time_loop(dlong.graph.replay, n_x, flush, stream))}
        launches += dlong.launches * n_x
        if vfa.read_status(dlong.status) != 0:
            raise RuntimeError("split decode device status not OK after timing")
    torch.cuda.synchronize()
    sampler.mark("stop")
    clocks = sampler.stop()
    per[head_name]["fwd"] = pre_ms
    keys = sorted({(w, p) for w in per for p in per[w]})
    vals = max_over_ranks([per[w][p] for w, p in keys] + [dec_ms], world, dev)
    for (w, p), x in zip(keys, vals):
        per[w][p] = x
    dec_ms = vals[-1]
    pre_ms = per[head_name]["fwd"]

    # ---------------- end to end through the public API with host buffers
    # The headline batch goes through in chunks of whole sequences (each chunk
    # a vfa_varlen_fwd call on its slices with its own rebased cu_seqlens):
    # chunk c + 1's inputs copy in while chunk c computes and chunk c - 1's
    # outputs copy out, on three streams.  Every byte of every input and
    # output crosses the link inside the timed region, every step.
    case = head.case
    out, lse = head.out, head.lse
    h_q, h_k, h_v = case.q.pin_memory(), case.k.pin_memory(), case.v.pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    cq_np, ck_np = case.cu_seqlens_q, case.cu_seqlens_k
    n_chunks = max(1, min(args.e2e_chunks, case.batch))
    tok = (cq_np[1:] - cq_np[:-1]) + (ck_np[1:] - ck_np[:-1])
    bounds, acc, target = [0], 0, tok.sum() / n_chunks
    for b_ in range(case.batch):
        acc += int(tok[b_])
        if acc >= target * len(bounds) and len(bounds) < n_chunks and b_ + 1 < case.batch:
            bounds.append(b_ + 1)
    bounds.append(case.batch)
    chunks = []
    for b0, b1 in zip(bounds[:-1], bounds[1:]):
        q0, q1, k0, k1 = int(cq_np[b0]), int(cq_np[b1]), int(ck_np[b0]), int(ck_np[b1])
        h_cq = torch.from_numpy((cq_np[b0:b1 + 1] - q0).astype(np.int32)).pin_memory()
        h_ck = torch.from_numpy((ck_np[b0:b1 + 1] - k0).astype(np.int32)).pin_memory()
        lens = cq_np[b0 + 1:b1 + 1] - cq_np[b0:b1]
        chunks.append(dict(q=(q0, q1), k=(k0, k1), h_cq=h_cq, h_ck=h_ck,
                           d_cq=torch.empty_like(h_cq, device=dev),
                           d_ck=torch.empty_like(h_ck, device=dev),
                           max_q=int(lens.max()) if len(lens) else 0,
                           ws=vfa.alloc_workspace(b1 - b0, q1 - q0, k1 - k0, case.num_heads,
                                                  case.head_dim, device=dev)))
    # heaviest chunk first (attention work grows with Lq * Lk per sequence): its
    # compute then overlaps the other chunks' copies instead of trailing them
    def chunk_work(ch):
        lq = np.diff(ch["h_cq"].numpy().astype(np.int64))
        lk = np.diff(ch["h_ck"].numpy().astype(np.int64))
        return int((lq * lk).sum())
    chunks.sort(key=chunk_work, reverse=True)
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v)) + \
        sum(c["h_cq"].numel() * 4 + c["h_ck"].numel() * 4 for c in chunks)
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
    e2e_steps = max(5, min(args.steps, 100))
    s_in = [torch.cuda.Stream() for _ in range(args.e2e_copy_streams)]
    s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in s_in] for _ in chunks]
    ev_cmp = [torch.cuda.Event() for _ in chunks]
    d_q, d_k, d_v = head.q, head.k, head.v

    def e2e_step():
        for c, ch in enumerate(chunks):
            (q0, q1), (k0, k1) = ch["q"], ch["k"]
            jobs = [(d_q[q0:q1], h_q[q0:q1]), (d_k[k0:k1], h_k[k0:k1]),
                    (d_v[k0:k1], h_v[k0:k1]), (ch["d_cq"], ch["h_cq"]), (ch["d_ck"], ch["h_ck"])]
            for n_, (dst, src) in enumerate(jobs):
                with torch.cuda.stream(s_in[n_ % len(s_in)]):
                    dst.copy_(src, non_blocking=True)
            for si, st_ in enumerate(s_in):
                ev_in[c][si].record(st_)
        for c, ch in enumerate(chunks):
            (q0, q1), (k0, k1) = ch["q"], ch["k"]
            for e_ in ev_in[c]:
                s_cmp.wait_event(e_)
            vfa.varlen_fwd(d_q[q0:q1], d_k[k0:k1], d_v[k0:k1], ch["d_cq"], ch["d_ck"],
                           ch["max_q"], case.softmax_scale, case.causal, out=out[q0:q1],
                           lse=lse[q0:q1], workspace=ch["ws"], stream=s_cmp)
            ev_cmp[c].record(s_cmp)
        with torch.cuda.stream(s_out):
            for c, ch in enumerate(chunks):
                q0, q1 = ch["q"]
                s_out.wait_event(ev_cmp[c])
                h_out[q0:q1].copy_(out[q0:q1], non_blocking=True)
                h_lse[q0:q1].copy_(lse[q0:q1], non_blocking=True)
        s_out.synchronize()

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if not (torch.equal(h_out.to(dev), out) and torch.equal(h_lse.to(dev), lse)):
        raise RuntimeError("end-to-end outputs differ from the device result")
    if world > 1:
        dist.barrier()
    # each step's host-side time (copies in, compute, copies out, synchronised),
    # reduced by the median like the device-timed legs
    e2e_times = []
    for _ in range(e2e_steps):
        te = time.perf_counter()
        e2e_step()
        e2e_times.append(time.perf_counter() - te)
    e2e_s = _median(e2e_times)
    launches += 2 * len(chunks) * e2e_steps
    e2e_s = max_over_ranks([e2e_s], world, dev)[0]
    link = link_bandwidth(max(h2d, d2h), dev)
    link_ms = 1e3 * max(h2d / (link["h2d"] * 1e9), d2h / (link["d2h"] * 1e9))

    if rank != 0:
        dist.destroy_process_group()
        return

    def prefill_entry(w):
        leg, r = legs[w], per[w]
        c = leg.case
        D = c.head_dim
        e = {"sequences": c.batch, "total_q": c.total_q, "total_k": c.total_k,
             "num_heads": c.num_heads, "head_dim": D, "causal": c.causal,
             "gflop": leg.flops / 1e9}
        f = tensor_roofline(leg.flops, r["fwd"], peaks["bf16_tflops"],
                            peaks["source"] + " bf16 burst", _traffic(f"prefill_d{D}@{w}"),
                            "vfa_varlen_fwd (scheduler + prefill kernel, timed together)")
        f["frac_of_sustained"] = f["achieved"] / peaks["bf16_tflops_sustained"]
        e["forward"] = {"value": world * f["achieved"], "unit": "TFLOP/s", "ms": r["fwd"],
                        "roofline": f}
        if "bwd" in r:
            b = tensor_roofline(leg.bwd_flops, r["bwd"], peaks["bf16_tflops"],
                                peaks["source"] + " bf16 burst", _traffic(f"bwd_d{D}@{w}"),
                                "vfa_varlen_bwd (all its kernels, timed together)")
            e["backward"] = {"value": world * b["achieved"], "unit": "TFLOP/s", "ms": r["bwd"],
                             "gflop": leg.bwd_flops / 1e9, "roofline": b}
        if "fp8" in r:
            # half the FLOPs (S = Q K^T) at the FP8 rate (2x bf16, nominal), half (P V) at bf16
            peak8 = 4.0 * peaks["bf16_tflops"] / 3.0
            f8 = tensor_roofline(leg.flops, r["fp8"], peak8,
                                 peaks["source"] + " bf16 burst x 4/3 (S at the nominal FP8 "
                                 "rate of 2x bf16, P V at bf16)",
                                 _traffic(f"prefill_fp8_d{D}@{w}"),
                                 "vfa_varlen_fwd_fp8 (scheduler + prefill kernel)")
            e["fp8"] = {"value": world * f8["achieved"], "unit": "TFLOP/s", "ms": r["fp8"],
                        "roofline": f8}
        if not args.no_cpu_baseline:
            secs = args.cpu_seconds if w == head_name else min(3.0, args.cpu_seconds)
            rate, threads, nrows, spent = cpu_oracle_rate(c, secs, args.seed)
            e["cpu_baseline"] = {
                "value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                "sample": f"{nrows} random (token, head) rows of the {w} workload "
                          f"({spent:.1f} s, fp64)"}
        return e

    configs = {w: prefill_entry(w) for w in names}
    hc = configs[head_name]
    value = world * head.flops / (pre_ms * 1e-3) / 1e12
    ach_dec = dec.bytes / (dec_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": pre_ms + dec_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": head_name, "seed": args.seed, "sequences": case.batch,
            "total_tokens": case.total_q, "num_heads": case.num_heads,
            "head_dim": case.head_dim, "causal": case.causal,
            "gflop_per_step": head.flops / 1e9,
            "l2": "flushed (256 MiB write) before each timed call",
            "timing": "CUDA events on the launching stream; median over the timed calls",
            "decode_workload": "64 seqs, ctx U{128..8192}, 32q/8kv heads, D=128, bs 16, "
                               f"{len(dec.tiles)} tile steps of 32 blocks, CUDA graph",
            "parallelism": f"replicas x{world}",
        },
        "prefill_ms": pre_ms,
        "roofline": hc["forward"]["roofline"],
        "decode": {
            "value": world * ach_dec, "unit": "GB/s", "ms": dec_ms, "bytes_per_pass": dec.bytes,
            "roofline": {"bound": "hbm", "achieved": ach_dec, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": ach_dec / peaks["hbm_gbs"],
                         "traffic": _traffic("decode_step_d128_g4"),
                         "traffic_unit": "DRAM bytes per step launch (ncu, tile 4)",
                         "kernel": "whole decode pass (init + steps + finalize)",
                         "peak_source": peaks["source"]},
        },
        "configs": configs,
        "e2e": {"value": world * head.flops / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3, "chunks": len(chunks), "copy_streams": len(s_in),
                "link_gbs": link, "link_bound_ms": link_ms, "frac_of_link": link_ms / (e2e_s * 1e3),
                "how": "vfa_varlen_fwd per chunk of sequences, heaviest chunk first; copy-in, "
                       "compute and copy-out overlapped on three streams; pinned host buffers; "
                       "median of the steps' host times (each synchronised); "
                       "link_gbs = one pinned "
                       "cudaMemcpyAsync per direction over the larger byte count (best of 5), "
                       "link_bound_ms = the slower direction's bytes / its bandwidth"},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s": wall,
    }
    if dlong is not None:
        ms = per["decode-long"]["pass"]
        ach = dlong.bytes / (ms * 1e-3) / 1e9
        c = dlong.case
        line["decode_long"] = {
            "value": world * ach, "unit": "GB/s", "ms": ms, "bytes_per_pass": dlong.bytes,
            "sequences": c.num_seqs, "contexts": c.context_lengths, "num_splits": dlong.splits,
            "how": "init + one split tile step (every block of each context, cut into "
                   "num_splits runs per (sequence, kv head)) + finalize, one CUDA graph",
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                         "traffic": _traffic("decode_step_split_d128_g4@decode-long"),
                         "kernel": "whole pass (init + split step + finalize)",
                         "peak_source": peaks["source"]},
        }
    for part in ("backward", "fp8"):
        if part in hc:
            line[part] = hc[part]
    if "cpu_baseline" in hc:
        line["cpu_baseline"] = hc["cpu_baseline"]
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="longtail", choices=list(PREFILL_CONFIGS))
    ap.add_argument("--configs", default=None,
                    help="comma-separated prefill workloads to time besides the headline "
                         "(default: all)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward's timed loops")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the FP8 q / k forward's timed loops")
    ap.add_argument("--profile", choices=["prefill", "decode", "backward", "fp8", "decode-long"],
                    default=None,
                    help="run only W + K passes of one part of the headline workload (for ncu "
                         "captures); no JSON line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode-long", action="store_true",
                    help="skip the long-context split decode leg")
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="sequence chunks the end-to-end leg pipelines through (1 = no overlap)")
    ap.add_argument("--e2e-copy-streams", type=int, default=1,
                    help="host-to-device copy streams of the end-to-end leg")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
