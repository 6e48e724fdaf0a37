"""Benchmark: varlen attention forward TFLOP/s and paged GQA decode HBM GB/s on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload packed|longtail|cross-d64|cross-d256|tiny]

One step is one pass of the whole hot path on one batch of synthetic input:
the varlen forward (device tile scheduler + prefill kernel) over the packed
training batch (16 sequences, lengths U{1..2048}, H=16, D=128, causal), then
a full paged-decode pass (init, every 32-block tile step, finalize) over the
decode workload (64 sequences, context U{128..8192}, 32 q / 8 kv heads,
D=128, block size 16), captured as one CUDA graph.  `value` is the forward's
algorithmic TFLOP/s (4 * H * D * attended pairs); the decode half is
reported under "decode" in GB/s of algorithmic bytes, and the varlen backward
(vfa_varlen_bwd on the same batch) under "backward", timed in its own loop
outside the step.  L2 is flushed (a
256 MiB write) before each timed part; device time comes from CUDA events
on the launching stream.  Under torchrun each rank runs its own replica
(the path has no exchange step), so scaling is weak.

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
    rows_per_step = max(1, int(budget * rate * 1e12 / max(1, 4 * case.head_dim * 1024)))
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


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist
    from variable_length_flashattention_gb300 import accounting as A
    from variable_length_flashattention_gb300 import build as cuda_build
    from variable_length_flashattention_gb300 import vfa, workloads as W

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

    # ---------------- inputs (resident in HBM before timing)
    case = W.VARLEN_WORKLOADS[args.workload](args.seed + rank)
    d_q, d_k, d_v = case.q.to(dev), case.k.to(dev), case.v.to(dev)
    d_cuq = torch.from_numpy(case.cu_seqlens_q).to(dev)
    d_cuk = torch.from_numpy(case.cu_seqlens_k).to(dev)
    out = torch.empty_like(d_q)
    lse = torch.empty(case.total_q, case.num_heads, dtype=torch.float32, device=dev)
    ws = vfa.alloc_workspace(case.batch, case.total_q, case.total_k, case.num_heads,
                             case.head_dim, device=dev)
    flops = A.varlen_flops(case)

    dcase = W.decode(args.seed + rank)
    S, Hq, D = dcase.num_seqs, dcase.num_q_heads, dcase.head_dim
    dq, dk, dv = dcase.q.to(dev), dcase.k_pool.to(dev), dcase.v_pool.to(dev)
    tiles = []
    for t in range(dcase.num_steps):
        tb, tc = dcase.tile(t)
        tiles.append((torch.from_numpy(tb).to(dev), torch.from_numpy(tc).to(dev)))
    dm = torch.empty(S, Hq, device=dev)
    dl = torch.empty(S, Hq, device=dev)
    do = torch.empty(S, Hq, D, device=dev)
    dout = torch.empty(S, Hq, D, dtype=torch.bfloat16, device=dev)
    dstatus = torch.zeros(1, dtype=torch.int32, device=dev)
    dbytes = A.decode_bytes(dcase)

    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def prefill():
        vfa.varlen_fwd(d_q, d_k, d_v, d_cuq, d_cuk, case.max_seqlen_q, case.softmax_scale,
                       case.causal, out=out, lse=lse, workspace=ws)

    def decode_pass():
        vfa.decode_init(dm, dl, do, dstatus)
        for tb, tc in tiles:
            vfa.decode_step(dq, dk, dv, tb, tc, dm, dl, do, dstatus)
        vfa.decode_finalize(dl, do, out=dout)

    # warm up once, check status words, then capture the decode pass as a graph
    prefill()
    decode_pass()
    torch.cuda.synchronize()
    if vfa.read_status(ws) != 0 or vfa.read_status(dstatus) != 0:
        raise RuntimeError("device status not OK in warm-up")
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        decode_pass()
    stream.wait_stream(side)
    with torch.cuda.graph(graph):
        decode_pass()
    torch.cuda.synchronize()

    # backward inputs: the forward's out / lse for these q, k, v and a seeded dout
    has_bwd = case.head_dim in (64, 128) and not args.no_backward
    if has_bwd:
        g_out = W.upstream_grad(case, args.seed + rank).to(dev)
        b_dq, b_dk, b_dv = torch.empty_like(d_q), torch.empty_like(d_k), torch.empty_like(d_v)
        b_ws = vfa.alloc_bwd_workspace(case.batch, case.total_q, case.num_heads, case.head_dim,
                                       device=dev)

        def backward():
            vfa.varlen_bwd(d_q, d_k, d_v, out, g_out, lse, d_cuq, d_cuk, case.softmax_scale,
                           case.causal, dq=b_dq, dk=b_dk, dv=b_dv, workspace=b_ws)

        backward()
        torch.cuda.synchronize()
        if vfa.read_status(b_ws) != 0:
            raise RuntimeError("backward device status not OK in warm-up")

    has_fp8 = case.head_dim == 128 and not args.no_fp8
    if has_fp8:
        f8 = W.fp8_qk(case)
        d_q8, d_k8 = f8.q8.to(dev), f8.k8.to(dev)
        out8 = torch.empty_like(d_q)
        lse8 = torch.empty_like(lse)

        def forward_fp8():
            vfa.varlen_fwd_fp8(d_q8, d_k8, d_v, d_cuq, d_cuk, case.max_seqlen_q,
                               case.softmax_scale, f8.descale_q, f8.descale_k, case.causal,
                               out=out8, lse=lse8, workspace=ws)

    launches_per_step = 2 + (2 + len(tiles))
    if args.profile:
        part = {"prefill": prefill, "decode": graph.replay,
                "backward": backward if has_bwd else None,
                "fp8": forward_fp8 if has_fp8 else None}[args.profile]
        for i in range(args.warmup + args.steps):
            flush.fill_(float(i))
            part()
        torch.cuda.synchronize()
        print(f"profile run: {args.profile} x {args.warmup + args.steps}", flush=True)
        return
    n_ev = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_ev)]

    for _ in range(args.warmup):
        flush.fill_(1.0)
        prefill()
        flush.fill_(2.0)
        graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.5)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark("start")
    t0 = time.perf_counter()
    nvtx = torch.cuda.nvtx
    for i in range(args.steps):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        nvtx.range_push("varlen_fwd")
        prefill()
        nvtx.range_pop()
        ev[i][1].record(stream)
        flush.fill_(float(-i))
        ev[i][2].record(stream)
        nvtx.range_push("decode_pass")
        graph.replay()
        nvtx.range_pop()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - t0
    sampler.mark("stop")
    clocks = sampler.stop()
    pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[2].elapsed_time(e[3]) for e in ev]
    if vfa.read_status(ws) != 0 or vfa.read_status(dstatus) != 0:
        raise RuntimeError("device status not OK after timing")
    pre_mean = sum(pre_ms) / len(pre_ms)
    dec_mean = sum(dec_ms) / len(dec_ms)

    # ---------------- FP8 q / k forward: its own timed loop (not part of the step)
    fp8_mean = None
    if has_fp8:
        f_steps = max(5, min(args.steps, 500))
        for _ in range(max(3, args.warmup)):
            flush.fill_(4.0)
            forward_fp8()
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(f_steps)]
        torch.cuda.synchronize()
        for i in range(f_steps):
            flush.fill_(float(i))
            fev[i][0].record(stream)
            forward_fp8()
            fev[i][1].record(stream)
        torch.cuda.synchronize()
        if vfa.read_status(ws) != 0:
            raise RuntimeError("fp8 forward device status not OK after timing")
        fp8_mean = sum(e[0].elapsed_time(e[1]) for e in fev) / f_steps
        fp8_mean = max_over_ranks([fp8_mean], world, dev)[0]

    # ---------------- backward: its own timed loop (not part of the step)
    bwd_mean = None
    if has_bwd:
        b_steps = max(5, min(args.steps, 300))
        for _ in range(max(3, args.warmup)):
            flush.fill_(3.0)
            backward()
        bev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(b_steps)]
        torch.cuda.synchronize()
        for i in range(b_steps):
            flush.fill_(float(i))
            bev[i][0].record(stream)
            backward()
            bev[i][1].record(stream)
        torch.cuda.synchronize()
        if vfa.read_status(b_ws) != 0:
            raise RuntimeError("backward device status not OK after timing")
        bwd_mean = sum(e[0].elapsed_time(e[1]) for e in bev) / b_steps
        bwd_mean = max_over_ranks([bwd_mean], world, dev)[0]
    step_ms = pre_mean + dec_mean
    pre_mean, dec_mean, step_ms = max_over_ranks([pre_mean, dec_mean, step_ms], world, dev)

    # ---------------- end to end through the public API with host buffers
    # The batch goes through in chunks of whole sequences (each chunk a
    # vfa_varlen_fwd call on its slices with its own rebased cu_seqlens): chunk
    # c + 1's inputs copy in while chunk c computes and chunk c - 1's outputs
    # copy out, on three streams.  Every byte of every input and output still
    # crosses the link inside the timed region, every step.
    h_q = case.q.pin_memory()
    h_k = case.k.pin_memory()
    h_v = case.v.pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    cq_np, ck_np = case.cu_seqlens_q, case.cu_seqlens_k
    n_chunks = max(1, min(args.e2e_chunks, case.batch))
    # split sequences into chunks of about equal q + k tokens
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
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v)) + \
        sum(c["h_cq"].numel() * 4 + c["h_ck"].numel() * 4 for c in chunks)
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
    e2e_steps = max(5, min(args.steps, 200))
    # q, k and v of a chunk travel on separate copy streams (several copy engines)
    s_in = [torch.cuda.Stream() for _ in range(args.e2e_copy_streams)]
    s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in s_in] for _ in chunks]
    ev_cmp = [torch.cuda.Event() for _ in chunks]

    def e2e_step():
        torch.cuda.nvtx.range_push("e2e_step")
        for c, ch in zip(range(len(chunks)), chunks):
            (q0, q1), (k0, k1) = ch["q"], ch["k"]
            jobs = [(d_q[q0:q1], h_q[q0:q1]), (d_k[k0:k1], h_k[k0:k1]),
                    (d_v[k0:k1], h_v[k0:k1]), (ch["d_cq"], ch["h_cq"]), (ch["d_ck"], ch["h_ck"])]
            for n_, (dst, src) in enumerate(jobs):
                si = n_ % len(s_in)
                with torch.cuda.stream(s_in[si]):
                    dst.copy_(src, non_blocking=True)
            for si, st_ in enumerate(s_in):
                ev_in[c][si].record(st_)
        for c, ch in zip(range(len(chunks)), chunks):
            (q0, q1), (k0, k1) = ch["q"], ch["k"]
            for e_ in ev_in[c]:
                s_cmp.wait_event(e_)
            vfa.varlen_fwd(d_q[q0:q1], d_k[k0:k1], d_v[k0:k1], ch["d_cq"], ch["d_ck"],
                           ch["max_q"], case.softmax_scale, case.causal, out=out[q0:q1],
                           lse=lse[q0:q1], workspace=ch["ws"], stream=s_cmp)
            ev_cmp[c].record(s_cmp)
        with torch.cuda.stream(s_out):
            for c, ch in zip(range(len(chunks)), chunks):
                q0, q1 = ch["q"]
                s_out.wait_event(ev_cmp[c])
                h_out[q0:q1].copy_(out[q0:q1], non_blocking=True)
                h_lse[q0:q1].copy_(lse[q0:q1], non_blocking=True)
        s_out.synchronize()
        torch.cuda.nvtx.range_pop()

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    if not (torch.equal(h_out.to(dev), out) and torch.equal(h_lse.to(dev), lse)):
        raise RuntimeError("end-to-end outputs differ from the device result")

    if world > 1:
        dist.barrier()
    te = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = (time.perf_counter() - te) / e2e_steps
    e2e_s = max_over_ranks([e2e_s], world, dev)[0]

    if rank != 0:
        dist.destroy_process_group()
        return

    value = world * flops / (pre_mean * 1e-3) / 1e12
    dec_gbs = world * dbytes / (dec_mean * 1e-3) / 1e9
    ach_pre = flops / (pre_mean * 1e-3) / 1e12
    ach_dec = dbytes / (dec_mean * 1e-3) / 1e9
    traffic = _traffic("prefill_d128")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": args.workload, "seed": args.seed, "sequences": case.batch,
            "total_tokens": case.total_q, "num_heads": case.num_heads,
            "head_dim": case.head_dim, "causal": case.causal,
            "gflop_per_step": flops / 1e9, "l2": "flushed (256 MiB write) before each timed part",
            "decode_workload": "64 seqs, ctx U{128..8192}, 32q/8kv heads, D=128, bs 16, "
                               f"{len(tiles)} tile steps of 32 blocks, CUDA graph",
            "parallelism": f"replicas x{world}",
        },
        "prefill_ms": pre_mean,
        "roofline": {
            "bound": "tensor", "achieved": ach_pre, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": ach_pre / peaks["bf16_tflops"], "traffic": traffic,
            "kernel": "vfa_varlen_fwd (scheduler + prefill kernel, timed together)",
            "peak_source": peaks["source"] + " bf16 burst",
            "frac_of_sustained": ach_pre / peaks["bf16_tflops_sustained"],
        },
        "decode": {
            "value": dec_gbs, "unit": "GB/s", "ms": dec_mean, "bytes_per_pass": dbytes,
            "roofline": {"bound": "hbm", "achieved": ach_dec, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": ach_dec / peaks["hbm_gbs"],
                         "traffic": _traffic("decode_step_d128_g4"),
                         "traffic_unit": "DRAM bytes per step launch (ncu, tile 4)",
                         "kernel": "whole decode pass (init + steps + finalize)",
                         "peak_source": peaks["source"]},
        },
        "e2e": {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_s * 1e3, "chunks": len(chunks), "copy_streams": len(s_in),
                "how": "vfa_varlen_fwd per chunk of sequences; copy-in, compute and copy-out "
                       "overlapped on three streams; pinned host buffers"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s": wall,
    }
    if fp8_mean is not None:
        ach_8 = flops / (fp8_mean * 1e-3) / 1e12
        # half the FLOPs (S = Q K^T) at the FP8 rate (2x bf16, nominal), half (P V) at bf16
        peak8 = 4.0 * peaks["bf16_tflops"] / 3.0
        line["fp8"] = {
            "value": world * ach_8, "unit": "TFLOP/s", "ms": fp8_mean, "steps": f_steps,
            "gpu_launches": 2 * f_steps,
            "how": "vfa_varlen_fwd_fp8 on the same batch (q, k as E4M3 codes with a power-of-"
                   "two descale, v bf16); own timed loop with an L2 flush before each call",
            "roofline": {"bound": "tensor", "achieved": ach_8, "peak": peak8, "unit": "TFLOP/s",
                         "frac": ach_8 / peak8, "traffic": _traffic("prefill_fp8_d128"),
                         "kernel": "vfa_varlen_fwd_fp8 (scheduler + prefill kernel)",
                         "peak_source": peaks["source"] + " bf16 burst x 4/3 (S at the nominal "
                                        "FP8 rate of 2x bf16, P V at bf16)"},
        }
    if bwd_mean is not None:
        bflops = A.varlen_bwd_flops(case)
        ach_b = bflops / (bwd_mean * 1e-3) / 1e12
        line["backward"] = {
            "value": world * ach_b, "unit": "TFLOP/s", "ms": bwd_mean,
            "gflop": bflops / 1e9, "steps": b_steps, "gpu_launches": 4 * b_steps,
            "how": "vfa_varlen_bwd on the same batch (its forward's out / lse, seeded dout); "
                   "own timed loop with an L2 flush before each call",
            "roofline": {"bound": "tensor", "achieved": ach_b, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": ach_b / peaks["bf16_tflops"],
                         "traffic": _traffic("bwd_d128"),
                         "traffic_unit": "DRAM bytes per launch of the main kernel (ncu)",
                         "kernel": "vfa_varlen_bwd (prep + Delta + main + dQ kernels, "
                                   "timed together)",
                         "peak_source": peaks["source"] + " bf16 burst"},
        }
    if not args.no_cpu_baseline:
        rate, threads, nrows, secs = cpu_oracle_rate(case, args.cpu_seconds, args.seed)
        line["cpu_baseline"] = {
            "value": rate, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{nrows} random (token, head) rows of the {args.workload} workload "
                      f"({secs:.1f} s, fp64)"}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="packed",
                    choices=["packed", "longtail", "cross-d64", "cross-d256", "tiny",
                             "tiny-causal"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward's timed loop")
    ap.add_argument("--no-fp8", action="store_true",
                    help="skip the FP8 q / k forward's timed loop")
    ap.add_argument("--profile", choices=["prefill", "decode", "backward", "fp8"], default=None,
                    help="run only W + K passes of one part (for ncu captures); no JSON line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=4,
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
