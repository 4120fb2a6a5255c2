"""Benchmark of chunked Gated Delta Rule prefill on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1-5] [--shard]
                    [--impl ours|reference]

One step = one gdn_chunk_prefill call over the whole workload (inputs resident
in HBM).  Prints ONE JSON line (rank 0).  The default workload is the long-context
prefill: 2 sequences x 65536 tokens, 16 q/k heads, 32 v heads, head_dim 128, fp32
state pools, batch_invariant off (the library splits each sequence into chunk
segments, three launches per call).  Without ``--workload`` the line also carries,
under ``also``, the same measurement of that workload with batch_invariant on and of
workloads 3 (16 x 4096, bf16 state) and 5 (mixed lengths, pooled states).

Under torchrun (``--gpus N``) every rank runs its own copy of the workload (weak
scaling); with ``--shard`` the ranks split one batch by sequence
(``sharding.shard_problem``) and ``value`` is that batch's tokens over the slowest
rank's time (strong scaling).

``--impl reference`` times the CPU oracle (fp64 token recurrence on all host
cores) on a bounded sample of the same workload: it is the only comparison arm
this operation has.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gated_delta_rule_24_gb300 import workloads as W  # noqa: E402

METRIC = "GDN prefill tokens/s (all heads) and % of bf16-tensor/HBM roofline, 1xGB300"
HEAD_DIM = 128
CHUNK = 64


def algorithmic_work(p):
    """Algorithmic bytes and flops of one prefill call (chunked-algorithm model).

    bytes: q, k read once per q/k head, v once per v head, output written once,
    g and beta read once (at their dtype), initial state read and final state
    written once per (sequence, head).
    flops: per token and sab head 6 D^2 (three state-sized products) +
    2 C (Dk + Dv) + 2 C Dv (the chunk-local products), plus 4 C Dk per token and
    q/k head for K K^T and Q K^T.
    """
    T, Hqk, Hv, H, N = p.T, p.H_qk, p.H_v, p.H, p.N
    D = HEAD_DIM
    b = 2 * T * Hqk * D * 2 + T * Hv * D * 2 + T * H * D * 2
    b += T * H * (p.g.element_size() if p.g is not None else 0)
    b += T * H * (p.beta.element_size() if p.beta is not None else 0)
    if p.initial_state is not None:
        b += N * H * D * D * p.initial_state.element_size()
    if p.output_final_state:
        b += N * H * D * D * torch.tensor([], dtype=p.state_dtype).element_size()
    f = T * (H * (6 * D * D + 2 * CHUNK * (D + D) + 2 * CHUNK * D) + Hqk * 4 * CHUNK * D)
    return b, f


def planned_splits(p, sms: int) -> int:
    """Segments per sequence that the library's split-K planner picks for this call (its
    host-only plan query; only used to count launches)."""
    if p.batch_invariant or p.N == 0:
        return 1
    import gated_delta_rule_24_gb300 as gdn
    return gdn.testing_split_plan(p.N, p.H, p.T, sms)["P"]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def recorded_traffic(kernel: str, workload: str, source: str = "prefill.cu"):
    """Bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source (matched by hash); else None."""
    src = os.path.join(ROOT, "gated_delta_rule_24_gb300", "csrc", source)
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        text = open(os.path.join(ROOT, "profiles", "traffic.md")).read()
    except OSError:
        return None
    for line in text.splitlines():
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == kernel and cells[1] == workload and cells[2] == digest:
            try:
                return float(cells[3])
            except ValueError:
                return None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.dev = device_index
        self.window = None

    def start(self):
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(self.dev)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = []
        for ts, line in self.samples:
            if self.window and not (self.window[0] - 0.15 <= ts <= self.window[1] + 0.15):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[2:]))
            except ValueError:
                continue
        if not rows:
            rows = []
            for _, line in self.samples[-5:]:
                parts = [x.strip() for x in line.split(",")]
                try:
                    rows.append((float(parts[0]), float(parts[1]), parts[2:]))
                except (ValueError, IndexError):
                    pass
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4)
                          if len(r) > i + 1 and r[i + 1].lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


L2_BYTES = 129 << 20
FLUSH_BYTES = 256 << 20


def needs_flush(p) -> bool:
    """Workloads whose algorithmic bytes do not exceed twice the L2 get an L2 flush
    between timed launches (a 256 MB buffer written on the launch stream)."""
    return algorithmic_work(p)[0] < 2 * L2_BYTES


def config_of(p, workload: int, gpus: int, shard: bool = False):
    l2 = ("flushed: a 256 MB buffer is written between timed launches, which are timed one by one"
          if needs_flush(p) else
          f"no flush: each step streams {algorithmic_work(p)[0] / 1e6:.0f} MB, more than twice the 129 MB L2")
    par = (f"sequence shards x{gpus} (one batch split by sequence across ranks, token-balanced; no "
           f"collective)" if shard else
           f"replicas x{gpus} (independent problems per GPU, no collective)")
    return {"workload": p.name, "description": W.WORKLOADS[workload], "tokens": p.T, "num_seqs": p.N,
            "H_qk": p.H_qk, "H_v": p.H_v, "num_sab_heads": p.H, "head_dim": HEAD_DIM, "chunk": CHUNK,
            "state_dtype": str(p.state_dtype).replace("torch.", ""),
            "batch_invariant": bool(p.batch_invariant), "use_qk_l2norm": bool(p.use_qk_l2norm),
            "l2": l2, "parallelism": par}


def oracle_sample(p, n_units, seed=0):
    """Time the oracle on ``n_units`` (sequence, head) units of ``p``; returns
    (tokens/s all heads, seconds, token-heads, threads)."""
    import random

    import oracle
    rng = random.Random(seed)
    all_units = [(n, h) for n in range(p.N) for h in range(p.H)]
    units = rng.sample(all_units, min(n_units, len(all_units)))
    U = oracle.Units(p.q, p.k, p.v, p.g, p.beta, p.initial_state, p.state_indices, p.cu_seqlens, units)
    threads = os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.recurrence_units(U, p.scale, p.use_qk_l2norm, nthreads=threads)
    dt = time.perf_counter() - t0
    token_heads = int(U.len.sum())
    return token_heads / p.H / dt, dt, token_heads, threads


def chunked_sample(p, n_units, seed=0):
    """The oracle's chunked (WY/UT) numpy form timed on ``n_units`` random units: a
    second, blocked CPU baseline beside the token recurrence."""
    import random

    from oracle.chunked import chunked as oracle_chunked
    rng = random.Random(seed)
    units = rng.sample([(n, h) for n in range(p.N) for h in range(p.H)], min(n_units, p.N * p.H))
    t0 = time.perf_counter()
    oracle_chunked(p.q, p.k, p.v, p.g, p.beta, p.scale, p.initial_state, p.state_indices,
                           p.cu_seqlens, p.use_qk_l2norm, units=units)
    dt = time.perf_counter() - t0
    cu = p.cu_seqlens.tolist()
    th = sum(cu[n + 1] - cu[n] for n, _ in units)
    return {"value": th / p.H / dt, "unit": "tokens/s", "cores": "one process (numpy's own BLAS threads)",
            "kind": "oracle, chunked form (numpy fp64)",
            "sample": f"{len(units)} random (sequence, head) units ({th} token-heads), {dt:.1f} s wall"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    p = W.make_workload(args.workload, seqs=args.seqs)
    # (sequence, head) units per step: about 256 K token-heads (a fraction of a second of
    # the oracle on the host cores), at least one unit
    per_unit = max(1, p.T // max(p.N, 1))
    units = args.ref_units if args.ref_units > 0 else max(1, min(64, (1 << 18) // per_unit, p.N * p.H))
    for _ in range(args.warmup):
        oracle_sample(p, max(1, units // 4), seed=1)
    vals, times = [], []
    tot_th, tot_t = 0, 0.0
    for s in range(args.steps):
        v, dt, th, threads = oracle_sample(p, units, seed=100 + s)
        vals.append(v)
        times.append(dt)
        tot_th += th
        tot_t += dt
    value = tot_th / p.H / tot_t
    sample = (f"{units} random (sequence, head) units of the workload per step "
              f"({units * (p.T // max(p.N, 1))} token-heads), fp64 token recurrence")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(p, args.workload, args.gpus),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def measure_prefill(p, workload: int, args, dev, pg, ws: int, rank: int, steps: int, cpu: bool,
                    global_tokens=None, shard: bool = False):
    """Time gdn_chunk_prefill on problem ``p`` (this rank's part): ``steps`` launches with
    inputs resident in HBM, then the same call end to end from pinned host buffers.
    Returns the measured fields of a bench line (rank 0), or None on other ranks."""
    import gated_delta_rule_24_gb300 as gdn

    pd = p.to(dev)
    out = torch.empty(p.T, p.H, HEAD_DIM, dtype=p.q.dtype, device=dev)
    st = torch.zeros(p.state_slots, p.H, HEAD_DIM, HEAD_DIM, dtype=p.state_dtype, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(s=stream):
        gdn.gdn_chunk_prefill(pd.q, pd.k, pd.v, pd.g, pd.beta, p.scale, pd.initial_state, pd.state_indices,
                              st, pd.cu_seqlens, p.use_qk_l2norm, p.batch_invariant, out, s)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    assert gdn.device_status(stream) == 0

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start_all = torch.cuda.Event(enable_timing=True)
    end_all = torch.cuda.Event(enable_timing=True)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if needs_flush(p) else None
    start_all.record(stream)
    for i in range(steps):
        if flush is not None:
            with torch.cuda.stream(stream):
                flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    end_all.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if pg:
        pg.barrier()
    sampler.mark(t_wall0, t_wall1)
    clocks = sampler.stop()
    total_ms = start_all.elapsed_time(end_all)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if flush is not None:  # the flushes are not the workload's time
        total_ms = sum(launch_ms)
    assert gdn.device_status(stream) == 0
    if pg:
        t = torch.tensor([total_ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / steps
    tokens = global_tokens if global_tokens is not None else ws * p.T

    # ---- end to end through the C ABI with host buffers (copies inside the timed region).
    # Every step copies its inputs in from pinned host memory and its output and final
    # states back; the copies of one step overlap the compute of its neighbours (three
    # streams, two device buffer sets), as a serving loop would run them.
    pin = {k: (None if getattr(p, k) is None else getattr(p, k).pin_memory())
           for k in ("q", "k", "v", "g", "beta", "initial_state", "state_indices", "cu_seqlens")}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    st_h = torch.empty(st.shape, dtype=st.dtype).pin_memory()
    dbuf = [{k: (None if v is None else torch.empty(v.shape, dtype=v.dtype, device=dev)) for k, v in pin.items()}
            for _ in range(2)]
    outs = [(torch.empty_like(out), torch.empty_like(st)) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pin.values() if v is not None)
    d2h = out_h.numel() * out_h.element_size() + st_h.numel() * st_h.element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        b = i & 1
        db, (ob, sb) = dbuf[b], outs[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[b])  # step i - 2 has read these inputs
            for k, v in pin.items():
                if v is not None:
                    db[k].copy_(v, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # step i - 2's results have been copied out
        gdn.gdn_chunk_prefill(db["q"], db["k"], db["v"], db["g"], db["beta"], p.scale, db["initial_state"],
                              db["state_indices"], sb, db["cu_seqlens"], p.use_qk_l2norm, p.batch_invariant, ob,
                              stream)
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            out_h.copy_(ob, non_blocking=True)
            st_h.copy_(sb, non_blocking=True)
            ev_out[b].record(s_out)

    e2e_steps = max(3, min(steps, 10))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if pg:
        t = torch.tensor([e2e_ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        e2e_ms = float(t.item())
    del dbuf, outs, pd, out, st
    if rank != 0:
        return None

    P = planned_splits(p, torch.cuda.get_device_properties(dev).multi_processor_count)
    launches = 1 if P == 1 else 3  # split-K: pass 1, fix-up, pass 2
    hbm, tflops, tflops_sus, peak_src = measured_peaks()
    B, F = algorithmic_work(p)
    avg_launch_s = statistics.mean(launch_ms) / 1000.0
    achieved_gbs = B / avg_launch_s / 1e9
    kernel = "gdn_prefill_kernel" if P == 1 else "gdn_prefill_kernel x2 + gdn_split_fixup_kernel (split-K)"
    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                "frac": achieved_gbs / hbm,
                "traffic": recorded_traffic("gdn_prefill_kernel", p.name if P == 1 else f"{p.name}_split{P}"),
                "peak_source": peak_src, "kernel": kernel, "timed": "whole call per step (CUDA events)",
                "algorithmic_bytes_per_launch": B, "algorithmic_flops_per_launch": F,
                "tensor_tflops": F / avg_launch_s / 1e12, "tensor_frac": F / avg_launch_s / 1e12 / tflops,
                "launch_ms_avg": avg_launch_s * 1000, "launch_ms_median": statistics.median(launch_ms),
                "launch_ms_p20": statistics.quantiles(launch_ms, n=5)[0] if len(launch_ms) > 1 else launch_ms[0],
                "launch_ms_p80": statistics.quantiles(launch_ms, n=5)[3] if len(launch_ms) > 1 else launch_ms[0],
                "split_k_segments": P}
    cpu_line = None
    if cpu:
        try:
            n_cpu = args.cpu_units if args.cpu_units > 0 else p.N * p.H
            v, dt, th, threads = oracle_sample(p, n_cpu, seed=7)
            what = ("every (sequence, head) unit" if n_cpu >= p.N * p.H
                    else f"{n_cpu} random (sequence, head) units")
            cpu_line = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                        "sample": f"{what} ({th} token-heads) of the workload, fp64 token recurrence, "
                                  f"{dt:.1f} s wall"}
        except Exception as e:  # the GPU number stands without it
            cpu_line = {"value": None, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                        "sample": f"failed: {e}"}
    return {"value": tokens / (ms_per_step / 1000.0), "unit": "tokens/s", "steps": steps,
            "ms_per_step": ms_per_step, "config": config_of(p, workload, ws, shard), "clocks": clocks,
            "e2e": {"value": tokens / (e2e_ms / 1000.0), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": steps * launches, "roofline": roofline, "cpu_baseline": cpu_line}


# Extra workloads measured beside the headline one (same JSON line, key "also"): the
# headline's other batch_invariant setting and the other full-size workloads.
EXTRAS = [("w4_batch_invariant", 4, True), ("w3", 3, None), ("w5", 5, None)]


def run_ours(args):
    from gated_delta_rule_24_gb300 import build
    from gated_delta_rule_24_gb300.sharding import shard_problem
    import gated_delta_rule_24_gb300 as gdn

    ws, rank, local = dist_env()
    pg = None
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    build.build()
    gdn.gdn_init(dev.index)

    p = W.make_workload(args.workload, seqs=args.seqs)
    if args.batch_invariant is not None:
        p.batch_invariant = bool(args.batch_invariant)
    global_tokens = None
    whole = p
    if args.shard:  # strong scaling: one batch split by sequence across the ranks
        global_tokens = p.T
        _, p = shard_problem(p, ws, rank)
    res = measure_prefill(p, args.workload, args, dev, pg, ws, rank, args.steps, not args.no_cpu_baseline,
                          global_tokens=global_tokens, shard=args.shard)
    if res is not None and args.shard:
        res["config"].update(workload=whole.name, tokens=whole.T, num_seqs=whole.N,
                             rank0_shard={"tokens": p.T, "num_seqs": p.N})
    also = {}
    if args.extras and not args.shard:
        for key, wl, bi in EXTRAS:
            q = W.make_workload(wl)
            if bi is not None:
                q.batch_invariant = bi
            r = measure_prefill(q, wl, args, dev, pg, ws, rank, min(args.steps, 50), not args.no_cpu_baseline)
            if r is not None:
                also[key] = r
    if rank != 0:
        pg.destroy_process_group()
        return 0
    line = {"metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["ms_per_step"], "higher_is_better": True,
            "scaling": "strong" if args.shard else "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": res["config"], "clocks": res["clocks"], "e2e": res["e2e"],
            "gpu_launches": res["gpu_launches"], "roofline": res["roofline"], "cpu_baseline": res["cpu_baseline"]}
    if not args.no_cpu_baseline:
        try:  # the blocked numpy form on about 8k token-heads (one unit for long sequences)
            line["cpu_baseline_chunked"] = chunked_sample(p, max(1, 8192 * p.N // max(p.T, 1)), seed=7)
        except Exception as e:
            line["cpu_baseline_chunked"] = {"value": None, "kind": "oracle, chunked form", "sample": f"failed: {e}"}
    if also:
        line["also"] = also
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


DECODE_METRIC = "GDN decode tokens/s (one token per sequence, all heads) and % of HBM roofline, 1xGB300"


def decode_bytes(p):
    """Algorithmic bytes of one decode step: every addressed state read and written once,
    q/k per q/k head, v per v head, output, gates and state indices once."""
    D = HEAD_DIM
    es = torch.tensor([], dtype=p.state_dtype).element_size()
    b = 2 * p.N * p.H * D * D * es
    b += p.N * (2 * p.H_qk + p.H_v + p.H) * D * 2
    b += p.N * p.H * (p.g.element_size() + p.beta.element_size())
    b += p.N * p.state_indices.element_size()
    return b


def run_decode(args):
    """One step = one gdn_decode_step over the decode batch that follows workload 5
    (1024 sequences, one token each, 8/16 heads, 4096-slot bf16 pool)."""
    import gated_delta_rule_24_gb300 as gdn
    from gated_delta_rule_24_gb300 import build

    ws, rank, local = dist_env()
    pg = None
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        pg = dist
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    build.build()
    gdn.gdn_init(dev.index)
    p = W.make_decode_workload(device=dev)
    pool = p.initial_state  # the state cache, updated in place every step
    out = torch.empty(p.T, p.H, HEAD_DIM, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(q=p.q, k=p.k, v=p.v, g=p.g, beta=p.beta, idx=p.state_indices):
        gdn.gdn_decode_step(q, k, v, g, beta, p.scale, pool, idx, p.use_qk_l2norm, out, stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    assert gdn.device_status(stream) == 0
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    stream.synchronize()
    t_wall1 = time.time()
    if pg:
        pg.barrier()
    sampler.mark(t_wall0, t_wall1)
    clocks = sampler.stop()
    assert gdn.device_status(stream) == 0
    ms = e0.elapsed_time(e1) / args.steps
    if pg:
        t = torch.tensor([ms], device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t.item())

    # end to end: this step's q/k/v/g/beta/indices from pinned host memory, the output back;
    # the state pool is the device-resident cache the step updates.  The copies of one step
    # overlap the compute of its neighbours (three streams, two device buffer sets).
    pin = {n: getattr(p, n).cpu().pin_memory() for n in ("q", "k", "v", "g", "beta", "state_indices")}
    dbuf = [{n: torch.empty_like(t, device=dev) for n, t in pin.items()} for _ in range(2)]
    outs = [torch.empty_like(out) for _ in range(2)]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = out_h.numel() * out_h.element_size()
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        bb = i & 1
        db = dbuf[bb]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[bb])
            for n, t in pin.items():
                db[n].copy_(t, non_blocking=True)
            ev_in[bb].record(s_in)
        stream.wait_event(ev_in[bb])
        if i >= 2:
            stream.wait_event(ev_out[bb])
        gdn.gdn_decode_step(db["q"], db["k"], db["v"], db["g"], db["beta"], p.scale, pool, db["state_indices"],
                            p.use_qk_l2norm, outs[bb], stream)
        ev_comp[bb].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[bb])
            out_h.copy_(outs[bb], non_blocking=True)
            ev_out[bb].record(s_out)

    n_e2e = max(3, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for i in range(n_e2e):
        e2e_step(i)
    b.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = a.elapsed_time(b) / n_e2e
    if rank != 0:
        pg.destroy_process_group()
        return 0
    hbm, _, _, peak_src = measured_peaks()
    B = decode_bytes(p)
    achieved = B / (ms / 1000.0) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": recorded_traffic("gdn_decode_kernel", p.name, "decode.cu"),
                "peak_source": peak_src, "kernel": "gdn_decode_kernel",
                "algorithmic_bytes_per_launch": B, "launch_ms_avg": ms}
    cpu = None
    if not args.no_cpu_baseline:
        v, dt, th, threads = oracle_sample(p.to("cpu"), p.N * p.H, seed=7)
        cpu = {"value": v, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"the whole decode batch ({p.N * p.H} (sequence, head) units), fp64 token "
                         f"recurrence, {dt:.2f} s wall"}
    line = {"metric": DECODE_METRIC, "value": ws * p.N / (ms / 1000.0), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": p.name, "description": "decode step after workload 5: 1024 sequences x 1 "
                       "token, 8 q/k heads, 16 v heads, bf16 state pool [4096, 16, 128, 128] through int32 "
                       "state_indices, updated in place", "num_seqs": p.N, "H_qk": p.H_qk, "H_v": p.H_v,
                       "num_sab_heads": p.H, "head_dim": HEAD_DIM, "state_dtype": "bfloat16",
                       "l2": "no flush: each step reads and writes 1 GB of state, 8x the 129 MB L2",
                       "parallelism": f"replicas x{ws} (independent problems per GPU, no collective)"},
            "clocks": clocks, "e2e": {"value": ws * p.N / (e2e_ms / 1000.0), "unit": "tokens/s",
                                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps, "roofline": roofline, "cpu_baseline": cpu}
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=None, choices=[1, 2, 3, 4, 5],
                    help="the workload (default: 4, with the others as extra keys)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch-invariant", type=int, default=None)
    ap.add_argument("--ref-units", type=int, default=0,
                    help="(sequence, head) units per oracle step of --impl reference (0: about 256 K token-heads)")
    ap.add_argument("--cpu-units", type=int, default=0,
                    help="units of the cpu_baseline sample (0: every unit of the workload)")
    ap.add_argument("--seqs", type=int, default=None,
                    help="truncate the workload to this many sequences (small profiling cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode", action="store_true",
                    help="time the decode step (one token per sequence) instead of the prefill")
    ap.add_argument("--shard", action="store_true",
                    help="under torchrun: split one batch of the workload by sequence across the ranks "
                         "(strong scaling) instead of one copy per rank")
    ap.add_argument("--no-extras", action="store_true",
                    help="only the headline workload (no 'also' keys)")
    args = ap.parse_args(argv)
    args.extras = args.workload is None and not args.no_extras and not args.decode
    if args.workload is None:
        args.workload = 4
    if args.warmup < 3:
        args.warmup = 3
    return args


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.decode:
        return run_decode(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
