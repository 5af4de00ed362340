"""Benchmark of the co-batched layer step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload l8b]
                    [--impl cf|reference] [--decode-sms N] [--sweep-decode-sms]

Prints ONE JSON line (rank 0).  A step is one cf_layer_step over the
workload's synthetic batch (all of: RMSNorm, fused QKV GEMM with RoPE and
paged append, the decode || prefill attention fork, O-proj, RMSNorm, SwiGLU
FFN).  `value` is stacked tokens per second (T rows per step) with inputs
resident in HBM; `e2e` times the same step through host (pinned) buffers
with the per-step host->device copies of x and of the batch metadata and the
device->host copy of the output inside the timed region (on their own
streams, double-buffered: a step's copies overlap its neighbours' compute,
as a serving loop would run them).  N > 1 runs N
independent replicas (one per GPU, no collective in the data path) and
reports the total over ranks divided by the slowest rank's time.

--impl reference times the CPU fp64 oracle (the only reference arm: no other
implementation of this method exists) on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "co-batched layer step µs & tokens/s; decode attn % HBM peak; GEMM % BF16 peak"

# DRAM bytes (read + write) per launch of each workload's roofline kernel,
# from one ncu capture of that kernel build at that shape (the summary named
# in "source"); an entry is removed whenever its kernel changes.
DOMINANT_TRAFFIC = {
    ("q32b", "prefill"): {"bytes": 351844608 + 93404160, "source": "profiles/prefill_attn_q32b_4096on28672.md"},
}

# The kernels of a step that a roofline can name: phase of the engine's
# per-phase timers, bound, and what the roofline object calls it.
ROOFLINE_KERNELS = {
    "qkv": ("tensor", "fused QKV GEMM + QK-norm/RoPE/KV-append epilogue"),
    "oproj": ("tensor", "O-proj GEMM + residual"),
    "gateup": ("tensor", "gate/up GEMM + SwiGLU epilogue"),
    "down": ("tensor", "down GEMM + residual"),
    "decode": ("hbm", "split-K decode attention over paged KV"),
    "prefill": ("tensor", "causal chunked-prefill attention (tcgen05)"),
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ distributed
def dist_setup(gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("CF_BENCH_BACKEND", "nccl")
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return rank, world, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, value: float, device=None) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, value: float, device=None) -> float:
    if pg is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms (a timed region of a
    few tens of steps lasts only a few hundred milliseconds)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._thr = threading.Thread(target=self._read, daemon=True)
            self._thr.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        import statistics
        parsed = []
        for t, line in self.rows:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                parsed.append((t, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [p for p in parsed if self.t0 and self.t1 and self.t0 <= p[0] <= self.t1]
        use = inside if inside else parsed
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i, v in enumerate(p[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(p[1] for p in use), "sm_max_mhz": max(p[2] for p in use),
                "reasons": reasons, "samples": len(use), "in_timed_region": bool(inside)}


# ------------------------------------------------------------------ work accounting
def work_of(w, b):
    """Algorithmic FLOPs / bytes of one step (what the roofline fractions use)."""
    s = w.shape
    T = b.n_tokens
    H, d, Hq, Hkv, F = s.hidden, s.head_dim, s.n_q_heads, s.n_kv_heads, s.ffn_dim
    gemm = {
        "qkv": 2.0 * T * H * s.qkv_dim,
        "oproj": 2.0 * T * Hq * d * H,
        "gateup": 2.0 * T * H * 2 * F,
        "down": 2.0 * T * F * H,
    }
    weights = {"qkv": 2.0 * s.qkv_dim * H, "oproj": 2.0 * H * Hq * d, "gateup": 4.0 * F * H, "down": 2.0 * H * F}
    keys = sum(int(c) + 1 for c in b.dec_ctx)
    dec_bytes = keys * Hkv * d * 2 * 2 + b.n_decode * Hq * d * 2 * 2
    pairs = sum(l * cp + l * (l + 1) // 2 for l, cp, _ in b.chunks)
    pre_flops = 4.0 * d * Hq * pairs
    return {"gemm_flops": gemm, "weight_bytes": weights, "decode_bytes": float(dec_bytes),
            "decode_keys": keys, "prefill_flops": pre_flops, "prefill_pairs": pairs}


def s_hidden(w):
    return w.shape.hidden


# ------------------------------------------------------------------ CPU oracle
REFERENCE_BUDGET_S = 90.0


def oracle_sample(w, b, x, weights, kp, vp, rows):
    import numpy as np
    import oracle
    W64 = oracle.LayerWeights64.from_torch({k: v.cpu() for k, v in weights.items()})
    x64 = oracle.to_f64(x)
    t0 = time.perf_counter()
    oracle.layer_step(x64, W64, w.shape, b, kp, vp, rows=rows)
    return time.perf_counter() - t0


def reference_rows(b, frac=1.0):
    """Bounded sample for the CPU oracle: the first 64 rows of the first chunk
    + all decodes, or the leading fraction `frac` of each (at least 8 chunk
    rows, 2 decodes)."""
    l = b.chunks[0][0] if b.chunks else 0
    P, nd = b.prefill_rows, b.n_decode
    nc = min(l, max(min(8, l), int(round(64 * frac))))
    ndec = min(nd, max(min(2, nd), int(round(nd * frac))))
    return list(range(nc)) + list(range(P, P + ndec))


def workload_config(w, b, world):
    """The `config` object both arms report."""
    return {"workload": f"{w.name}: {w.description}", "tokens_per_step": b.n_tokens, "n_decode": b.n_decode,
            "prefill_len": b.prefill_rows, "prefill_prefix": b.prefill_prefix,
            "chunks": [[int(l), int(c)] for l, c, _ in b.chunks],
            "decode_keys": int(sum(int(c) + 1 for c in b.dec_ctx)), "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (weights + KV > 129 MB), no flush"}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        return max((i.get("num_threads", 0) for i in info), default=os.cpu_count())
    except Exception:
        return os.cpu_count()


# ------------------------------------------------------------------ main arm
def run_cf(args, rank, world, local, pg):
    import numpy as np
    import torch

    import co_prefill_decode_gb300 as cf
    import workload as wl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = wl.WORKLOADS[args.workload]
    b = wl.make_batch(w, args.seed)
    x = wl.make_x(w, b, args.seed, "cuda")
    W = wl.make_weights(w, args.seed, "cuda", unit_gains=True)
    kp, vp = wl.make_pools(w, b, args.seed, "cuda")
    T = b.n_tokens
    eng = cf.Engine(cf.make_config(w.shape, T, max(b.n_decode, 1), args.decode_sms), W)
    eng.cf_set_graphs(args.graphs)   # piecewise CUDA graphs of the linear segments
    eng.cf_set_prefill_pairing(args.prefill_pairing)
    eng.cf_set_prefill_split(args.prefill_split)
    eng.cf_set_split_k(args.split_k)
    dec_ctx = torch.as_tensor(b.dec_ctx, device=dev)
    dec_pages = torch.as_tensor(b.dec_pages, device=dev)
    if len(b.chunks) > 1:   # several prefill chunks: the chunk-list form of the batch
        lens, prefixes, table = b.chunk_table()
        pre_pages = torch.as_tensor(table, device=dev)
        batch = cf.batch_of(b.n_decode, dec_ctx, dec_pages, 0, 0, None, chunks=(lens, prefixes, pre_pages))
    else:
        pre_pages = torch.as_tensor(b.pre_pages if len(b.pre_pages) else np.zeros(1, np.int32), device=dev)
        batch = cf.batch_of(b.n_decode, dec_ctx, dec_pages, b.prefill_len, b.prefill_prefix, pre_pages)
    pool = cf.pool_of(kp, vp)
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream()

    def step():
        eng.cf_layer_step(batch, x, out, pool, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st, msg = eng.cf_get_error()
    if st != 0:
        raise RuntimeError(msg)
    calib = None
    if args.decode_sms == 0 and b.n_decode > 0 and b.prefill_rows > 0:
        # ConfluxServe §6.1: decode gets the fewest SMs that keep 90% of its
        # solo bandwidth; the library measured it on the first warm-up step
        calib = {"rule": "min SMs reaching 90% of standalone decode bandwidth (measured by the library on "
                         "the first step of the batch's bucket)", "chosen": eng.cf_engine_decode_sms(),
                 "points": [{"sms": n, "ms": round(t, 4)} for n, t in eng.cf_calibration_points()]}

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.4)
    n_launch0 = eng.cf_launch_count()
    barrier(pg)
    torch.cuda.synchronize()
    clocks.mark("t0")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    clocks.mark("t1")
    launches = eng.cf_launch_count() - n_launch0
    ms_total = ev0.elapsed_time(ev1)
    ms_total = max_over_ranks(pg, ms_total, dev)
    clocks.stop()

    # per-phase breakdown in a separate pass: the engine's own events between
    # the kernels of a step would otherwise sit inside the timed region
    eng.cf_set_profiling(True)
    eng.cf_get_phase_times()   # reset
    for _ in range(min(args.steps, 50)):
        step()
    torch.cuda.synchronize()
    phases, nsteps = eng.cf_get_phase_times()
    eng.cf_set_profiling(False)

    # e2e: host buffers, copies inside the timed region.  Every step copies its
    # input rows and batch metadata from pinned host memory and reads its output
    # back; the copies run on their own streams, double-buffered, so step i's
    # input copy overlaps step i-1 and its output read overlaps step i+1.
    x_host = x.cpu().pin_memory()
    meta_dev0 = (dec_ctx, dec_pages, pre_pages)
    meta_host = [t.cpu().pin_memory() for t in meta_dev0]
    xs = [x, torch.empty_like(x)]
    outs = [out, torch.empty_like(out)]
    out_hosts = [torch.empty(x_host.shape, dtype=x_host.dtype).pin_memory() for _ in range(2)]
    metas = [meta_dev0, tuple(torch.empty_like(t) for t in meta_dev0)]
    if len(b.chunks) > 1:
        batches = [cf.batch_of(b.n_decode, m[0], m[1], 0, 0, None, chunks=(lens, prefixes, m[2])) for m in metas]
    else:
        batches = [cf.batch_of(b.n_decode, m[0], m[1], b.prefill_len, b.prefill_prefix, m[2]) for m in metas]
    h2d = x_host.numel() * 2 + sum(t.numel() * 4 for t in meta_host)
    d2h = out_hosts[0].numel() * 2
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        k = i % 2
        with torch.cuda.stream(s_in):
            if used[k]:
                s_in.wait_event(ev_done[k])   # step i-2 has finished with these buffers
            xs[k].copy_(x_host, non_blocking=True)
            for hsrc, ddst in zip(meta_host, metas[k]):
                ddst.copy_(hsrc, non_blocking=True)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if used[k]:
            stream.wait_event(ev_read[k])     # step i-2's output has been read back
        eng.cf_layer_step(batches[k], xs[k], outs[k], pool, stream)
        ev_done[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[k])
            out_hosts[k].copy_(outs[k], non_blocking=True)
            ev_read[k].record(s_out)
        used[k] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(pg)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    for k in range(2):
        stream.wait_event(ev_read[k])         # the last outputs are back on the host
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(pg)
    e2e_ok = bool(torch.equal(out_hosts[(args.steps - 1) % 2], out.cpu()))   # the read-back is the step's output
    ms_e2e = max_over_ranks(pg, e0.elapsed_time(e1), dev)
    st, msg = eng.cf_get_error()
    if st != 0:
        raise RuntimeError(msg)

    # Serialized execution (ConfluxServe §8.3, Fig. 14a): decode alone on all
    # SMs, then prefill alone on all SMs, same kernels and items.  Its phase
    # times give each path's isolated time; the larger one is the
    # contention-free bound of the fork.
    serial = None
    if b.n_decode > 0 and b.prefill_rows > 0:
        eng.cf_set_fork_mode(1)
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ns = min(args.steps, 50)
        s0.record(stream)
        for _ in range(ns):
            step()
        s1.record(stream)
        torch.cuda.synchronize()
        step_serial_ms = s0.elapsed_time(s1) / ns
        eng.cf_set_profiling(True)
        eng.cf_get_phase_times()
        for _ in range(ns):
            step()
        torch.cuda.synchronize()
        sph, sn = eng.cf_get_phase_times()
        eng.cf_set_profiling(False)
        eng.cf_set_fork_mode(0)
        sp = {k: v / max(sn, 1) for k, v in sph.items()}
        serial = {"step_ms": step_serial_ms, "attention_ms": sp["fork"], "decode_alone_ms": sp["decode"],
                  "prefill_alone_ms": sp["prefill"]}

    peaks = load_peaks()
    wk = work_of(w, b)
    per = {k: v / max(nsteps, 1) for k, v in phases.items()}   # ms per step
    tok_total = sum_over_ranks(pg, float(T * args.steps), dev)
    value = tok_total / (ms_total / 1e3)
    ms_step = ms_total / args.steps
    # per-kernel achieved rates (CUDA events around each phase inside the step)
    kern = {}
    for name, key in (("qkv", "qkv"), ("oproj", "oproj"), ("gateup", "gateup"), ("down", "down")):
        t = per[key] / 1e3
        kern[name] = {"ms": per[key], "tflops": wk["gemm_flops"][name] / t / 1e12 if t > 0 else None}
    t_dec, t_pre = per["decode"] / 1e3, per["prefill"] / 1e3
    kern["decode_attn"] = {"ms": per["decode"], "gbs": wk["decode_bytes"] / t_dec / 1e9 if t_dec > 0 else None,
                           "sms": eng.cf_engine_decode_sms()}
    kern["prefill_attn"] = {"ms": per["prefill"],
                            "tflops": wk["prefill_flops"] / t_pre / 1e12 if t_pre > 0 else None}
    kern["fork"] = {"ms": per["fork"], "to_decode_start_ms": per.get("fork_in"),
                    "decode_end_to_join_ms": per.get("fork_out")}
    fork_cmp = None
    if serial is not None:
        # fork vs serialized execution and the contention-free bound
        bound = max(serial["decode_alone_ms"], serial["prefill_alone_ms"])
        gap = serial["attention_ms"] - bound
        fork_cmp = {"fork_ms": per["fork"], "serial_ms": serial["attention_ms"], "isolated_max_ms": bound,
                    "decode_alone_ms": serial["decode_alone_ms"], "prefill_alone_ms": serial["prefill_alone_ms"],
                    "fork_vs_serial": per["fork"] / serial["attention_ms"],
                    "gap_closed": (serial["attention_ms"] - per["fork"]) / gap if gap > 0 else None,
                    "step_ms_fork": ms_step, "step_ms_serial": serial["step_ms"],
                    "method": "attention region (QKV end to join) between CUDA events, per-phase pass of "
                              f"{min(args.steps, 50)} steps per mode; serial = decode then prefill, each alone on "
                              "all SMs, same kernels and work items"}
        t_dec_iso, t_pre_iso = serial["decode_alone_ms"] / 1e3, serial["prefill_alone_ms"] / 1e3
        kern["decode_attn"]["alone_gbs"] = wk["decode_bytes"] / t_dec_iso / 1e9 if t_dec_iso > 0 else None
        kern["prefill_attn"]["alone_tflops"] = wk["prefill_flops"] / t_pre_iso / 1e12 if t_pre_iso > 0 else None
    kern["rmsnorm"] = {"ms": per["rmsnorm"] + per["rmsnorm2"]}
    gemm_ms = sum(per[k] for k in ("qkv", "oproj", "gateup", "down"))
    gemm_tflops = sum(wk["gemm_flops"].values()) / (gemm_ms / 1e3) / 1e12
    # Kernels are timed inside the step loop at full clocks (see "clocks"), so
    # the fractions use the measured burst bf16 peak (the larger, stricter
    # denominator); the sustained power-capped figure is reported beside it.
    peak_tc = peaks["bf16_tflops"]
    # the roofline kernel: the one with the largest share of the step's time
    # (per-phase CUDA events on the stream each kernel runs on)
    dom_phase = max((k for k in ROOFLINE_KERNELS if per.get(k, 0) > 0), key=lambda k: per[k])
    bound, kname = ROOFLINE_KERNELS[dom_phase]
    t_dom = per[dom_phase] / 1e3
    if bound == "hbm":
        work_dom = wk["decode_bytes"]
        achieved, peak, unit = work_dom / t_dom / 1e9, peaks["hbm_gbs"], "GB/s"
        peak_src = peaks["source"] + " HBM copy bandwidth"
        algo_bytes = work_dom
    else:
        work_dom = wk["prefill_flops"] if dom_phase == "prefill" else wk["gemm_flops"][dom_phase]
        achieved, peak, unit = work_dom / t_dom / 1e12, peak_tc, "TFLOP/s"
        peak_src = peaks["source"] + " burst bf16 (sustained: %.0f)" % peaks["bf16_tflops_sustained"]
        if dom_phase == "prefill":   # each request's K and V read once, Q read and O written
            algo_bytes = sum((c + l) * w.shape.n_kv_heads * w.shape.head_dim * 4 for l, c, _ in b.chunks) + \
                b.prefill_rows * w.shape.n_q_heads * w.shape.head_dim * 4
        else:
            n_out = {"qkv": w.shape.qkv_dim, "oproj": s_hidden(w), "gateup": w.shape.ffn_dim, "down": s_hidden(w)}
            k_in = {"qkv": s_hidden(w), "oproj": w.shape.n_q_heads * w.shape.head_dim, "gateup": s_hidden(w),
                    "down": w.shape.ffn_dim}
            algo_bytes = wk["weight_bytes"][dom_phase] + 2.0 * T * (k_in[dom_phase] + n_out[dom_phase])
    traffic = DOMINANT_TRAFFIC.get((args.workload, dom_phase))
    roofline = {"kernel": kname, "phase": dom_phase, "bound": bound, "achieved": achieved, "peak": peak,
                "unit": unit, "frac": achieved / peak, "share_of_step": per[dom_phase] / max(1e-9, per["step"]),
                "work_per_launch": work_dom, "launch_ms": per[dom_phase],
                "traffic": traffic["bytes"] if traffic else None, "algorithmic_bytes": algo_bytes,
                "peak_source": peak_src, "traffic_source": traffic["source"] if traffic else None,
                "timing": "CUDA events around the kernel on its stream, per-phase pass after the timed region"}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "layer_step_us": ms_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations and KV)",
        "config": dict(workload_config(w, b, world), graphs=bool(args.graphs),
                       prefill_pairing=args.prefill_pairing, prefill_split=args.prefill_split,
                       split_k=args.split_k),
        "decode_attn_hbm_frac": (kern["decode_attn"]["gbs"] or 0) / peaks["hbm_gbs"],
        "gemm_bf16_frac": gemm_tflops / peak_tc,
        "prefill_attn_bf16_frac": (kern["prefill_attn"]["tflops"] or 0) / peak_tc,
        "gemm_tflops": gemm_tflops,
        "fork_vs_serial": fork_cmp["fork_vs_serial"] if fork_cmp else None,
        "fork_vs_serial_detail": fork_cmp,
        "kernels": kern,
        "decode_sms_calibration": calib,
        "roofline": roofline,
        "e2e": {"value": tok_total / (ms_e2e / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "copies": "own streams, double-buffered", "output_read_back_ok": e2e_ok},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
        "peaks": peaks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle as it stands, repeated on its bounded sample for >= 10 s of CPU work
        rows = reference_rows(b)
        secs, reps = 0.0, 0
        while reps < 3 or (secs < 10.0 and reps < 20):
            secs += oracle_sample(w, b, x, W, kp, vp, rows)
            reps += 1
        line["cpu_baseline"] = {"value": len(rows) * reps / secs, "unit": "tokens/s", "cores": blas_threads(),
                                "kind": "oracle", "host_cores": os.cpu_count(),
                                "sample": f"fp64 oracle layer step on {len(rows)} of {T} rows (first 64 rows of the "
                                          f"first chunk + all decodes), {reps} repetitions, {secs:.1f} s"}
    if b.n_decode > 0 and b.prefill_rows > 0 and not args.no_share_sweep:
        # the share the rule picks against the share that minimises the fork
        sw = sweep_decode_sms(eng, step, args, cf, reps=10 if not args.sweep_decode_sms else None)
        best = min(sw, key=lambda r: r["fork"])
        line["decode_share_sweep"] = {"rule_sms": eng.cf_engine_decode_sms(), "rule_fork_ms": per["fork"],
                                      "best_sms": best["decode_sms"], "best_fork_ms": best["fork"],
                                      "points": [{"sms": r["decode_sms"], "frac": r["frac"], "fork_ms": r["fork"]}
                                                 for r in sw]}
    eng.close()
    return line


def sweep_decode_sms(eng, step, args, cf, reps=None):
    """Fork time (per-phase events) at decode shares of 10% .. 50% of the SMs."""
    import torch
    sms = cf.device_sm_count()
    res = []
    for frac in (0.10, 0.15, 0.20, 0.25, 0.30, 0.40, 0.50):
        n = max(1, int(round(sms * frac)))
        eng.cf_set_decode_sms(n)
        for _ in range(3):
            step()
        eng.cf_set_profiling(True)
        eng.cf_get_phase_times()
        for _ in range(reps or max(5, args.steps // 4)):
            step()
        ph, ns = eng.cf_get_phase_times()
        eng.cf_set_profiling(False)
        res.append({"decode_sms": n, "frac": frac, **{k: v / ns for k, v in ph.items()}})
    eng.cf_set_decode_sms(0)
    return res


# ------------------------------------------------------------------ single launches for ncu
def run_kernel_case(args):
    """One small launch of one kernel (plus a warm-up launch), for profilers.

    decode : decode attention, Qwen3-32B shape, 8 requests x 8192 cached keys
             (268 MB of KV, larger than L2)
    prefill: prefill attention, Qwen3-32B shape, 2048-token chunk on 4096 cached
             (8 query-tile pairs x 64 heads: several waves of paired items)
    prefill-long: prefill attention of the Qwen3-32B step, 4096-token chunk on
             28672 cached (1.1 GB of K/V in the pools)
    gemm   : gate/up GEMM + SwiGLU epilogue of the Llama-3.1-8B layer, T = 1040
    prefill-chunks: prefill attention over four chunks of different requests in
             one launch, Llama-3.1-8B shape, (l, c) = (1024, 0), (512, 4096),
             (256, 12288), (128, 2048)
    """
    import numpy as np
    import torch

    import co_prefill_decode_gb300 as cf
    import workload as wl
    which = args.kernel
    s = wl.LLAMA8B if which in ("gemm", "prefill-chunks") else wl.QWEN32B
    if which == "decode":
        w = wl.Workload("k", s, 8, (8192,) * 8, 0, 0)
    elif which == "prefill":
        w = wl.Workload("k", s, 0, (), 2048, 4096)
    elif which == "prefill-long":
        w = wl.Workload("k", s, 0, (), 4096, 28672)
    elif which == "prefill-chunks":
        w = wl.Workload("k", s, 0, (), 1024, 0, more_chunks=((512, 4096), (256, 12288), (128, 2048)))
    else:
        w = wl.Workload("k", s, 0, (), 1040, 0)
    b = wl.make_batch(w, args.seed)
    kp, vp = wl.make_pools(w, b, args.seed, "cuda")
    W = wl.make_weights(wl.Workload("k", s, 1, (1,), 0, 0), args.seed, "cuda", unit_gains=True)
    eng = cf.Engine(cf.make_config(s, 4096, 64), W)
    pool = cf.pool_of(kp, vp)
    Hq, d = s.n_q_heads, s.head_dim
    g = torch.Generator(device="cuda").manual_seed(args.seed)
    if which in ("prefill", "prefill-long", "prefill-chunks"):
        for l, cp, pages in b.chunks:   # each chunk's own K/V
            pos = np.arange(cp, cp + l)
            pg = torch.as_tensor(pages[pos // 16].astype(np.int64), device="cuda")
            off = torch.as_tensor(pos % 16, device="cuda")
            kp[pg, :, off, :] = torch.randn(l, s.n_kv_heads, d, device="cuda", generator=g).bfloat16()
            vp[pg, :, off, :] = torch.randn(l, s.n_kv_heads, d, device="cuda", generator=g).bfloat16()
    for _ in range(2):
        if which == "decode":
            q = torch.randn(b.n_decode, Hq, d, device="cuda", generator=g).bfloat16()
            o = torch.empty_like(q)
            eng.cf_decode_attn(q, Hq * d, pool, b.n_decode, torch.as_tensor(b.dec_ctx, device="cuda"),
                               torch.as_tensor(b.dec_pages, device="cuda"), b.dec_stride, o, Hq * d)
        elif which in ("prefill", "prefill-long"):
            q = torch.randn(b.prefill_len, Hq, d, device="cuda", generator=g).bfloat16()
            o = torch.empty_like(q)
            eng.cf_prefill_attn(q, pool, b.prefill_len, b.prefill_prefix, torch.as_tensor(b.pre_pages, device="cuda"), o)
        elif which == "prefill-chunks":
            lens, prefixes, table = b.chunk_table()
            q = torch.randn(b.prefill_rows, Hq, d, device="cuda", generator=g).bfloat16()
            o = torch.empty_like(q)
            eng.cf_prefill_attn_varlen(q, pool, lens, prefixes, torch.as_tensor(table, device="cuda"), o)
        else:
            A = torch.randn(1040, s.hidden, device="cuda", generator=g).bfloat16()
            C = torch.empty(1040, s.ffn_dim, device="cuda").bfloat16()
            eng.cf_gemm(A, W["w_gate"], C, cf.CF_EPI_SWIGLU, aux=W["w_up"])
    torch.cuda.synchronize()
    st, msg = eng.cf_get_error()
    if st != 0:
        raise RuntimeError(msg)
    return {"kernel_case": which, "ok": True}


# ------------------------------------------------------------------ latency estimator
# Table 4 of ConfluxServe (§8.4), measured on H100: estimator MAPE per model.
PAGES_ESTIMATOR_MAPE = {"l8b": ("Llama-8B", 4.4), "q14b": ("Qwen-14B", 4.8), "q32b": ("Qwen-32B", 4.1)}
LINEAR_PHASES = ("rmsnorm", "qkv", "oproj", "rmsnorm2", "gateup", "down")
# transformer layers of the models whose layer shapes the workloads take
MODEL_LAYERS = {"l8b": 32, "q14b": 40, "q32b": 64}
# ConfluxServe §3.1 (Fig. 3c), H100, Qwen3-14B with 16 decodes at 8K context:
# about 1K prefill tokens fit a 50 ms TBT and about 2.2K fit 100 ms
PAGES_TBT_CHUNK = {"q14b": {50.0: 1000, 100.0: 2200}}
TBT_QUANTUM = 128    # alignment quantum of the level: one GEMM row tile


def run_estimator(args):
    """Fits the iteration-latency estimator of ConfluxServe (§6.2 Eq. 2-6,
    App. D Eq. 7-10) for one layer on this GPU and measures its accuracy the
    way §8.4 does: MAPE over random heterogeneous iterations.

    1. Profiles in isolation (the engine's per-phase CUDA events): the
       shared linear region over a grid of token counts n (f_GEMM), the
       attention region of decode-only iterations against W = sum c_i (f_D)
       and of prefill-only iterations against W = l (c + (l+1)/2) (f_P).
    2. Calibrates alpha, beta on co-batched iterations (whole-step time,
       no profiling events).
    3. Predicts and measures a second, independent set of co-batched
       iterations; reports the MAPE.  One GPU: f_comm = 0, N = 1.
    Every fit, calibration and prediction goes through the library's
    estimator (cf_latency_fit_line / _calibrate / _predict)."""
    import numpy as np
    import torch

    import co_prefill_decode_gb300 as cf
    import workload as wl

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    ps = 16
    t_max = wl.EST_CHUNK[1] + wl.EST_DECODES[1]
    pages_dec = -(-(wl.EST_CONTEXT[1] + 1) // ps)
    pages_pre = -(-(wl.EST_CONTEXT[1] + wl.EST_CHUNK[1]) // ps)
    n_dec_max = wl.EST_DECODES[1]
    num_pages = n_dec_max * pages_dec + pages_pre
    lines = []
    for name in args.estimator.split(","):
        w = wl.WORKLOADS[name]
        s = w.shape
        g = torch.Generator(device=dev).manual_seed(args.seed)
        kp = torch.empty((num_pages, s.n_kv_heads, ps, s.head_dim), dtype=torch.bfloat16, device=dev)
        vp = torch.empty_like(kp)
        for t in (kp, vp):
            t.normal_(generator=g)
        perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(args.seed)).to(torch.int32)
        dec_pages = perm[:n_dec_max * pages_dec].view(n_dec_max, pages_dec).contiguous().to(dev)
        pre_pages = perm[n_dec_max * pages_dec:].contiguous().to(dev)
        x = torch.randn(t_max, s.hidden, generator=g, device=dev).to(torch.bfloat16)
        out = torch.empty_like(x)
        W = wl.make_weights(w, args.seed, "cuda", unit_gains=True)
        eng = cf.Engine(cf.make_config(s, t_max, n_dec_max, args.decode_sms), W)
        pool = cf.pool_of(kp, vp)

        def run(it, reps, profile):
            l, cp, ctx = it
            nd = len(ctx)
            dctx = torch.tensor(list(ctx) or [0], dtype=torch.int32, device=dev)
            b = cf.batch_of(nd, dctx, dec_pages, l, cp, pre_pages)
            T = l + nd
            eng.cf_layer_step(b, x[:T], out[:T], pool, stream)          # warm-up
            if profile:
                eng.cf_set_profiling(True)
                eng.cf_get_phase_times()
                for _ in range(reps):
                    eng.cf_layer_step(b, x[:T], out[:T], pool, stream)
                torch.cuda.synchronize()
                ph, n = eng.cf_get_phase_times()
                eng.cf_set_profiling(False)
                return {k: v / n for k, v in ph.items()}
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(reps)]
            for e0, e1 in evs:
                e0.record(stream)
                eng.cf_layer_step(b, x[:T], out[:T], pool, stream)
                e1.record(stream)
            torch.cuda.synchronize()
            return float(np.median([e0.elapsed_time(e1) for e0, e1 in evs]))

        clocks = ClockSampler(0)
        clocks.start()
        time.sleep(0.3)
        clocks.mark("t0")
        t_start = time.perf_counter()
        # 1. isolated profiles
        grid = sorted({32, 64, 128, 256, 384, 512, 768} | set(range(1024, t_max, 512)) | {t_max})
        n_gemm, t_gemm_prof = [], []
        for n in grid:
            ph = run((n, 0, ()), args.est_reps, True)
            n_gemm.append(n)
            t_gemm_prof.append(sum(ph[k] for k in LINEAR_PHASES))
        dec_iso = wl.estimator_batches(args.seed, args.est_profile, "decode")
        pre_iso = wl.estimator_batches(args.seed, args.est_profile, "prefill")
        wd, td = [], []
        for it in dec_iso:
            wd.append(float(sum(it[2])))
            td.append(run(it, args.est_reps, True)["fork"])
        wp, tp = [], []
        for it in pre_iso:
            wp.append(float(it[0]) * (it[1] + (it[0] + 1) / 2.0))
            tp.append(run(it, args.est_reps, True)["fork"])
        model = cf.cf_latency_model()
        model.gamma, model.gamma0 = cf.cf_latency_fit_line(n_gemm, t_gemm_prof)
        model.a_d, model.a_d0 = cf.cf_latency_fit_line(wd, td)
        model.a_p, model.a_p0 = cf.cf_latency_fit_line(wp, tp)

        def parts(it):
            l, cp, ctx = it
            return cf.cf_latency_predict(model, [(l, len(ctx), float(sum(ctx)))], [(l, cp)] if l else [], 1)

        # 2. contention factors from co-batched iterations (plain step time)
        cal = wl.estimator_batches(args.seed, args.est_calibrate, "calibrate")
        cal_meas = [run(it, args.est_reps, False) for it in cal]
        cal_parts = [parts(it) for it in cal]
        calib_mape = cf.cf_latency_calibrate(model, [p["t_gemm"] for p in cal_parts],
                                             [p["t_prefill"] for p in cal_parts],
                                             [p["t_decode"] for p in cal_parts], cal_meas, 4.0, 0.005)
        # 3. validation on an independent draw
        val = wl.estimator_batches(args.seed, args.est_validate, "validate")
        meas = np.array([run(it, args.est_reps, False) for it in val])
        pred = np.array([parts(it)["t_iter"] for it in val])
        ape = np.abs(pred - meas) / meas * 100.0
        # the same iterations without contention factors (alpha = beta = 1)
        m1 = cf.cf_latency_model(**{f: getattr(model, f) for f, _ in cf.cf_latency_model._fields_})
        m1.alpha = m1.beta = 1.0
        pred1 = np.array([cf.cf_latency_predict(m1, [(l, len(c), float(sum(c)))], [(l, cp)], 1)["t_iter"]
                          for l, cp, c in val])
        # 4. the dispatcher on one GPU (Algorithm 2 with N = 1): the largest
        # TBT-safe chunk for a new prompt next to 16 decodes at 8K, over
        # the model's layers, then that iteration measured
        tbt = []
        if name in MODEL_LAYERS:
            layers = MODEL_LAYERS[name]
            ctx16 = (8192,) * 16
            for tau in (50.0, 100.0):
                r = cf.cf_waterfill_dispatch(model, layers, tau, TBT_QUANTUM, [len(ctx16)], [float(sum(ctx16))],
                                             [0], [], (t_max - len(ctx16), 0))
                l = int(r["chunk"])
                meas_layer = run((l, 0, ctx16), args.est_reps, False) if l > 0 else None
                tbt.append({"tbt_ms": tau, "layers": layers, "chunk": l, "capped": l == t_max - len(ctx16),
                            "pred_ms": round(r["t_iter"], 3),
                            "meas_ms": round(layers * meas_layer, 3) if meas_layer else None,
                            "pages_h100_chunk": PAGES_TBT_CHUNK.get(name, {}).get(tau)})
        clocks.mark("t1")
        clocks.stop()
        page_model, page_mape = PAGES_ESTIMATOR_MAPE.get(name, (None, None))

        def r2(xs, ys, a, a0):
            xs, ys = np.asarray(xs), np.asarray(ys)
            res = ys - (a * xs + a0)
            return float(1.0 - (res ** 2).sum() / ((ys - ys.mean()) ** 2).sum())

        line = {
            "estimator": name, "workload": f"{name}: {s.n_q_heads}/{s.n_kv_heads} heads, H {s.hidden}, "
                                          f"F {s.ffn_dim}; one layer, one GPU",
            "mape_pct": round(float(ape.mean()), 3), "n_validate": len(val),
            "ape_p50_pct": round(float(np.percentile(ape, 50)), 3),
            "ape_p90_pct": round(float(np.percentile(ape, 90)), 3), "ape_max_pct": round(float(ape.max()), 3),
            "mape_alpha_beta_1_pct": round(float((np.abs(pred1 - meas) / meas).mean() * 100), 3),
            "calibrate": {"n": len(cal), "mape_pct": round(calib_mape, 3)},
            "coeffs_ms": {f: getattr(model, f) for f, _ in cf.cf_latency_model._fields_},
            "fit_r2": {"gemm": r2(n_gemm, t_gemm_prof, model.gamma, model.gamma0),
                       "decode": r2(wd, td, model.a_d, model.a_d0), "prefill": r2(wp, tp, model.a_p, model.a_p0)},
            "profiles": {"gemm_points": len(n_gemm), "decode_points": len(wd), "prefill_points": len(wp),
                         "reps": args.est_reps},
            "ranges": {"chunk": wl.EST_CHUNK, "decodes": wl.EST_DECODES, "context": wl.EST_CONTEXT},
            "step_ms": {"min": round(float(meas.min()), 4), "median": round(float(np.median(meas)), 4),
                        "max": round(float(meas.max()), 4)},
            "pages": {"model": page_model, "mape_pct": page_mape, "hardware": "H100 (context, not a target)"},
            "tbt_chunk": {"decodes": "16 @ 8192", "quantum": TBT_QUANTUM, "layers_only": True, "cases": tbt},
            "clocks": clocks.summary(), "seconds": round(time.perf_counter() - t_start, 1),
        }
        if args.estimator_out:
            with open(args.estimator_out, "a") as f:
                f.write(json.dumps({"estimator": name, "validate": [
                    {"l": l, "c_p": cp, "n_d": len(c), "ctx_sum": int(sum(c)), "meas_ms": float(mm),
                     "pred_ms": float(pp)} for (l, cp, c), mm, pp in zip(val, meas, pred)],
                    "gemm": list(zip(n_gemm, t_gemm_prof)), "decode": list(zip(wd, td)),
                    "prefill": list(zip(wp, tp))}) + "\n")
        lines.append(line)
        eng.close()
        del kp, vp, x, out, W
        torch.cuda.empty_cache()
    return lines


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle timed on the host cores, each step a
    bounded sample of the workload's rows sized so that all steps take about
    REFERENCE_BUDGET_S seconds.  Rank 0 only."""
    import workload as wl
    if rank != 0:
        return None
    w = wl.WORKLOADS[args.workload]
    b = wl.make_batch(w, args.seed)
    x = wl.make_x(w, b, args.seed)
    W = wl.make_weights(w, args.seed, unit_gains=True)
    kp, vp = wl.make_pools(w, b, args.seed)
    full = reference_rows(b)
    t_full = oracle_sample(w, b, x, W, kp, vp, full)            # also the first warm-up step
    frac = min(1.0, REFERENCE_BUDGET_S / max(1e-6, args.steps * t_full))
    rows = reference_rows(b, frac)
    for _ in range(args.warmup - 1):
        oracle_sample(w, b, x, W, kp, vp, rows)
    secs = [oracle_sample(w, b, x, W, kp, vp, rows) for _ in range(args.steps)]
    total = sum(secs)
    value = len(rows) * args.steps / total
    sample = (f"fp64 oracle layer step on {len(rows)} of {b.n_tokens} rows per step (leading chunk rows + "
              f"leading decodes, sized to ~{REFERENCE_BUDGET_S:.0f} s for {args.steps} steps)")
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": dict(workload_config(w, b, world), rows_per_step=len(rows)),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                             "host_cores": os.cpu_count(), "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="q32b",
                    help="tiny | l8b | q14b | mix | q32b (default: the largest single-GPU configuration) | mchunk")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", default="cf", choices=["cf", "reference"])
    ap.add_argument("--decode-sms", type=int, default=0)
    ap.add_argument("--sweep-decode-sms", action="store_true",
                    help="longer decode-share sweep (steps/4 profiled steps per share instead of 10)")
    ap.add_argument("--no-share-sweep", action="store_true", help="skip the decode-share sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graphs", type=int, default=0, choices=[0, 1],
                    help="replay the linear segments of the step as CUDA graphs (1) or launch eagerly (0)")
    ap.add_argument("--prefill-pairing", type=int, default=0, choices=[0, 1, 2, 3],
                    help="prefill work items: 0 automatic, 1 single tiles, 2 tile pairs, 3 head pairs")
    ap.add_argument("--prefill-split", type=int, default=0,
                    help="prefill key-range cuts: 0 automatic, 1 never, n >= 2 n ranges")
    ap.add_argument("--split-k", type=int, default=0,
                    help="GEMM split-K tail: 0 automatic, 1 whole tiles only, n >= 2 n k-chunks")
    ap.add_argument("--kernel", choices=["decode", "prefill", "prefill-long", "gemm", "prefill-chunks"], default=None,
                    help="run one small launch of one kernel (for ncu) instead of the benchmark")
    ap.add_argument("--estimator", default=None,
                    help="fit and validate the iteration-latency estimator for these workloads "
                         "(comma-separated, e.g. l8b,q14b,q32b) instead of the benchmark")
    ap.add_argument("--est-reps", type=int, default=3)
    ap.add_argument("--est-profile", type=int, default=40)
    ap.add_argument("--est-calibrate", type=int, default=50)
    ap.add_argument("--est-validate", type=int, default=200)
    ap.add_argument("--estimator-out", default=None, help="append per-iteration records (JSON lines) here")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.kernel:
        print(json.dumps(run_kernel_case(args)))
        return
    if args.estimator:
        for line in run_estimator(args):
            print(json.dumps(line), flush=True)
        return
    rank, world, local, pg = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_cf(args, rank, world, local, pg)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
