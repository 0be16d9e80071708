"""Benchmark of exact tiled attention, forward + backward, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--quick]

One step = the whole hot path on one batch: fa_fwd (O, L), fa_bwd_preprocess (D)
and fa_bwd (dQ, dK, dV), all through the C ABI.  The default workload is the
very-long-context shape B=1, H=32, N=32768, d=128, causal (its bf16 inputs,
1 GiB, exceed the 129 MB L2, so no flush is needed between steps).  Throughput
counts 4 N^2 d (forward) + 10 N^2 d (backward) FLOPs per head, halved with the
causal mask.  Prints ONE JSON line (rank 0).

--impl reference times the float64 CPU oracle instead (a deliberately slow
program, run as it stands on the host cores, each step a bounded sample of the
same workload).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import seeded_inputs as si  # noqa: E402

HEADLINE = "vlong_1x32x32768x128"
METRIC = "attention fwd+bwd TFLOP/s (bf16, d=128, N=4K-32K)"
UNIT = "TFLOP/s"


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# backward main kernel on the very long causal shape, from the ncu capture of this
# kernel on that shape; valid for the kernel as captured (set to None whenever the
# kernel changes).
_TRAFFIC = {("vlong_1x32x32768x128", True): 1621201835 + 1024701867}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------------ clocks sampling

class ClockSampler:
    """nvidia-smi samples of the SM clock, power and throttle reasons during the timed
    region; the raw samples go to $FA_CLOCKS_DIR (default: the temporary directory)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join(os.environ.get("FA_CLOCKS_DIR") or tempfile.gettempdir(), f"fa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
                except ValueError:
                    continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        pmax = max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= 0.5 * pmax] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3][1:5]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": pmax, "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------ our arm

class Runner:
    """Device buffers and the three C-ABI calls of one step (the general-mask entry
    points: Q, dO have Nq rows per head, K, V have Nk; optional sliding window)."""

    def __init__(self, fa, torch, w: si.Workload, causal: bool, dev, Nq=None, Nk=None, window=0):
        self.fa, self.torch, self.w, self.causal, self.window = fa, torch, w, causal, window
        self.Nq, self.Nk = Nq or w.N, Nk or w.N
        B, H, d = w.B, w.H, w.d
        Q, K, V, dO = si.make_qkvdo(B, H, max(self.Nq, self.Nk), d, w.seed, w.qk_mult)
        Q, dO = (t[:, :, :self.Nq].contiguous() for t in (Q, dO))
        K, V = (t[:, :, :self.Nk].contiguous() for t in (K, V))
        self.host_in = [t.pin_memory() for t in (Q, K, V, dO)]
        self.q, self.k, self.v, self.do = (t.to(dev, non_blocking=False) for t in self.host_in)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, self.Nq), dtype=torch.float32, device=dev)
        self.D = torch.empty((B, H, self.Nq), dtype=torch.float32, device=dev)
        self.dq = torch.empty_like(self.q)
        self.dk, self.dv = torch.empty_like(self.k), torch.empty_like(self.v)
        self.ws_bytes = fa.fa_bwd_workspace_size_ex(B, H, self.Nq, self.Nk, d, causal, window)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.s = self.stream.cuda_stream
        self.scale = w.scale

    def fwd(self):
        w, fa = self.w, self.fa
        fa.check(fa.fa_fwd_ex(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(), self.o.data_ptr(),
                              self.lse.data_ptr(), w.B, w.H, self.Nq, self.Nk, w.d, self.causal, self.window, self.scale,
                              self.s), "fa_fwd_ex")

    def bwd(self):
        w, fa = self.w, self.fa
        fa.check(fa.fa_bwd_preprocess(self.o.data_ptr(), self.do.data_ptr(), self.D.data_ptr(), w.B, w.H, self.Nq,
                                      w.d, self.s), "fa_bwd_preprocess")
        fa.check(fa.fa_bwd_ex(self.q.data_ptr(), self.k.data_ptr(), self.v.data_ptr(), self.o.data_ptr(),
                              self.do.data_ptr(), self.lse.data_ptr(), self.D.data_ptr(), self.dq.data_ptr(),
                              self.dk.data_ptr(), self.dv.data_ptr(), w.B, w.H, self.Nq, self.Nk, w.d, self.causal,
                              self.window, self.scale, self.ws.data_ptr(), self.ws_bytes, self.s), "fa_bwd_ex")

    def visible_pairs(self):
        """(query, key) entries the mask leaves visible per head (the masked FLOP count is
        4 d and 10 d times this), counted from the mask's definition."""
        off = self.Nk - self.Nq
        i = np.arange(self.Nq, dtype=np.int64)
        hi = np.minimum(self.Nk - 1, i + off) if self.causal else np.full_like(i, self.Nk - 1)
        lo = np.maximum(0, i + off - self.window + 1) if self.window > 0 else np.zeros_like(i)
        return int((hi - lo + 1).sum())

    @staticmethod
    def launches_per_step(bwd_form):
        """Kernels this library launches per step: the forward, the preprocess, then with a
        one-kernel backward (forms 1, 3) the workspace clear, the backward kernel and the dQ
        convert, or with the two-kernel backward (form 2) its key-tile and query-tile kernels."""
        return 4 if bwd_form == 2 else 5


def time_steps(torch, r: Runner, steps: int, warmup: int, flush=None, kernel_events=False):
    """Times K steps with CUDA events on the launching stream.  Returns per-phase
    milliseconds (totals over the K steps); with kernel_events, also the totals of
    the forward kernel's and the backward main kernel's own launches (events the
    library records around those launches on the same stream)."""
    for _ in range(warmup):
        r.fwd()
        r.bwd()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)] if kernel_events else None
    if kev:
        for e in (x for row in kev for x in row):
            e.record(r.stream)  # creates the handle the library records into
        torch.cuda.synchronize()
    for i in range(steps):
        if flush is not None:
            flush()
        if kev:
            r.fa.check(r.fa.fa_debug_set_kernel_events(0, kev[i][0].cuda_event, kev[i][1].cuda_event), "events")
            r.fa.check(r.fa.fa_debug_set_kernel_events(1, kev[i][2].cuda_event, kev[i][3].cuda_event), "events")
        ev[i][0].record(r.stream)
        r.fwd()
        ev[i][1].record(r.stream)
        r.bwd()
        ev[i][2].record(r.stream)
    torch.cuda.synchronize()
    if kev:
        r.fa.check(r.fa.fa_debug_set_kernel_events(0, None, None), "events")
        r.fa.check(r.fa.fa_debug_set_kernel_events(1, None, None), "events")
    fwd = sum(e[0].elapsed_time(e[1]) for e in ev)
    bwd = sum(e[1].elapsed_time(e[2]) for e in ev)
    if not kev:
        return fwd, bwd
    fwd_k = sum(e[0].elapsed_time(e[1]) for e in kev)
    bwd_k = sum(e[2].elapsed_time(e[3]) for e in kev)
    return fwd, bwd, fwd_k, bwd_k


def e2e_steps(torch, r: Runner, steps: int, pipelined: bool = True):
    """The step through the C ABI with host buffers, timed on the caller's stream:
    pinned host -> device copies of Q, K, V, dO and device -> pinned host copies of O,
    L, dQ, dK, dV inside the timed region.  pipelined: one fa_fwd_bwd_host call
    per step (heads in chunks, copies overlapped with the kernels); otherwise the
    copies and the three device calls one after another on one stream.  Returns the
    median milliseconds of three blocks of `steps` steps."""
    fa, w = r.fa, r.w
    outs = [r.o, r.lse, r.dq, r.dk, r.dv]
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in r.host_in)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    dev_in = [r.q, r.k, r.v, r.do]
    ws_bytes = fa.fa_fwd_bwd_host_workspace_size(w.B, w.H, r.Nq, r.Nk, w.d, r.causal, r.window, 0)
    ws = torch.empty(ws_bytes + 256, dtype=torch.uint8, device=r.q.device) if pipelined else None
    base = (ws.data_ptr() + 255) // 256 * 256 if pipelined else 0

    def step():
        if pipelined:
            fa.check(fa.fa_fwd_bwd_host(*(t.data_ptr() for t in r.host_in), *(t.data_ptr() for t in host_out), w.B,
                                        w.H, r.Nq, r.Nk, w.d, r.causal, r.window, r.scale, 0, base, ws_bytes, r.s),
                     "fa_fwd_bwd_host")
            return
        for d_, h_ in zip(dev_in, r.host_in):
            d_.copy_(h_, non_blocking=True)
        r.fwd()
        r.bwd()
        for h_, d_ in zip(host_out, outs):
            h_.copy_(d_, non_blocking=True)

    step()  # warm-up: creates the library's copy streams
    torch.cuda.synchronize()
    # three blocks of `steps` steps; the median block (host memory traffic from other
    # processes on the machine can slow a single block)
    blocks = []
    for _ in range(3):
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(r.stream)
        for _ in range(steps):
            step()
        stop.record(r.stream)
        torch.cuda.synchronize()
        blocks.append(start.elapsed_time(stop))
    del ws
    return statistics.median(blocks), h2d, d2h


def cpu_oracle_sample(w: si.Workload, causal: bool, budget_s: float = 12.0, max_rows=None):
    """Times the float64 oracle (forward + backward) on the first n rows of head 0.
    With the causal mask those rows see only keys 0..n-1, so this is an exact
    sub-problem with 4 n^2 d + 10 n^2 d (halved) counted FLOPs.  n doubles from
    512 until the budget is used."""
    import oracle
    Q, K, V, dO = si.make_qkvdo(1, 1, w.N, w.d, seed=w.seed, qk_mult=w.qk_mult)
    q, k, v, do = (si.to_f64(t)[0, 0] for t in (Q, K, V, dO))
    n, spent, flops, last = 512, 0.0, 0.0, None
    limit = min(w.N, max_rows or w.N)
    while True:
        t0 = time.perf_counter()
        oracle.standard_attention_fwd(q[:n], k[:n], v[:n], causal)
        oracle.standard_attention_bwd(q[:n], k[:n], v[:n], do[:n], causal)
        dt = time.perf_counter() - t0
        f = 14.0 * n * n * w.d * (0.5 if causal else 1.0)
        spent += dt
        flops += f
        last = (n, dt, f)
        if spent >= budget_s or n >= limit or spent + 4.5 * dt > 2.5 * budget_s:
            break
        n = min(2 * n, limit)
    n, dt, f = last
    return {"value": f / dt / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"float64 NumPy oracle fwd+bwd on query rows 0..{n - 1} of head 0 "
                      f"({'causal' if causal else 'full'}; an exact sub-problem of {w.name}), "
                      f"{dt:.2f} s for {f / 1e9:.1f} GFLOP counted"}


def rank_env():
    """(world size, rank, local rank) from the launcher's environment (1, 0, 0 alone)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(ms, dist, device):
    """The slowest rank's timed region: every rank gets the maximum (no-op alone)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step, steps, world, total_ms):
    """Throughput of the whole job: every rank runs a full replica of the step
    (weak scaling, no data-path collective), so the job does world times the work
    in the slowest rank's time."""
    return world * flops_per_rank_step * steps / (total_ms / 1e3) / 1e12


def run_ours(args):
    import torch

    import exact_tiled_attention_26_gb300 as fa

    world, rank, local = rank_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    w = si.WORKLOADS[args.workload]
    causal = True if len(w.causal) == 1 and w.causal[0] else (args.causal if args.causal is not None else w.causal[-1])
    fa.check(fa.fa_debug_set_bwd_split(args.bwd_split), "fa_debug_set_bwd_split")
    fa.check(fa.fa_debug_set_fwd_form(args.fwd_form), "fa_debug_set_fwd_form")
    r = Runner(fa, torch, w, causal, dev, window=args.window)
    flops_f, flops_b = w.fwd_flops(causal), w.bwd_flops(causal)
    if args.window:  # FLOPs on the visible entries only
        flops_f = 4.0 * w.d * w.B * w.H * r.visible_pairs()
        flops_b = 2.5 * flops_f

    # warm-up (also compiles nothing: the library is prebuilt), then the timed region
    for _ in range(args.warmup):
        r.fwd()
        r.bwd()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        fwd_ms, bwd_ms, fwd_k_ms, bwd_k_ms = time_steps(torch, r, args.steps, 0, kernel_events=True)
    st, detail = fa.fa_poll_device_error(r.s)
    fa.check(st, f"device status word (site {detail:#x})")
    total_ms = max_over_ranks(fwd_ms + bwd_ms, dist, dev)
    ms_step = total_ms / args.steps
    value = whole_job_tflops(flops_f + flops_b, args.steps, world, total_ms)

    peaks, peak_src = _peaks()
    # The kernels run at burst clocks (about 2 GHz in 25 ms steps, well short of the
    # seconds-long loop behind the sustained figure): the burst cuBLAS figure is the
    # roofline's peak; the sustained one is kept as a labelled second ratio.
    burst = float(peaks.get("bf16_tflops"))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    sustained_mhz = (peaks.get("clocks_under_load") or {}).get("sm_mhz_median")
    clocks = clk.summary()
    bwd_tflops = flops_b * args.steps / (bwd_ms / 1e3) / 1e12
    fwd_tflops = flops_f * args.steps / (fwd_ms / 1e3) / 1e12
    bwd_kernel_tflops = flops_b * args.steps / (bwd_k_ms / 1e3) / 1e12
    fwd_kernel_tflops = flops_f * args.steps / (fwd_k_ms / 1e3) / 1e12
    st_forms, f_form, b_form = fa.fa_selected_forms(w.B, w.H, r.Nq, r.Nk, w.d, causal, args.window)
    bwd_kernel = {1: "bwd_tile_kernel" if w.d >= 64 else "bwd_kernel", 2: "bwd_kv_kernel + bwd_q_kernel",
                  3: "bwd_persist_kernel"}.get(b_form, "?") if st_forms == fa.FA_OK else "?"
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded iid N(0,1) bf16 Q, K, V, dO)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal,
                   "global_batch": w.B * world, "seq_len": w.N, "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": "no flush: inputs (Q, K, V, dO) total "
                         f"{4 * w.B * w.H * w.N * w.d * 2 / 2**30:.2f} GiB, larger than the 129 MB L2"},
        "fwd_tflops": round(fwd_tflops, 2), "bwd_tflops": round(bwd_tflops, 2),
        "fwd_kernel_tflops": round(fwd_kernel_tflops, 2), "bwd_kernel_tflops": round(bwd_kernel_tflops, 2),
        "frac_of_bf16_peak": round(value / world / burst, 4),
        "frac_of_bf16_peak_basis": f"{peak_src} burst bf16_tflops {burst}",
        "frac_of_sustained_bf16_peak": round(value / world / sustained, 4),
        "sustained_basis": (f"{peak_src} bf16_tflops_sustained {sustained}, taken at a median SM clock of "
                            f"{sustained_mhz} MHz; this run's median SM clock {clocks.get('sm_mhz')} MHz"),
        "roofline": {
            "bound": "tensor",
            "kernel": f"{bwd_kernel} (the d=128 backward main kernel; form {b_form})",
            "achieved": round(bwd_kernel_tflops, 2), "peak": burst, "unit": "TFLOP/s",
            "frac": round(bwd_kernel_tflops / burst, 4),
            "traffic": None if args.window else _TRAFFIC.get((w.name, causal)),
            "peak_source": f"{peak_src} bf16_tflops (burst: the kernel runs at burst clocks, see clocks)",
            "timing": ("CUDA events the library records on the launching stream around each launch of the main "
                       "kernel, summed over the timed steps (workspace clear, dQ convert and preprocess excluded)"),
            "algorithmic": "10 N^2 d / 2 FLOPs per head (causal) per launch",
            "frac_of_sustained": round(bwd_kernel_tflops / sustained, 4),
        },
        "gpu_launches": Runner.launches_per_step(b_form) * args.steps,
        "clocks": clocks,
    }
    if args.window:
        line["config"]["window"] = args.window
    if st_forms == fa.FA_OK:
        line["config"]["forms"] = {"fwd": f_form, "bwd": b_form}
    if not args.quick and rank == 0:
        # end to end through the C ABI with host buffers
        steps_e2e = max(2, min(args.steps, 5))
        ms, h2d, d2h = e2e_steps(torch, r, steps_e2e)
        ms_serial, _, _ = e2e_steps(torch, r, steps_e2e, pipelined=False)
        hc = fa.fa_fwd_bwd_host_chunk_heads(w.B, w.H, w.N, w.N, w.d, 0)
        line["e2e"] = {"value": round((flops_f + flops_b) * steps_e2e / (ms / 1e3) / 1e12, 2), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": round(ms / steps_e2e, 3),
                       "api": f"fa_fwd_bwd_host (pinned host arrays; {hc} head{'s' if hc != 1 else ''} per chunk, "
                              "copies overlapped)",
                       "serial_ms_per_step": round(ms_serial / steps_e2e, 3)}
        line["per_config"] = per_config(fa, torch, dev, burst)
        line["cpu_baseline"] = cpu_oracle_sample(w, causal)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def per_config(fa, torch, dev, burst):
    """The other full-size shapes, each timed briefly; L2 is flushed before every
    step (a 256 MiB write) because their inputs are near or below the L2 size."""
    flush_buf = torch.empty(256 * 2**20, dtype=torch.uint8, device=dev)
    out = {}
    for name, causal in (("mid_2x16x4096x128", False), ("mid_2x16x4096x128", True),
                         ("long_1x32x8192x128", True), ("long_1x32x8192x128_qk4", True),
                         ("small_4x8x1024x64", True)):
        w = si.WORKLOADS[name]
        r = Runner(fa, torch, w, causal, dev)
        fwd_ms, bwd_ms = time_steps(torch, r, 10, 3, flush=lambda: flush_buf.zero_())
        ff, fb = w.fwd_flops(causal) * 10, w.bwd_flops(causal) * 10
        out[f"{name}{'_causal' if causal else ''}"] = {
            "fwd_tflops": round(ff / fwd_ms / 1e9, 1), "bwd_tflops": round(fb / bwd_ms / 1e9, 1),
            "fwd_bwd_tflops": round((ff + fb) / (fwd_ms + bwd_ms) / 1e9, 1),
            "frac_of_bf16_peak": round((ff + fb) / (fwd_ms + bwd_ms) / 1e9 / burst, 4),
            "ms_per_step": round((fwd_ms + bwd_ms) / 10, 4)}
        del r
    # the general mask (FLOPs counted on the visible entries: 4 d and 10 d per entry)
    for label, name, Nq, Nk, window in (
            ("long_1x32x8192x128_causal_window1024", "long_1x32x8192x128", 8192, 8192, 1024),
            ("prefill_1x32_2048q_32768k_x128_causal", "vlong_1x32x32768x128", 2048, 32768, 0)):
        w = si.WORKLOADS[name]
        r = Runner(fa, torch, w, True, dev, Nq=Nq, Nk=Nk, window=window)
        fwd_ms, bwd_ms = time_steps(torch, r, 10, 3, flush=lambda: flush_buf.zero_())
        vp = r.visible_pairs() * w.B * w.H
        ff, fb = 4.0 * w.d * vp * 10, 10.0 * w.d * vp * 10
        out[label] = {"fwd_tflops": round(ff / fwd_ms / 1e9, 1), "bwd_tflops": round(fb / bwd_ms / 1e9, 1),
                      "fwd_bwd_tflops": round((ff + fb) / (fwd_ms + bwd_ms) / 1e9, 1),
                      "ms_per_step": round((fwd_ms + bwd_ms) / 10, 4), "visible_pairs_per_head": vp // (w.B * w.H)}
        del r
    # decode (one new query per sequence against an 8192-key cache): forward only, HBM-bound
    w = si.Workload("decode_16x32x1q_8192k_x128", 16, 32, 8192, 128, (True,), seed=5)
    r = Runner(fa, torch, w, True, dev, Nq=1, Nk=8192)
    for _ in range(3):
        r.fwd()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    total = 0.0
    for _ in range(10):
        flush_buf.zero_()
        ev[0].record(r.stream)
        r.fwd()
        ev[1].record(r.stream)
        torch.cuda.synchronize()
        total += ev[0].elapsed_time(ev[1])
    ms = total / 10
    bytes_ = w.B * w.H * (2 * 8192 * w.d * 2 + 2 * w.d * 2 + 4)  # K, V read; q read, o and L written
    hbm = float(_peaks()[0].get("hbm_gbs", 0.0)) or None
    out["decode_16x32x1q_8192k_x128_fwd"] = {"ms": round(ms, 4), "gbs": round(bytes_ / ms / 1e6, 1),
                                             "hbm_peak_gbs": hbm}
    del r
    return out


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    _, rank, _ = rank_env()
    if rank != 0:  # under torchrun only rank 0 times the oracle
        return
    w = si.WORKLOADS[args.workload]
    causal = True
    import oracle
    Q, K, V, dO = si.make_qkvdo(1, 1, w.N, w.d, seed=w.seed, qk_mult=w.qk_mult)
    q, k, v, do = (si.to_f64(t)[0, 0] for t in (Q, K, V, dO))
    n = min(2048, w.N)  # rows 0..n-1 of head 0: an exact causal sub-problem of the workload
    flops = 14.0 * n * n * w.d * 0.5

    def step():
        oracle.standard_attention_fwd(q[:n], k[:n], v[:n], causal)
        oracle.standard_attention_bwd(q[:n], k[:n], v[:n], do[:n], causal)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = flops * args.steps / dt / 1e12
    sample = (f"float64 NumPy oracle fwd+bwd on query rows 0..{n - 1} of head 0 of {w.name} (causal: an exact "
              f"sub-problem), {flops / 1e9:.2f} GFLOP counted per step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded iid N(0,1), bf16-rounded, widened to f64)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(si.WORKLOADS))
    ap.add_argument("--causal", type=int, default=None, help="for workloads that run both mask modes")
    ap.add_argument("--quick", action="store_true", help="headline timing only (for profiler runs)")
    ap.add_argument("--bwd-split", type=int, default=0, choices=[0, 1, 2, 3],
                    help="backward form for d=128: 1 one kernel + dQ reduction, 2 two kernels, 3 form 1 persistent, "
                         "0 library default")
    ap.add_argument("--fwd-form", type=int, default=0, choices=[0, 1, 2, 3],
                    help="forward kernel: 1 one query tile per CTA, 2 two per CTA (d=128), 3 persistent, "
                         "0 library default")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window over the workload's causal mask (with --quick: profiler runs of the "
                         "windowed kernels)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and not args.quick:
        ap.error("at least 3 warm-up steps")
    if args.window and (not args.quick or args.impl != "ours"):
        ap.error("--window is for --quick runs of this library")
    if (args.fwd_form or args.bwd_split) and not args.quick:
        ap.error("--fwd-form and --bwd-split are for --quick runs (the full run times the library's own choice)")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
