"""Benchmark of the exact-attention hot path on GB300 (one JSON line on rank 0).

A step is one pass of the hot path over synthetic inputs already resident in
device memory:
  * forward, fp16, B=4, H=12, M=N=2048, D=64, scale 0.125, non-causal
    (the workload the headline TFLOP/s is quoted on);
  * backward at the same shape, when the library provides it;
  * flash decoding, bf16, B=8, H=32, N=32768, D=128, n_splits=64 (the K/V cache,
    4.29 GB, is far larger than L2).
Step i runs the forward and the backward on input set i % 12 of twelve seeded
sets (the forward alone touches 12 x 25 MB, the backward 12 x 51 MB: both more
than twice the 129 MB L2, so every call reads its inputs from HBM). The K
calls of each part run back to back on one stream between one pair of CUDA
events. `value` is the forward's TFLOP/s (4*B*H*M*N*D per call); the decode
GB/s (K+V bytes read per call) is reported in the `decode` object. `configs`
times every configuration of the workload list on its own, the same way (calls
back to back over copies of its inputs larger than twice L2; one isolated call
with L2 flushed is reported beside it). `e2e` repeats the forward through the C ABI
on pinned host buffers (fa_fwd_host: the inputs copied in and O/LSE copied back
inside the timed region, overlapped with the kernels chunk by chunk).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

`--impl reference` times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same forward workload, on the host cores.
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

METRIC = "attn fwd TFLOP/s & % tensor peak (B4 H12 N2048 D64); decode KV GB/s & % HBM"
FWD = dict(B=4, H=12, M=2048, N=2048, D=64, scale=0.125, causal=False, dtype="f16")
DEC = dict(B=8, H=32, N=32768, D=128, n_splits=64, dtype="bf16")
L2_FLUSH_BYTES = 512 << 20  # > 129 MB of L2
ROTATE = 12  # input sets of the forward/backward workload used in turn: the forward's 12 x 25 MB > 2 x L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
ROT_BYTES = 300 << 20  # rotated input copies of a configuration: more than twice L2 (129 MB)


def rotation(set_bytes: int, cap: int = 1024) -> int:
    """How many copies of a configuration's inputs (and outputs, workspace) to use in turn, so that
    together they exceed ROT_BYTES and no call finds the previous call's data in L2."""
    return max(2, min(cap, -(-ROT_BYTES // max(1, set_bytes))))


def time_calls(torch, stream, flush, run, n_sets: int, calls: int = 20, isolated: int = 10):
    """`run(i)` issues one call on copy i of the inputs. Returns (seconds per call back to back,
    seconds per call isolated). Back to back: max(calls, 2 n_sets) calls rotating over the copies
    between one pair of CUDA events (the headline's protocol). Isolated: one call between two
    events with L2 flushed (a 512 MB write) before it, which adds the event pair's own time
    (about 2 us) and a cold L2 to every call."""
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for i in range(3):
        run(i % n_sets)
    n = max(calls, 2 * n_sets)
    a, b = ev(), ev()
    a.record(stream)
    for i in range(n):
        run(i % n_sets)
    b.record(stream)
    recs = []
    for i in range(isolated):
        flush.zero_()
        x, y = ev(), ev()
        x.record(stream)
        run(i % n_sets)
        y.record(stream)
        recs.append((x, y))
    torch.cuda.synchronize()
    return a.elapsed_time(b) / n / 1e3, sum(x.elapsed_time(y) for x, y in recs) / len(recs) / 1e3


def fwd_flops(c=FWD) -> float:
    f = 4.0 * c["B"] * c["H"] * c["M"] * c["N"] * c["D"]
    return f / 2 if c["causal"] else f


def dec_bytes(c=DEC) -> float:
    return 2.0 * c["B"] * c["H"] * c["N"] * c["D"] * 2  # K and V, 2 bytes each


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks
def other_gpu_processes(device_index: int):
    """Compute processes on this GPU other than this one (nvidia-smi), or None if unavailable."""
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(device_index), "--query-compute-apps=pid,used_memory",
                              "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20).stdout
    except Exception:
        return None
    me = os.getpid()
    procs = []
    for ln in out.splitlines():
        f = [x.strip() for x in ln.split(",")]
        if len(f) >= 2 and f[0].isdigit() and int(f[0]) != me:
            procs.append({"pid": int(f[0]), "mib": f[1]})
    return procs


class ClockSampler:
    """nvidia-smi samples (50 ms) of SM clock and throttle reasons while running, each stamped with
    the host clock so that they can be binned by phase."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        # the timed region starts once nvidia-smi is up and sampling (its start-up, slower on a
        # machine where it has not run yet, then stays out of the region), after 5 s at most
        t_end = time.perf_counter() + 5.0
        while self.proc is not None and len(self.lines) < 2 and time.perf_counter() < t_end:
            time.sleep(0.02)
        time.sleep(0.1)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def __exit__(self, *a):
        time.sleep(0.3)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, phases=None):
        """Median and minimum SM clock, the throttle reasons seen, and with `phases` (name -> host
        perf_counter window) the median and minimum of the samples that fall in each window."""
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for t, ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append((t, float(f[1])))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        mhz = [c for _, c in sm]
        out = {"sm_mhz": statistics.median(mhz), "sm_min_mhz": min(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
               "samples": len(mhz)}
        if phases:
            by = {}
            for name, (a, b) in phases.items():
                w = [c for t, c in sm if a <= t <= b]
                by[name] = {"median": statistics.median(w), "min": min(w), "samples": len(w)} if w else None
            out["phases"] = by
        return out


# ------------------------------------------------------------- CPU oracle
def oracle_forward_sample(budget_s: float, max_heads: int = 480):
    """Times the fp64 oracle forward on whole heads of the forward workload (cycling
    over four seeded heads, up to ten passes over its 48) until `budget_s` of work
    has run; returns (TFLOP/s, heads, seconds, threads)."""
    import numpy as np

    import oracle
    from exact_attention_gb300 import synth
    c = FWD
    q, k, v = synth.attention_inputs(1, 4, c["M"], c["N"], c["D"], c["dtype"], seed=0)
    q, k, v = (synth.to_f64(x, c["dtype"]) for x in (q, k, v))
    heads, t_total = 0, 0.0
    while t_total < budget_s and heads < max_heads:
        h = heads % 4
        t0 = time.perf_counter()
        oracle.forward(q[0, h], k[0, h], v[0, h], c["scale"], c["causal"])
        t_total += time.perf_counter() - t0
        heads += 1
    flops = heads * 4.0 * c["M"] * c["N"] * c["D"]
    return flops / t_total / 1e12, heads, t_total, blas_threads()


def oracle_decode_sample(budget_s: float):
    import oracle
    from exact_attention_gb300 import synth
    c = DEC
    q = synth.decode_query(1, 4, c["D"], c["dtype"], 0)
    heads, t_total, nbytes = 0, 0.0, 0.0
    while t_total < budget_s and heads < 256:
        kh, vh = synth.decode_head_kv(0, heads % 4, c["N"], c["D"], c["dtype"], 0)
        t0 = time.perf_counter()
        oracle.decode(synth.to_f64(q[0, heads % 4], c["dtype"]), synth.to_f64(kh, c["dtype"]),
                      synth.to_f64(vh, c["dtype"]), 1 / math.sqrt(c["D"]))
        t_total += time.perf_counter() - t0
        heads += 1
        nbytes += 2.0 * c["N"] * c["D"] * 2
    return nbytes / t_total / 1e9, heads, t_total


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(n[0])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


# --------------------------------------------------------------- distributed
def dist_setup(n_gpus: int):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device: str = "cuda") -> float:
    """The slowest rank's time: the whole job takes as long as its slowest replica."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, steps: int, seconds_max: float, world: int) -> float:
    """Whole-job throughput of `world` replicas that each did `units_per_rank` per step for
    `steps` steps, timed by the slowest rank (weak scaling: per-rank work is fixed)."""
    return world * steps * units_per_rank / seconds_max


# --------------------------------------------------------------- our arm
def run_ours(args):
    import numpy as np
    import torch

    from exact_attention_gb300 import build as fa_build
    fa_build.build()
    import exact_attention_gb300 as fa
    from exact_attention_gb300 import synth

    rank, world, local = dist_setup(args.gpus)
    stream = torch.cuda.current_stream()
    peaks, peaks_src = load_peaks()

    def dev(a, dt):
        if dt == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    c = FWD
    # ROTATE input sets of the forward/backward workload, used in turn by consecutive steps: together
    # they are larger than L2 (129 MB), so every call reads its inputs from HBM
    sets = []
    for r in range(ROTATE):
        q, k, v, do = synth.attention_inputs(c["B"], c["H"], c["M"], c["N"], c["D"], c["dtype"],
                                             seed=rank * ROTATE + r, with_dout=True)
        qd, kd, vd, dod = dev(q, "f16"), dev(k, "f16"), dev(v, "f16"), dev(do, "f16")
        sets.append(dict(q=qd, k=kd, v=vd, do=dod, o=torch.empty_like(qd),
                         lse=torch.empty((c["B"], c["H"], c["M"]), dtype=torch.float32, device="cuda"),
                         dq=torch.empty_like(qd), dk=torch.empty_like(kd), dv=torch.empty_like(vd)))
    qd, kd, vd, dod = (sets[0][n] for n in ("q", "k", "v", "do"))
    od, lse = sets[0]["o"], sets[0]["lse"]
    # backward workspace: delta, then the f32 dQ accumulator of the fused dK/dV/dQ pass (fa_bwd_ws)
    bws_bytes = fa.fa_bwd_ws_workspace_bytes(c["B"], c["H"], c["M"], c["D"])
    bws = torch.empty(bws_bytes, dtype=torch.uint8, device="cuda")
    BHMND = (c["B"], c["H"], c["M"], c["N"], c["D"])

    d = DEC
    qdec = dev(synth.decode_query(d["B"], d["H"], d["D"], d["dtype"], rank), "bf16")
    kc = torch.empty((d["B"], d["H"], d["N"], d["D"]), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    for b, h, kh, vh in synth.iter_decode_heads(d["B"], d["H"], d["N"], d["D"], d["dtype"], rank):
        kc[b, h] = dev(kh, "bf16")
        vc[b, h] = dev(vh, "bf16")
    odec = torch.empty_like(qdec)
    ws = torch.empty(fa.fa_decode_workspace_bytes(d["B"], d["H"], d["D"], d["n_splits"]) // 4,
                     dtype=torch.float32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    # forward workspace (split schedule), zero-filled once as fa_fwd_ws requires
    fws_bytes = fa.fa_fwd_workspace_bytes(*BHMND, c["causal"], fa.FA_F16)
    fws = torch.zeros(max(fws_bytes, 16), dtype=torch.uint8, device="cuda")

    def check(s, what):
        if s != fa.FA_OK:
            raise RuntimeError(f"{what}: {fa.fa_status_string(s)}: {fa.fa_last_error_message()}")

    def run_fwd(i=0):
        t = sets[i % ROTATE]
        check(fa.fa_fwd_ws(t["q"], t["k"], t["v"], t["o"], t["lse"], fws if fws_bytes else None, fws_bytes, *BHMND,
                           c["scale"], c["causal"], fa.FA_F16, stream), "fa_fwd_ws")

    have_bwd = True

    def run_bwd(i=0):
        nonlocal have_bwd
        if not have_bwd:
            return
        t = sets[i % ROTATE]
        s = fa.fa_bwd_ws(t["q"], t["k"], t["v"], t["o"], t["do"], t["lse"], t["dq"], t["dk"], t["dv"], bws, bws_bytes,
                         *BHMND, c["scale"], c["causal"], fa.FA_F16, stream)
        if s == fa.FA_ERR_UNSUPPORTED:
            have_bwd = False
            return
        check(s, "fa_bwd_ws")

    def run_dec():
        check(fa.fa_decode(qdec, kc, vc, odec, ws, d["B"], d["H"], d["N"], d["D"], 1 / math.sqrt(d["D"]),
                           d["n_splits"], fa.FA_BF16, stream), "fa_decode")

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    NCHUNK = 10  # events inside each part: per-chunk times show whether a slow part was slow throughout

    def steps(n, chunks=None):
        """n steps: step i runs the forward and the backward on input set i % ROTATE and one decode.
        Each part's n calls run back to back between one pair of CUDA events; returns their times.
        With `chunks` (a dict), each part's calls are also cut into NCHUNK chunks between events."""
        e = [ev() for _ in range(6)]

        def part(k, run):
            marks = []
            for i in range(n):
                if chunks is not None and i % max(1, n // NCHUNK) == 0 and len(marks) < NCHUNK:
                    marks.append((i, ev()))
                    marks[-1][1].record(stream)
                run(i)
            if chunks is not None:
                end = ev()
                end.record(stream)
                chunks[k] = (marks, end)
        e[0].record(stream)
        part("fwd", run_fwd)
        e[1].record(stream)
        e[2].record(stream)
        part("bwd", run_bwd)
        e[3].record(stream)
        e[4].record(stream)
        part("decode", lambda i: run_dec())
        e[5].record(stream)
        return e

    steps(args.warmup)
    check(fa.fa_last_status(stream), "warm-up")
    torch.cuda.synchronize()

    load_before = os.getloadavg()[0] if hasattr(os, "getloadavg") else None
    foreign = other_gpu_processes(local)
    chunk_ev = {}
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e = steps(args.steps, chunk_ev)
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - t0
    check(fa.fa_last_status(stream), "timed steps")
    t_fwd = e[0].elapsed_time(e[1]) / 1e3
    t_bwd = e[2].elapsed_time(e[3]) / 1e3
    t_dec = e[4].elapsed_time(e[5]) / 1e3
    t_step = e[0].elapsed_time(e[5]) / 1e3
    # the device starts the first forward as soon as it is queued: the phases' windows on the host clock
    clock_phases = {"fwd": (t0, t0 + t_fwd), "bwd": (t0 + t_fwd, t0 + t_fwd + t_bwd),
                    "decode": (t0 + t_fwd + t_bwd, t0 + t_step)}
    t_fwd = max_over_ranks(t_fwd, world)
    t_bwd = max_over_ranks(t_bwd, world)
    t_dec = max_over_ranks(t_dec, world)
    t_step = max_over_ranks(t_step, world)
    K = args.steps
    fwd_tflops = whole_job_rate(fwd_flops(), K, t_fwd, world) / 1e12
    dec_gbs = whole_job_rate(dec_bytes(), K, t_dec, world) / 1e9
    bwd_tflops = whole_job_rate(2.5 * fwd_flops(), K, t_bwd, world) / 1e12 if have_bwd and t_bwd > 0 else None

    # ---- end to end through the C ABI on pinned host buffers (fa_fwd_host: Q, K, V copied in
    # and O, LSE copied out every step, chunked over heads so the copies overlap the kernels)
    hq, hk, hv = (x.cpu().pin_memory() for x in (qd, kd, vd))
    ho = torch.empty_like(hq).pin_memory()
    hl = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    hws_bytes = fa.fa_fwd_host_workspace_bytes(*BHMND, c["causal"], fa.FA_F16)
    hws = torch.zeros(hws_bytes, dtype=torch.uint8, device="cuda")
    e2e_recs = []
    for i in range(args.warmup + args.steps):
        a, b = ev(), ev()
        a.record(stream)
        check(fa.fa_fwd_host(hq, hk, hv, ho, hl, hws, hws_bytes, *BHMND, c["scale"], c["causal"], fa.FA_F16, stream),
              "fa_fwd_host")
        b.record(stream)
        if i >= args.warmup:
            e2e_recs.append((a, b))
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_recs) / 1e3, world)
    e2e_tflops = whole_job_rate(fwd_flops(), K, t_e2e, world) / 1e12
    h2d = 3 * qd.numel() * qd.element_size()
    d2h = od.numel() * od.element_size() + lse.numel() * 4

    # decode end to end: cache and query from pinned host memory every call
    dec_e2e = None
    if args.decode_e2e:
        hkc, hvc = kc.cpu().pin_memory(), vc.cpu().pin_memory()
        hqd, hod = qdec.cpu().pin_memory(), torch.empty_like(qdec.cpu()).pin_memory()
        tt = []
        for i in range(2 + min(args.steps, 5)):
            a, b = ev(), ev()
            a.record(stream)
            kc.copy_(hkc, non_blocking=True)
            vc.copy_(hvc, non_blocking=True)
            qdec.copy_(hqd, non_blocking=True)
            run_dec()
            hod.copy_(odec, non_blocking=True)
            b.record(stream)
            if i >= 2:
                tt.append((a, b))
        torch.cuda.synchronize()
        td = sum(a.elapsed_time(b) for a, b in tt) / 1e3 / len(tt)
        dec_e2e = {"value": round(dec_bytes() / td / 1e9, 1), "unit": "GB/s",
                   "h2d_bytes_per_step": int(2 * kc.numel() * 2 + qdec.numel() * 2),
                   "d2h_bytes_per_step": int(odec.numel() * 2)}

    if rank != 0:
        barrier(world)
        return

    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # ---- f32 forward on its own (one head, M=N=4096, D=64), L2 flushed before each call
    f32 = None
    if world == 1:
        q32, k32, v32 = synth.attention_inputs(1, 1, 4096, 4096, 64, "f32", seed=0)
        q32, k32, v32 = (torch.from_numpy(x).to("cuda") for x in (q32, k32, v32))
        ws32_bytes = fa.fa_fwd_workspace_bytes(1, 1, 4096, 4096, 64, 0, fa.FA_F32)
        n32 = rotation(4 * q32.numel() * 4 + ws32_bytes)
        sets32 = [dict(q=q32.clone(), k=k32.clone(), v=v32.clone(), o=torch.empty_like(q32),
                       l=torch.empty((1, 1, 4096), dtype=torch.float32, device="cuda"),
                       ws=torch.zeros(max(ws32_bytes, 16), dtype=torch.uint8, device="cuda")) for _ in range(n32)]

        def run_f32(i):
            t = sets32[i]
            check(fa.fa_fwd_ws(t["q"], t["k"], t["v"], t["o"], t["l"], t["ws"] if ws32_bytes else None, ws32_bytes,
                               1, 1, 4096, 4096, 64, 0.125, 0, fa.FA_F32, stream), "fa_fwd_ws f32")

        t32, t32_iso = time_calls(torch, stream, flush, run_f32, n32, calls=30)
        check(fa.fa_last_status(stream), "f32 forward")
        del sets32
        tf32 = 4.0 * 4096 * 4096 * 64 / t32 / 1e12
        peak32 = peak_tf / 6.0
        f32 = {"config": "f32 forward, 1 head, M=N=4096, D=64, scale 0.125 through fa_fwd_ws (operands split into three bf16 parts, six products; key blocks of each query tile shared by 4 SMs, merged by the part that finishes last; the split prologue is inside the timed call)", "value": round(tf32, 2),
               "unit": "TFLOP/s", "us_per_call": round(t32 * 1e6, 1), "us_isolated": round(t32_iso * 1e6, 1),
               "l2": f"calls back to back over {n32} copies of the inputs (> 2 x L2); us_isolated: one call, L2 flushed",
               "roofline": {"kernel": "f32_presplit_kernel + fwd_f32ws_kernel<non-causal>", "bound": "tensor",
                            "achieved": round(tf32, 2), "peak": round(peak32, 1), "unit": "TFLOP/s",
                            "frac": round(tf32 / peak32, 4),
                            "peak_source": f"{peaks_src} bf16 burst / 6 products (each f32 product is six bf16 ones)",
                            "traffic": None}}

    # ---- grouped-query decode on its own: four query rows per K/V head of the same cache,
    # with the LSE (fa_decode_ex); the cache is larger than L2, so no flush is needed
    dec_rows = None
    if world == 1:
        R = 4
        qr = dev(synth.normal(np.random.default_rng(7), (d["B"], d["H"], R, d["D"]), "bf16"), "bf16")
        outr = torch.empty_like(qr)
        lser = torch.empty((d["B"], d["H"], R), dtype=torch.float32, device="cuda")
        wsr = torch.empty(fa.fa_decode_ex_workspace_bytes(d["B"], d["H"], R, d["D"], d["n_splits"]) // 4,
                          dtype=torch.float32, device="cuda")

        def run_rows():
            check(fa.fa_decode_ex(qr, kc, vc, outr, lser, wsr, d["B"], d["H"], R, d["N"], d["D"],
                                  1 / math.sqrt(d["D"]), d["n_splits"], fa.FA_BF16, stream), "fa_decode_ex")

        for _ in range(3):
            run_rows()
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(20):
            run_rows()
        b.record(stream)
        torch.cuda.synchronize()
        check(fa.fa_last_status(stream), "grouped-query decode")
        tr = a.elapsed_time(b) / 20 / 1e3
        gbs_r = dec_bytes() / tr / 1e9
        dec_rows = {"config": f"bf16 B{d['B']} H{d['H']} (K/V heads) x 4 query rows, N{d['N']} D{d['D']}, n_splits "
                              f"{d['n_splits']}, LSE written", "value": round(gbs_r, 1), "unit": "GB/s",
                    "us_per_call": round(tr * 1e6, 1),
                    "roofline": {"kernel": "decode_split_kernel<128,bf16,4 rows>", "bound": "hbm",
                                 "achieved": round(gbs_r, 1), "peak": peak_bw, "unit": "GB/s",
                                 "frac": round(gbs_r / peak_bw, 4), "peak_source": f"{peaks_src} copy bandwidth",
                                 "traffic": None}}

    configs = None
    if world == 1 and not args.no_configs:
        configs = bench_configs(fa, synth, dev, stream, flush, check, peak_tf, peak_bw, peaks_src)

    launches_per_step = 1 + (3 if have_bwd else 0) + 2
    traffic = load_traffic()
    if f32 is not None:
        f32["roofline"]["traffic"] = traffic.get("f32")
    line = {
        "metric": METRIC,
        "value": round(fwd_tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(t_step / K * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": "attention forward fp16 B4 H12 M=N=2048 D64 scale 0.125 non-causal "
                        "(+ backward same shape + decode bf16 B8 H32 N32768 D128 n_splits 64 per step)",
            "global_batch": FWD["B"] * world,
            "seq_len": FWD["N"],
            "head_dim": FWD["D"],
            "heads": FWD["H"],
            "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2: forward and backward rotate over 12 input sets (forward 12 x 25 MB, backward "
                  "12 x 51 MB, both > 2 x 129 MB), "
                  "calls back to back; decode cache 4.29 GB > L2; configs and f32: calls back to back over copies of their "
                  "inputs larger than 2 x L2 (us_isolated: one call with L2 flushed)",
        },
        "roofline": {
            "kernel": "fwd_d64_kernel<f16,non-causal>",
            "bound": "tensor",
            "achieved": round(fwd_tflops / world, 2),
            "peak": peak_tf,
            "unit": "TFLOP/s",
            "frac": round(fwd_tflops / world / peak_tf, 4),
            "peak_source": f"{peaks_src} bf16 burst (fp16 dense rate equals bf16)",
            "traffic": traffic.get("fwd"),
        },
        "decode": {
            "metric": "decode KV GB/s",
            "value": round(dec_gbs, 1),
            "unit": "GB/s",
            "ms_per_call": round(t_dec / K * 1e3, 4),
            "roofline": {
                "kernel": "decode_split_kernel<128,bf16>",
                "bound": "hbm",
                "achieved": round(dec_gbs / world, 1),
                "peak": peak_bw,
                "unit": "GB/s",
                "frac": round(dec_gbs / world / peak_bw, 4),
                "peak_source": f"{peaks_src} copy bandwidth",
                "traffic": traffic.get("decode"),
            },
            "e2e": dec_e2e,
        },
        "f32": f32,
        "decode_rows": dec_rows,
        "configs": configs,
        "backward": None if bwd_tflops is None else {
            "value": round(bwd_tflops, 2), "unit": "TFLOP/s", "ms_per_call": round(t_bwd / K * 1e3, 4),
            "flops": "2.5 x forward",
            # the whole call (delta, the fused dK/dV/dQ pass, dQ's conversion) against the tensor
            # peak; traffic is the fused kernel's from one ncu capture of this workload
            "roofline": {"kernel": "bwd_fused64_kernel<f16,non-causal> (+ delta, dQ conversion)",
                         "bound": "tensor", "achieved": round(bwd_tflops / world, 2), "peak": peak_tf,
                         "unit": "TFLOP/s", "frac": round(bwd_tflops / world / peak_tf, 4),
                         "peak_source": f"{peaks_src} bf16 burst (fp16 dense rate equals bf16)",
                         "traffic": traffic.get("bwd_fused")}},
        "e2e": {"value": round(e2e_tflops, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": launches_per_step * K,
        "clocks": clk.summary(clock_phases),
        "wall_s": round(wall, 3),
        # the main step's parts cut into chunks (microseconds per call in each), the host's load
        # average before the timed region and other processes on this GPU: context for a slow run
        "chunks_us_per_call": {k: [round(a.elapsed_time(b) * 1e3 / max(1, j - i), 2)
                                   for (i, a), (j, b) in zip(m, m[1:] + [(args.steps, end)])]
                               for k, (m, end) in chunk_ev.items()},
        "host_load": round(load_before, 2) if load_before is not None else None,
        "other_gpu_processes": foreign,
    }
    if not args.no_cpu_baseline and world == 1:
        tf, heads, secs, thr = oracle_forward_sample(args.cpu_seconds)
        gbs, dheads, dsecs = oracle_decode_sample(max(2.0, args.cpu_seconds / 4))
        line["cpu_baseline"] = {
            "value": round(tf, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
            "sample": f"fp64 oracle forward on {heads} whole heads (M=N=2048, D=64) of the forward workload, "
                      f"{secs:.1f} s; decode oracle {round(gbs, 2)} GB/s on {dheads} heads of the cache",
        }
    barrier(world)
    print(json.dumps(line), flush=True)


def bench_configs(fa, synth, dev, stream, flush, check, peak_tf, peak_bw, peaks_src, calls=20):
    """Every configuration of the workload list, each timed on its own. `value` and `us_per_call`:
    calls back to back over enough copies of the inputs (with their outputs and workspace) that
    together they exceed twice L2, between one pair of CUDA events, as the headline is timed.
    `us_isolated`: one call between two events with L2 flushed before it (the event pair's own
    ~2 us and a cold L2 included). Decode: its 4.29 GB cache is larger than L2, calls back to back."""
    import torch

    out = {}

    def nbytes(*ts):
        return sum(t.numel() * t.element_size() for t in ts)

    def tensor_entry(desc, flops, t, t_iso, n_sets, kernel, peak=peak_tf, peak_note=None):
        tf = flops / t / 1e12
        return {"config": desc, "value": round(tf, 2), "unit": "TFLOP/s", "us_per_call": round(t * 1e6, 2),
                "us_isolated": round(t_iso * 1e6, 2),
                "l2": f"calls back to back over {n_sets} copies of the inputs (> 2 x L2); us_isolated: one call, "
                      f"L2 flushed",
                "roofline": {"kernel": kernel, "bound": "tensor", "achieved": round(tf, 2), "peak": round(peak, 1),
                             "unit": "TFLOP/s", "frac": round(tf / peak, 4),
                             "peak_source": peak_note or f"{peaks_src} bf16 burst (fp16 dense rate equals bf16)",
                             "traffic": None}}

    def attn(B, H, M, N, D, dtype, seed, with_dout=False):
        arrs = synth.attention_inputs(B, H, M, N, D, dtype, seed=seed, with_dout=with_dout)
        return [dev(a, dtype) for a in arrs]

    code = {"f32": fa.FA_F32, "f16": fa.FA_F16, "bf16": fa.FA_BF16}

    def forward_entry(name, B, H, M, N, D, dtype, causal, scale, desc, kernel):
        q, k, v = attn(B, H, M, N, D, dtype, seed=M + N)
        nb = fa.fa_fwd_workspace_bytes(B, H, M, N, D, causal, code[dtype])
        n = rotation(2 * nbytes(q) + nbytes(k, v) + B * H * M * 4 + nb)
        sets = [dict(q=q.clone(), k=k.clone(), v=v.clone(), o=torch.empty_like(q),
                     lse=torch.empty((B, H, M), dtype=torch.float32, device="cuda"),
                     ws=torch.zeros(max(nb, 16), dtype=torch.uint8, device="cuda")) for _ in range(n)]

        def run(i):
            t = sets[i]
            check(fa.fa_fwd_ws(t["q"], t["k"], t["v"], t["o"], t["lse"], t["ws"] if nb else None, nb, B, H, M, N, D,
                               scale, causal, code[dtype], stream), name)

        t, t_iso = time_calls(torch, stream, flush, run, n, calls)
        check(fa.fa_last_status(stream), name)
        flops = 4.0 * B * H * M * N * D / (2 if causal else 1)
        peak, note = peak_tf, None
        if dtype == "f32":
            peak = peak_tf / 6.0
            note = f"{peaks_src} bf16 burst / 6 products (each f32 product is six bf16 ones)"
        out[name] = tensor_entry(desc, flops, t, t_iso, n, kernel, peak, note)

    # fp16 forward, B4 H12 D64, M = N over {512, 1024, 2048}; bf16 and causal at 2048
    for n in (512, 1024, 2048):
        forward_entry(f"fwd_f16_N{n}", 4, 12, n, n, 64, "f16", False, 0.125,
                      f"fp16 forward B4 H12 M=N={n} D64 scale 0.125 non-causal (fa_fwd_ws)",
                      "fwd_d64_kernel<f16,non-causal>")
    forward_entry("fwd_bf16_N2048", 4, 12, 2048, 2048, 64, "bf16", False, 0.125,
                  "bf16 forward B4 H12 M=N=2048 D64 scale 0.125 non-causal", "fwd_d64_kernel<bf16,non-causal>")
    forward_entry("fwd_f16_N2048_causal", 4, 12, 2048, 2048, 64, "f16", True, 0.125,
                  "fp16 forward B4 H12 M=N=2048 D64 scale 0.125 causal (FLOP halved)", "fwd_d64_kernel<f16,causal>")
    # FP8 forward (E4M3 operands, fp16 I/O) at the fp16 workload's largest shape: the whole call
    # (three quantisation launches, then the attention kernel), against the fp8 tensor peak
    q, k, v = attn(4, 12, 2048, 2048, 64, "f16", seed=2048)
    signs = torch.from_numpy(synth.hadamard_signs(64, 0)).cuda()
    nb = fa.fa_fwd_fp8_workspace_bytes(4, 12, 2048, 2048, 64)
    n = rotation(2 * nbytes(q) + nbytes(k, v) + nb)
    sets = [dict(q=q.clone(), k=k.clone(), v=v.clone(), o=torch.empty_like(q),
                 lse=torch.empty((4, 12, 2048), dtype=torch.float32, device="cuda"),
                 ws=torch.empty(nb, dtype=torch.uint8, device="cuda")) for _ in range(n)]
    for causal in (False, True):
        def run(i):
            t = sets[i]
            check(fa.fa_fwd_fp8(t["q"], t["k"], t["v"], t["o"], t["lse"], signs, t["ws"], nb, 4, 12, 2048, 2048, 64,
                                0.125, causal, fa.FA_F16, stream), "fa_fwd_fp8")

        t, t_iso = time_calls(torch, stream, flush, run, n, calls)
        check(fa.fa_last_status(stream), "fa_fwd_fp8")
        tag = "causal" if causal else "noncausal"
        out[f"fwd_fp8_N2048_{tag}"] = tensor_entry(
            f"FP8 forward (E4M3 operands after the Hadamard-times-sign transform, per-block scales; fp16 I/O) "
            f"B4 H12 M=N=2048 D64 scale 0.125 {tag}: quantisation + attention per call",
            4.0 * 4 * 12 * 2048 * 2048 * 64 / (2 if causal else 1), t, t_iso, n,
            f"fwd_fp8_kernel<f16,{tag}> (+ fp8 quantisation)",
            peak_tf * 2.0, f"{peaks_src} bf16 burst x nominal fp8/bf16 (4.5/2.25)")
    del sets
    # f32, one head, 256^2 (the 4096^2 case is the main line's `f32` object)
    forward_entry("fwd_f32_N256", 1, 1, 256, 256, 64, "f32", False, 0.125,
                  "f32 forward 1 head Nq=Nk=256 D64 scale 0.125 (fa_fwd_ws: three bf16 parts, six products)",
                  "f32_presplit_kernel + fwd_f32ws_kernel<non-causal>")
    # fp16 forward + backward, Z1 H2 N1024 D64, sm_scale 0.5, causal and not
    for causal in (False, True):
        tag = "causal" if causal else "noncausal"
        forward_entry(f"cfg4_fwd_{tag}", 1, 2, 1024, 1024, 64, "f16", causal, 0.5,
                      f"fp16 forward Z1 H2 N1024 D64 sm_scale 0.5 {tag}", f"fwd_d64_kernel<f16,{tag}>")
    for causal in (False, True):
        for M, B, H, name0 in ((1024, 1, 2, "cfg4"), (2048, 4, 12, "bwd")):
            if name0 == "bwd" and causal:
                continue
            q, k, v, do = attn(B, H, M, M, 64, "f16", seed=20, with_dout=True)
            o = torch.empty_like(q)
            lse = torch.empty((B, H, M), dtype=torch.float32, device="cuda")
            check(fa.fa_fwd(q, k, v, o, lse, B, H, M, M, 64, 0.5, causal, fa.FA_F16, stream), "fa_fwd")
            nb = fa.fa_bwd_ws_workspace_bytes(B, H, M, 64)
            n = rotation(8 * nbytes(q) + nbytes(lse) + nb)
            sets = [dict(q=q.clone(), k=k.clone(), v=v.clone(), o=o.clone(), do=do.clone(), lse=lse.clone(),
                         dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
                         ws=torch.empty(nb, dtype=torch.uint8, device="cuda"),
                         dws=torch.empty((B, H, M), dtype=torch.float32, device="cuda")) for _ in range(n)]
            flops = 2.5 * 4.0 * B * H * M * M * 64 / (2 if causal else 1)
            tag = "causal" if causal else "noncausal"

            def run_ws(i):
                t = sets[i]
                check(fa.fa_bwd_ws(t["q"], t["k"], t["v"], t["o"], t["do"], t["lse"], t["dq"], t["dk"], t["dv"],
                                   t["ws"], nb, B, H, M, M, 64, 0.5, causal, fa.FA_F16, stream), "fa_bwd_ws")

            def run3(i):
                t = sets[i]
                check(fa.fa_bwd(t["q"], t["k"], t["v"], t["o"], t["do"], t["lse"], t["dq"], t["dk"], t["dv"],
                                t["dws"], B, H, M, M, 64, 0.5, causal, fa.FA_F16, stream), "fa_bwd")

            t, t_iso = time_calls(torch, stream, flush, run_ws, n, calls)
            desc = f"fp16 backward B{B} H{H} N{M} D64 scale 0.5 {tag}"
            out[f"{name0}_bwd_fused_{tag}"] = tensor_entry(
                desc + " through fa_bwd_ws (delta, fused dK/dV/dQ, dQ conversion; FLOP = 2.5 x forward)", flops, t,
                t_iso, n, f"bwd_fused64_kernel<f16,{tag}>")
            # automatic schedule: dK/dV and dQ on CTA pairs for non-causal calls with fewer key
            # tiles than SMs (the Z1 H2 case), single CTAs otherwise
            t, t_iso = time_calls(torch, stream, flush, run3, n, calls)
            paired = not causal and B * H * (M // 128) < 152
            kern3 = "bwd_dkdv64_pair_kernel + bwd_dq64_pair_kernel" if paired else "bwd_dkdv64_kernel + bwd_dq_kernel"
            out[f"{name0}_bwd_3kernels_{tag}"] = tensor_entry(
                desc + " through fa_bwd (delta, dK/dV, dQ kernels; FLOP = 2.5 x forward)", flops, t, t_iso, n,
                f"{kern3}<f16,{tag}>")
            if not causal:  # the other form, forced
                with fa.schedule(fa.FA_SCHED_BWD_PAIR, 0 if paired else 1):
                    t, t_iso = time_calls(torch, stream, flush, run3, n, calls)
                other = "single_cta" if paired else "pair"
                kern_o = "bwd_dkdv64_kernel + bwd_dq_kernel" if paired else "bwd_dkdv64_pair_kernel + bwd_dq64_pair_kernel"
                out[f"{name0}_bwd_3kernels_{other}_{tag}"] = tensor_entry(
                    desc + f" through fa_bwd with the dK/dV and dQ kernels forced to {other.replace('_', ' ')} "
                    f"(FLOP = 2.5 x forward)", flops, t, t_iso, n, f"{kern_o}<f16,{tag}>")
            check(fa.fa_last_status(stream), "backward configurations")
            del sets
    # bf16 decode B8 H32 N32768 D128 at n_splits 16 and 256 (64 is the main line's)
    d = DEC
    qdec = dev(synth.decode_query(d["B"], d["H"], d["D"], d["dtype"], 0), "bf16")
    kc = torch.empty((d["B"], d["H"], d["N"], d["D"]), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    g = torch.Generator(device="cuda").manual_seed(0)
    kc.normal_(generator=g)
    vc.normal_(generator=g)
    odec = torch.empty_like(qdec)
    for ns in (16, 256):
        ws = torch.empty(fa.fa_decode_workspace_bytes(d["B"], d["H"], d["D"], ns) // 4, dtype=torch.float32,
                         device="cuda")

        def run(i):
            check(fa.fa_decode(qdec, kc, vc, odec, ws, d["B"], d["H"], d["N"], d["D"], 1 / math.sqrt(d["D"]), ns,
                               fa.FA_BF16, stream), "fa_decode")

        t, _ = time_calls(torch, stream, flush, run, 1, calls, isolated=1)
        gbs = dec_bytes() / t / 1e9
        out[f"decode_splits{ns}"] = {
            "config": f"bf16 decode B8 H32 N32768 D128 n_splits {ns} (cache 4.29 GB > L2, calls back to back)",
            "value": round(gbs, 1), "unit": "GB/s", "us_per_call": round(t * 1e6, 2),
            "roofline": {"kernel": "decode_split_kernel<128,bf16> + decode_combine_kernel", "bound": "hbm",
                         "achieved": round(gbs, 1), "peak": peak_bw, "unit": "GB/s", "frac": round(gbs / peak_bw, 4),
                         "peak_source": f"{peaks_src} copy bandwidth", "traffic": None}}
    check(fa.fa_last_status(stream), "decode configurations")
    del kc, vc
    torch.cuda.empty_cache()
    return out


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, when it matches the kernels."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            return json.load(f)
    except Exception:
        return {}


# ---------------------------------------------------------- reference arm
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per_step = max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_forward_sample(per_step / 4, max_heads=1)
    vals, secs, heads = [], 0.0, 0
    for _ in range(args.steps):
        tf, h, s, thr = oracle_forward_sample(per_step)
        vals.append(tf)
        secs += s
        heads += h
    value = statistics.median(vals)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "attention forward fp16 inputs B4 H12 M=N=2048 D64 scale 0.125 non-causal, "
                               "sampled whole heads per step", "global_batch": FWD["B"], "seq_len": FWD["N"],
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"{heads} whole heads over {args.steps} steps ({secs:.1f} s)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PROFILE_CASES = {
    # inputs larger than L2 (129 MB) so DRAM counters mean something, a few GB at most
    "fwd": dict(B=16, H=16, M=4096, N=4096, D=64, dtype="f16"),     # Q/K/V 0.4 GB
    "fwd_bench": dict(B=4, H=12, M=2048, N=2048, D=64, dtype="f16"),  # the headline workload itself
    "fwd_fp8": dict(B=4, H=12, M=2048, N=2048, D=64, dtype="f16"),  # FP8 forward at the same shape
    "decode": dict(B=8, H=8, N=32768, D=128, n_splits=64, dtype="bf16"),  # K/V 1.07 GB
    "bwd": dict(B=8, H=16, M=2048, N=2048, D=64, dtype="f16"),  # Q/K/V/O/dO 0.34 GB (fused pass)
    "bwd3": dict(B=8, H=16, M=2048, N=2048, D=64, dtype="f16"),  # the same through the three kernels
    "decode_rows": dict(B=8, H=8, N=32768, D=128, n_splits=64, rows=4, dtype="bf16"),  # K/V 1.07 GB
    "f32": dict(B=1, H=1, M=4096, N=4096, D=64, dtype="f32"),  # the f32 workload (L2-resident, 3 MB)
    "f32_big": dict(B=4, H=12, M=2048, N=2048, D=64, dtype="f32"),  # Q/K/V 100 MB, split planes 200 MB
}


def run_profile(kind: str, launches: int = 5):
    """A few launches of one kernel on its profiling case (for ncu); prints nothing else."""
    import torch

    from exact_attention_gb300 import build as fa_build
    fa_build.build()
    import exact_attention_gb300 as fa
    torch.cuda.set_device(0)
    g = torch.Generator(device="cuda").manual_seed(0)
    c = PROFILE_CASES[kind]
    if kind in ("fwd", "fwd_bench"):
        shp = (c["B"], c["H"], c["M"], c["D"])
        q = torch.randn(shp, generator=g, device="cuda").half()
        k = torch.randn(shp, generator=g, device="cuda").half()
        v = torch.randn(shp, generator=g, device="cuda").half()
        o = torch.empty_like(q)
        lse = torch.empty(shp[:3], device="cuda")
        for _ in range(launches):
            fa.forward(q, k, v, 0.125, False, out=o, lse=lse)
    elif kind in ("f32", "f32_big"):
        shp = (c["B"], c["H"], c["M"], c["D"])
        q, k, v = (torch.randn(shp, generator=g, device="cuda") for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty(shp[:3], device="cuda")
        for _ in range(launches):
            fa.forward(q, k, v, 0.125, False, out=o, lse=lse)
    elif kind == "fwd_fp8":
        shp = (c["B"], c["H"], c["M"], c["D"])
        q, k, v = (torch.randn(shp, generator=g, device="cuda").half() for _ in range(3))
        signs = torch.where(torch.rand(c["D"], generator=g, device="cuda") < 0.5, -1, 1).to(torch.int8)
        ws = None
        for _ in range(launches):
            _, _, ws = fa.forward_fp8(q, k, v, 0.125, False, signs, workspace=ws)
    elif kind in ("bwd", "bwd3"):
        shp = (c["B"], c["H"], c["M"], c["D"])
        q, k, v, do = (torch.randn(shp, generator=g, device="cuda").half() for _ in range(4))
        o, lse = fa.forward(q, k, v, 0.125, False)
        for _ in range(launches):
            fa.backward(q, k, v, o, do, lse, 0.125, False, fused=kind == "bwd")
    else:
        q = torch.randn((c["B"], c["H"], c.get("rows", 1), c["D"]), generator=g, device="cuda").bfloat16()
        kc = torch.randn((c["B"], c["H"], c["N"], c["D"]), generator=g, device="cuda").bfloat16()
        vc = torch.randn_like(kc)
        out = torch.empty_like(q)
        for _ in range(launches):
            res = fa.decode(q, kc, vc, 1 / math.sqrt(c["D"]), c["n_splits"], out=out,
                            lse=True if "rows" in c else None)
            out = res[0]
    torch.cuda.synchronize()
    s = fa.fa_last_status()
    if s != fa.FA_OK:
        raise RuntimeError(fa.fa_last_error_message())
    print(f"profile case {kind}: {c}, {launches} launches ok")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--decode-e2e", action="store_true", default=True)
    ap.add_argument("--no-decode-e2e", dest="decode_e2e", action="store_false")
    ap.add_argument("--profile", choices=sorted(PROFILE_CASES), help="run a few launches of one kernel and exit")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-configuration sweep")
    args = ap.parse_args()
    if args.profile:
        run_profile(args.profile)
        return
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
