"""Benchmark of the exact-attention hot path on GB300 (one JSON line on rank 0).

A step is one pass of the hot path over synthetic inputs already resident in
device memory:
  * forward, fp16, B=4, H=12, M=N=2048, D=64, scale 0.125, non-causal
    (the workload the headline TFLOP/s is quoted on); L2 is flushed before it;
  * backward at the same shape, when the library provides it;
  * flash decoding, bf16, B=8, H=32, N=32768, D=128, n_splits=64 (the K/V cache,
    4.29 GB, is far larger than L2).
Each part is timed with CUDA events on the stream it runs on. `value` is the
forward's TFLOP/s (4*B*H*M*N*D per call); the decode GB/s (K+V bytes read per
call) is reported in the `decode` object. `e2e` repeats the forward through the
C ABI on pinned host buffers (fa_fwd_host: the inputs copied in and O/LSE copied
back inside the timed region, overlapped with the kernels chunk by chunk).

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
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


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
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons while running."""

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
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        time.sleep(0.3)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
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
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


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
    q, k, v, do = synth.attention_inputs(c["B"], c["H"], c["M"], c["N"], c["D"], c["dtype"], seed=rank,
                                         with_dout=True)
    qd, kd, vd, dod = dev(q, "f16"), dev(k, "f16"), dev(v, "f16"), dev(do, "f16")
    od = torch.empty_like(qd)
    lse = torch.empty((c["B"], c["H"], c["M"]), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
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

    def run_fwd():
        check(fa.fa_fwd_ws(qd, kd, vd, od, lse, fws if fws_bytes else None, fws_bytes, *BHMND, c["scale"], c["causal"],
                           fa.FA_F16, stream), "fa_fwd_ws")

    have_bwd = True

    def run_bwd():
        nonlocal have_bwd
        if not have_bwd:
            return
        s = fa.fa_bwd_ws(qd, kd, vd, od, dod, lse, dq, dk, dv, bws, bws_bytes, *BHMND, c["scale"], c["causal"],
                         fa.FA_F16, stream)
        if s == fa.FA_ERR_UNSUPPORTED:
            have_bwd = False
            return
        check(s, "fa_bwd_ws")

    def run_dec():
        check(fa.fa_decode(qdec, kc, vc, odec, ws, d["B"], d["H"], d["N"], d["D"], 1 / math.sqrt(d["D"]),
                           d["n_splits"], fa.FA_BF16, stream), "fa_decode")

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def step(record):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        run_fwd()
        e1.record(stream)
        flush.zero_()
        e2, e3 = ev(), ev()
        e2.record(stream)
        run_bwd()
        e3.record(stream)
        e4, e5 = ev(), ev()
        e4.record(stream)
        run_dec()
        e5.record(stream)
        if record is not None:
            record.append((e0, e1, e2, e3, e4, e5))

    for _ in range(args.warmup):
        step(None)
    check(fa.fa_last_status(stream), "warm-up")
    torch.cuda.synchronize()

    recs = []
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        w0 = ev()
        w0.record(stream)
        for _ in range(args.steps):
            step(recs)
        w1 = ev()
        w1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - t0
    check(fa.fa_last_status(stream), "timed steps")
    t_fwd = sum(r[0].elapsed_time(r[1]) for r in recs) / 1e3
    t_bwd = sum(r[2].elapsed_time(r[3]) for r in recs) / 1e3
    t_dec = sum(r[4].elapsed_time(r[5]) for r in recs) / 1e3
    t_step = w0.elapsed_time(w1) / 1e3  # includes the untimed L2 flushes
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
    # ---- f32 forward on its own (one head, M=N=4096, D=64, 3xTF32), L2 flushed before each call
    f32 = None
    if world == 1:
        q32, k32, v32 = synth.attention_inputs(1, 1, 4096, 4096, 64, "f32", seed=0)
        q32, k32, v32 = (torch.from_numpy(x).to("cuda") for x in (q32, k32, v32))
        o32 = torch.empty_like(q32)
        l32 = torch.empty((1, 1, 4096), dtype=torch.float32, device="cuda")

        ws32_bytes = fa.fa_fwd_workspace_bytes(1, 1, 4096, 4096, 64, 0, fa.FA_F32)
        ws32 = torch.zeros(max(ws32_bytes, 16), dtype=torch.uint8, device="cuda")

        def run_f32():
            check(fa.fa_fwd_ws(q32, k32, v32, o32, l32, ws32 if ws32_bytes else None, ws32_bytes, 1, 1, 4096, 4096, 64,
                               0.125, 0, fa.FA_F32, stream), "fa_fwd_ws f32")

        for _ in range(3):
            run_f32()
        recs32 = []
        for _ in range(30):
            flush.zero_()
            a, b = ev(), ev()
            a.record(stream)
            run_f32()
            b.record(stream)
            recs32.append((a, b))
        torch.cuda.synchronize()
        check(fa.fa_last_status(stream), "f32 forward")
        t32 = sum(a.elapsed_time(b) for a, b in recs32) / len(recs32) / 1e3
        tf32 = 4.0 * 4096 * 4096 * 64 / t32 / 1e12
        peak32 = peak_tf * 1.1 / 2.25 / 3.0
        f32 = {"config": "f32 forward, 1 head, M=N=4096, D=64, scale 0.125 (3xTF32; key blocks of each query tile shared by 4 SMs, merged by the part that finishes last)", "value": round(tf32, 2),
               "unit": "TFLOP/s", "us_per_call": round(t32 * 1e6, 1),
               "roofline": {"kernel": "fwd_f32_kernel<non-causal>", "bound": "tensor", "achieved": round(tf32, 2),
                            "peak": round(peak32, 1), "unit": "TFLOP/s", "frac": round(tf32 / peak32, 4),
                            "peak_source": f"{peaks_src} bf16 burst x nominal tf32/bf16 (1.1/2.25) / 3 products",
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

    launches_per_step = 1 + (3 if have_bwd else 0) + 2
    traffic = load_traffic()
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
            "l2": "flushed (512 MB write) before the forward and the backward; decode cache 4.29 GB > L2",
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
        "clocks": clk.summary(),
        "wall_s": round(wall, 3),
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
    "decode": dict(B=8, H=8, N=32768, D=128, n_splits=64, dtype="bf16"),  # K/V 1.07 GB
    "bwd": dict(B=8, H=16, M=2048, N=2048, D=64, dtype="f16"),  # Q/K/V/O/dO 0.34 GB (fused pass)
    "bwd3": dict(B=8, H=16, M=2048, N=2048, D=64, dtype="f16"),  # the same through the three kernels
    "decode_rows": dict(B=8, H=8, N=32768, D=128, n_splits=64, rows=4, dtype="bf16"),  # K/V 1.07 GB
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
    if kind == "fwd":
        shp = (c["B"], c["H"], c["M"], c["D"])
        q = torch.randn(shp, generator=g, device="cuda").half()
        k = torch.randn(shp, generator=g, device="cuda").half()
        v = torch.randn(shp, generator=g, device="cuda").half()
        o = torch.empty_like(q)
        lse = torch.empty(shp[:3], device="cuda")
        for _ in range(launches):
            fa.forward(q, k, v, 0.125, False, out=o, lse=lse)
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
