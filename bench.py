"""Benchmark: FP8 attention forward TFLOP/s including quantisation.

One step = the whole hot path over one batch of synthetic input resident in
HBM: rotate-and-quantise Q, K and V (one launch), then the FP8 forward
(work-list, V-reference and attention launches). FLOPs = 4 B H N^2 d, halved
for causal workloads. The default workload is the FlashAttention-3 headline
shape: batch 2, 32 heads, sequence 8192, head_dim 128, non-causal, 0.1%
N(0, 10) outliers, E4M3 with 128-token block scales and a 128-point Hadamard
rotation of Q and K.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs under torch.distributed.run, one rank per GPU; every rank runs its
own replica of the workload (weak scaling, no collective on the data path).
`--impl reference` times the CPU oracle (quantiser + quantised-operand
emulation) on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "FP8 attn fwd TFLOP/s incl. quant (hd128, s8192); RMSE vs FP64 oracle"
UNIT = "TFLOP/s"
E4M3, ROW, COL = 0, 1, 2


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return None


def fp8_peak():
    """Dense FP8 tensor peak: measured bf16 GEMM burst x the nominal fp8/bf16
    ratio (4.5 / 2.25 PFLOP/s); the recipe's fallback when no measurement."""
    pk = load_peaks()
    if pk and pk.get("bf16_tflops"):
        return 2.0 * float(pk["bf16_tflops"]), "measured bf16 burst x2 (nominal fp8/bf16 ratio)"
    return 2.0 * 1900.0, "fallback 1.9 PFLOP/s bf16 x2"


def recorded_traffic(args, name, sources, key="bytes_per_launch"):
    """DRAM bytes from a committed ncu summary (profiles/<name>), or None when the
    kernel source changed since the capture or the workload differs (the
    captures are of workload 2 at full size, hardware exp2, E4M3)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name)
    if (args.workload != 2 or args.heads or args.seqlen or args.batch or args.exact or args.nvfp4
            or args.exp_mode != "hw" or args.no_rotate or not os.path.exists(path)):
        return None
    kv = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            a, b = line.split(":", 1)
            kv[a.strip()] = b.strip()
    h = hashlib.sha256()
    for f in sources:
        h.update(open(os.path.join(ROOT, "precision_attention_gb300", "csrc", f), "rb").read())
    if h.hexdigest()[:16] != kv.get("source_sha256_prefix"):
        return None
    return float(kv[key])


def attn_traffic(args):
    if args.sched != "static":   # the record is of the static-order kernel
        return None
    return recorded_traffic(args, "attn_fwd_traffic.txt", ("attn_fwd.cu", "ptx.cuh", "params.h"))


def quant_traffic(args):
    """DRAM bytes of one step's quantisation (the one launch for Q, K and V)."""
    if args.quant_split:
        return None
    return recorded_traffic(args, "quant_traffic.txt", ("quant.cu", "ptx.cuh", "params.h"), "bytes_per_step")


def hbm_peak():
    pk = load_peaks()
    if pk and pk.get("hbm_gbs"):
        return float(pk["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"pa_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5], parts[6], parts[7], parts[8]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        busy = [r for r in rows if r[0] > 0.5 * r[1]] or rows
        reasons = []
        for name, col in (("hw_slowdown", 2), ("hw_thermal_slowdown", 3), ("sw_thermal_slowdown", 4),
                          ("sw_power_cap", 5)):
            if any(r[col].lower() == "active" for r in rows):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
def max_over_ranks(values, device):
    """Element-wise maximum of per-rank timings (the slowest rank sets the job's
    time); a no-op without an initialised process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(world, flops_per_rank, ms_per_step):
    """Whole-job TFLOP/s: every rank runs its own replica (weak scaling), so the
    job does world x flops_per_rank in the slowest rank's step time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


# ---------------------------------------------------------------------------
def quant_bytes(T, H, d, in_elt, mx, block, nd, nv=False):
    """Algorithmic HBM bytes of one step's quantisation (Q, K, V): inputs read,
    codes written, scales written."""
    n = T * H * d
    if nv:   # NVFP4 Q, K: half a byte per element, an E4M3 scale per 16, fp32 per 128 tokens; E4M3 V
        blocks = H * ((T + 127) // 128 + nd) * 4
        return 3 * n * in_elt + 2 * (n // 2 + n // 16 + blocks) + n + blocks
    scales = (3 * H * (T + 127) // 128 * 512 / 4) if mx else 3 * H * ((T + block - 1) // block + nd) * 4
    return 3 * n * (in_elt + 1) + scales


def measure_fp8_peak(torch, dev):
    """Dense E4M3 GEMM throughput of the vendor library (torch._scaled_mm, i.e.
    cuBLASLt) at 8192^3, best of 10: the measured FP8 tensor peak the attention
    kernel is compared with (a reference number, not part of the path)."""
    try:
        N = 8192
        a = torch.randn(N, N, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(N, N, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.tensor(1.0, device=dev)
        for _ in range(5):
            torch._scaled_mm(a, b, one, one, out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(10):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch._scaled_mm(a, b, one, one, out_dtype=torch.bfloat16)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * N ** 3 / (best * 1e-3) / 1e12
    except Exception:   # the library's FP8 GEMM unavailable: report no number
        return None


def time_workload(args, pa, torch, dev, wid, exact, steps, warmup, clocks_idx=None, keep=False, exp_mode=0,
                  nv=False):
    """Time `steps` whole steps (quantise Q, K, V, then the FP8 forward) of one
    workload after `warmup` untimed ones; inputs resident in HBM. Returns the
    timings (and, with keep, the device tensors for the end-to-end leg)."""
    w = workloads.WORKLOADS[wid]
    hd = args.heads if wid == args.workload else None
    sl = args.seqlen if wid == args.workload else None
    bt = args.batch if wid == args.workload else None
    inp = workloads.make(wid, heads=hd, seqlen=sl, batch=bt)
    T, H, d = inp.q.shape
    cu_np = inp.cu_seqlens
    nd = len(cu_np) - 1
    causal, mx, seed = w.causal, w.mx, w.hadamard_seed
    rot = not args.no_rotate
    if exact and not causal:
        raise SystemExit("--exact needs a causal workload")
    flops = workloads.attention_flops(cu_np, H, d, causal)
    in_dt = torch.float32 if w.in_dtype == "f32" else torch.bfloat16
    q_h, k_h, v_h = (torch.from_numpy(np.ascontiguousarray(a)).to(in_dt).pin_memory() for a in (inp.q, inp.k, inp.v))
    q, k, v = (x.to(dev) for x in (q_h, k_h, v_h))
    cu = torch.from_numpy(cu_np.astype(np.int32)).to(dev)
    ws = pa.workspace(T, H, d, nd, dev)
    if nv:   # mixed NVFP4 / FP8: NVFP4 Q and K, E4M3 V in 128-token blocks
        if mx or exact:
            raise SystemExit("--nvfp4 takes an E4M3 workload without --exact")
        lq, lk, lv, blk = pa.ATTN_NVFP4, pa.ATTN_NVFP4, E4M3, 128
    elif mx:   # causal-exact: one V exponent per token
        lq, lk, lv, blk = ROW, ROW, (pa.ATTN_MX_TOKEN if exact else COL), 32
    else:
        lq = lk = lv = E4M3
        blk = 1 if exact else w.block
    Q = pa.empty_qtensor(T, H, d, nd, lq, blk, device=dev)
    K = pa.empty_qtensor(T, H, d, nd, lk, blk, device=dev)
    V = pa.empty_qtensor(T, H, d, nd, lv, blk, device=dev)
    o = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((H, T), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    attn_ev, step_ev = [], []

    def quantise(qi, ki, vi):
        # one launch for the three operands (FLAMIA section 4.3); --quant-split: one per tensor
        if args.quant_split:
            pa.attn_quantize(qi, cu, lq, blk, rot, seed, ws=ws, out=Q, stream=stream)
            pa.attn_quantize(ki, cu, lk, blk, rot, seed, ws=ws, out=K, stream=stream)
            pa.attn_quantize(vi, cu, lv, blk, False, 0, ws=ws, out=V, stream=stream)
        else:
            pa.attn_quantize_qkv(qi, ki, vi, cu, lq, blk, lv, blk, rot, seed, ws=ws, outs=(Q, K, V), stream=stream)

    def step(record=False):
        if record:
            es = torch.cuda.Event(enable_timing=True)
            es.record(stream)
            step_ev.append(es)
        quantise(q, k, v)
        if record:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
        pa.attn_fp8_fwd_ex(Q, K, V, cu, causal, exact, 0.0, exp_mode, ws=ws, out=o, lse=lse, stream=stream)
        if record:
            e1.record(stream)
            attn_ev.append((e0, e1))

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    st, flags = pa.attn_read_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {pa.attn_status_string(st)} flags {flags:#x}")
    dist = None
    if args.world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(clocks_idx) if clocks_idx is not None else None
    if sampler:
        sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step(record=True)
    t1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = sampler.stop() if sampler else None
    ms_total = t0.elapsed_time(t1)
    attn_ms = [a_.elapsed_time(b_) for a_, b_ in attn_ev]
    ends = step_ev[1:] + [t1]
    step_ms = [a_.elapsed_time(b_) for a_, b_ in zip(step_ev, ends)]
    st, flags = pa.attn_read_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {pa.attn_status_string(st)} flags {flags:#x}")
    r = {"inp": inp, "flops": flops, "ms_step": ms_total / steps, "attn_ms": float(np.mean(attn_ms)),
         "stats": {name: {"median": float(np.median(x)), "min": float(np.min(x)), "p90": float(np.percentile(x, 90))}
                   for name, x in (("step_ms", step_ms), ("attn_ms", attn_ms))},
         "clocks": clk, "T": T, "H": H, "d": d, "nd": nd, "mx": mx, "causal": causal, "exact": exact,
         "quant_bytes": quant_bytes(T, H, d, 4 if w.in_dtype == "f32" else 2, mx, blk, nd, nv)}
    r["quant_ms"] = r["ms_step"] - r["attn_ms"]
    if keep:
        r.update(dict(q=q, k=k, v=v, q_h=q_h, k_h=k_h, v_h=v_h, cu=cu, ws=ws, Q=Q, K=K, V=V, o=o, lse=lse,
                      lq=lq, lk=lk, lv=lv, blk=blk, rot=rot, seed=seed, stream=stream, quantise=quantise))
    else:
        r["acc"] = None if args.no_accuracy else accuracy_sample(inp, wid, q, k, v, cu, o, pa, torch)
        del q, k, v, Q, K, V, o, lse, ws
        torch.cuda.empty_cache()
    return r


def gpu_arm(args, rank, world, local_rank):
    import torch
    import precision_attention_gb300 as pa

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    args.world = world
    pa.attn_set_schedule(pa.ATTN_SCHED_TICKET if args.sched == "ticket" else pa.ATTN_SCHED_STATIC)
    w = workloads.WORKLOADS[args.workload]
    r = time_workload(args, pa, torch, dev, args.workload, bool(args.exact), args.steps, args.warmup,
                      clocks_idx=local_rank, keep=True, exp_mode=EXP_MODES[args.exp_mode], nv=args.nvfp4)
    T, H, d, nd = r["T"], r["H"], r["d"], r["nd"]
    q_h, k_h, v_h, cu, ws, Q, K, V = (r[x] for x in ("q_h", "k_h", "v_h", "cu", "ws", "Q", "K", "V"))
    lq, lk, lv, blk, rot, seed, stream = (r[x] for x in ("lq", "lk", "lv", "blk", "rot", "seed", "stream"))
    causal, exact = w.causal, bool(args.exact)
    o, lse = r["o"], r["lse"]
    q, k, v = r["q"], r["k"], r["v"]

    # end to end: every step copies its inputs in from pinned host memory and its
    # output and lse back out. The copies of step i + 1 overlap the compute of step
    # i: two device input sets and two output sets, an H2D and a D2H stream, and
    # events that keep every buffer's reuse ordered.
    o_h = torch.empty((T, H, d), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((H, T), dtype=torch.float32).pin_memory()
    sets_in = [(q, k, v), tuple(torch.empty_like(x) for x in (q, k, v))]
    sets_out = [(o, lse), (torch.empty_like(o), torch.empty_like(lse))]
    h2d_s = torch.cuda.Stream(dev)
    d2h_s = torch.cuda.Stream(dev)

    def run_e2e(n):
        ev = lambda: torch.cuda.Event()
        h2d_done = [ev(), ev()]
        comp_done = [ev(), ev()]
        d2h_done = [ev(), ev()]
        used = [False, False]

        def h2d(i):
            b = i % 2
            if used[b]:
                h2d_s.wait_event(comp_done[b])      # step i - 2 has consumed this input set
            with torch.cuda.stream(h2d_s):
                for dst, src in zip(sets_in[b], (q_h, k_h, v_h)):
                    dst.copy_(src, non_blocking=True)
            h2d_done[b].record(h2d_s)

        h2d_s.wait_stream(stream)
        h2d(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                h2d(i + 1)
            stream.wait_event(h2d_done[b])
            if used[b]:
                stream.wait_event(d2h_done[b])      # step i - 2's output has been read back
            qi, ki, vi = sets_in[b]
            oi, li = sets_out[b]
            r["quantise"](qi, ki, vi)
            pa.attn_fp8_fwd_ex(Q, K, V, cu, causal, exact, 0.0, EXP_MODES[args.exp_mode], ws=ws, out=oi, lse=li,
                               stream=stream)
            comp_done[b].record(stream)
            used[b] = True
            d2h_s.wait_event(comp_done[b])
            with torch.cuda.stream(d2h_s):
                o_h.copy_(oi, non_blocking=True)
                lse_h.copy_(li, non_blocking=True)
            d2h_done[b].record(d2h_s)
        stream.wait_stream(d2h_s)
        stream.wait_stream(h2d_s)

    e2e_steps = max(3, min(args.steps, 20))
    run_e2e(2)
    torch.cuda.synchronize()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    # three windows of e2e_steps steps; the median window is reported (the host link
    # is shared with the rest of the machine, and a transient slows one window)
    windows = []
    for _ in range(3):
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        run_e2e(e2e_steps)
        s1.record(stream)
        torch.cuda.synchronize()
        windows.append(s0.elapsed_time(s1) / e2e_steps)
    e2e_ms = sorted(windows)[1]
    h2d = sum(x.numel() * x.element_size() for x in (q_h, k_h, v_h))
    d2h = o_h.numel() * 2 + lse_h.numel() * 4

    # accuracy on sampled rows (outside the timed region): FP8 and BF16 paths vs FP64,
    # and the BF16 comparator path's own speed on the same inputs
    acc = None
    if rank == 0 and not args.no_accuracy:
        acc = accuracy_sample(r["inp"], args.workload, q, k, v, cu, o, pa, torch)
    bf16 = None
    if rank == 0:
        bf16 = time_bf16(pa, torch, q, k, v, cu, causal, r["flops"], ws)
    del sets_in, sets_out, o_h, lse_h
    for x in ("q", "k", "v", "Q", "K", "V", "o", "lse", "ws"):
        r.pop(x, None)
    del q, k, v, Q, K, V, o, lse
    torch.cuda.empty_cache()

    ms_step = r["ms_step"]
    if dist:
        ms_step, e2e_ms = max_over_ranks([ms_step, e2e_ms], dev)
    r.update({"ms_step": ms_step, "e2e_ms": e2e_ms, "e2e_windows_ms": windows, "e2e_steps": e2e_steps, "h2d": h2d,
              "d2h": d2h, "acc": acc, "bf16": bf16})
    # the other benchmark configurations, timed in this process (rank 0, N = 1 only)
    r["per_workload"] = None
    if (rank == 0 and world == 1 and not args.no_per_workload and args.heads is None and args.seqlen is None
            and args.exp_mode == "hw" and not args.nvfp4):
        per = {}
        for wid, ex in ((2, False), (3, False), (3, True), (4, False), (5, False), (5, True)):
            if wid == args.workload and ex == bool(args.exact):
                continue
            rr = time_workload(args, pa, torch, dev, wid, ex, min(args.steps, 30), 3, clocks_idx=local_rank)
            per[f"{workloads.WORKLOADS[wid].name}{' causal-exact' if ex else ''}"] = summarize(rr, wid, ex)
        # the mixed NVFP4/FP8 path (NVFP4 Q K^T) on the two E4M3 configurations
        for wid in (2, 3):
            rr = time_workload(args, pa, torch, dev, wid, False, min(args.steps, 30), 3, clocks_idx=local_rank, nv=True)
            e_ = summarize(rr, wid, False)
            e_["qk"] = "NVFP4"
            per[f"{workloads.WORKLOADS[wid].name} nvfp4-qk"] = e_
        r["per_workload"] = per
        # the bit-level exponentials (inference options) on the four non-exact configurations
        hw = {w_: (r["attn_ms"], r["acc"]) if w_ == args.workload and not args.exact else None for w_ in (2, 3, 4, 5)}
        for w_ in hw:
            if hw[w_] is None:
                e_ = per[workloads.WORKLOADS[w_].name]
                hw[w_] = (e_["attn_ms"], e_["accuracy"])
        bx = {}
        for w_ in (2, 3, 4, 5):
            for name, em in (("schraudolph", pa.ATTN_EXP_SCHRAUDOLPH), ("mitchell_p", pa.ATTN_EXP_MITCHELL_P)):
                rr = time_workload(args, pa, torch, dev, w_, False, min(args.steps, 30), 3, clocks_idx=local_rank,
                                   exp_mode=em)
                e_ = summarize(rr, w_, False)
                e_["exp_mode"] = name
                e_["attn_speedup_vs_hw_exp2"] = hw[w_][0] / rr["attn_ms"]
                if rr.get("acc") and hw[w_][1]:
                    e_["cosine_change_vs_hw_exp2"] = rr["acc"]["cosine_fp8_vs_fp64"] - hw[w_][1]["cosine_fp8_vs_fp64"]
                bx[f"{workloads.WORKLOADS[w_].name} {name}"] = e_
        r["bit_level_exp"] = bx
        r["backward"] = time_bwd(pa, torch, dev)
    r["fp8_peak_measured"] = measure_fp8_peak(torch, dev) if rank == 0 else None
    return r


def time_bf16(pa, torch, q, k, v, cu, causal, flops, ws, n=10):
    """The BF16 comparator path's forward time on the workload's bf16 inputs."""
    if q.dtype != torch.bfloat16:
        return None
    o = torch.empty_like(q)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    for _ in range(2):
        pa.attn_bf16_fwd(q, k, v, cu, causal, ws=ws, out=o, lse=lse)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(n):
        pa.attn_bf16_fwd(q, k, v, cu, causal, ws=ws, out=o, lse=lse)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    return {"attn_ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "kernel": "attn_fwd_kernel (BF16 operands)"}


def time_bwd(pa, torch, dev, n=10, B=2, H=32, N=8192, causals=(False, True), warmup=3):
    """The BF16 backward (attn_bf16_bwd: dQ, dK, dV) on the headline shape, non-causal
    and causal: seeded bf16 inputs of that shape, o and lse from attn_bf16_fwd, then
    n timed calls (CUDA events on the launching stream; the five [T, H, d] inputs are
    over 600 MB, larger than L2). FLOPs: 2.5 x the forward's (five matrix products of
    the forward's size; the kernel performs seven, as dQ forms S and dP again)."""
    pk = load_peaks()
    bf16_peak = float(pk["bf16_tflops"]) if pk and pk.get("bf16_tflops") else 1900.0
    out = {}
    d = 128
    T = B * N
    g = torch.Generator(device=dev).manual_seed(1234)
    q, k, v, do = (torch.randn((T, H, d), device=dev, generator=g).to(torch.bfloat16) for _ in range(4))
    cu = torch.arange(0, T + 1, N, dtype=torch.int32, device=dev)
    ws = pa.bwd_workspace(T, H, d, B, dev)
    outs = tuple(torch.empty_like(q) for _ in range(3))
    for causal in causals:
        o, lse = pa.attn_bf16_fwd(q, k, v, cu, causal)
        for _ in range(warmup):
            pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, causal, ws=ws, outs=outs)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            pa.attn_bf16_bwd(q, k, v, o, do, lse, cu, causal, ws=ws, outs=outs)
        e1.record()
        torch.cuda.synchronize()
        st, _ = pa.attn_read_device_status(ws)
        ms = e0.elapsed_time(e1) / n
        fl = 2.5 * workloads.attention_flops(cu.cpu().numpy(), H, d, causal)
        tf = fl / (ms * 1e-3) / 1e12
        out["causal" if causal else "non-causal"] = {
            "ms": ms, "tflops": tf, "frac_vs_bf16_measured": tf / bf16_peak, "status": st}
        del o, lse
    out.update({"config": {"batch": B, "heads": H, "seq_len": N, "head_dim": d, "dtype": "bf16"},
                "kernels": "sched_kernel, bwd_prep_kernel, attn_bwd_kernel (dK, dV), attn_bwd_dq_kernel (dQ): four launches per call",
                "flops": "2.5 x forward FLOPs (causal halved)", "bf16_peak": bf16_peak,
                "bf16_peak_basis": "MEASURED_PEAKS.json bf16_tflops (burst)" if pk else "fallback"})
    return out


def summarize(rr, wid, exact):
    peak, _ = fp8_peak()
    hbm, _ = hbm_peak()
    val = rr["flops"] / (rr["ms_step"] * 1e-3) / 1e12
    att = rr["flops"] / (rr["attn_ms"] * 1e-3) / 1e12
    return {"value": val, "unit": UNIT, "ms_per_step": rr["ms_step"], "attn_ms": rr["attn_ms"],
            "quant_ms": rr["quant_ms"], "attn_tflops": att, "frac_incl_quant": val / peak, "attn_frac": att / peak,
            "quant_gbs": rr["quant_bytes"] / (rr["quant_ms"] * 1e-3) / 1e9,
            "quant_hbm_frac": rr["quant_bytes"] / (rr["quant_ms"] * 1e-3) / 1e9 / hbm,
            "timing_stats": rr["stats"], "clocks": rr["clocks"], "accuracy": rr.get("acc"),
            "causal": rr["causal"], "causal_exact": exact, "mx": rr["mx"]}


def accuracy_sample(inp, wid, q, k, v, cu, o_fp8, pa, torch):
    import oracle
    rng = np.random.default_rng(123)
    rows = np.sort(rng.choice(inp.T, size=min(64, inp.T), replace=False)).astype(np.int32)
    causal = workloads.WORKLOADS[wid].causal
    ob, _ = pa.attn_bf16_fwd(q, k, v, cu, causal)
    o1, _ = oracle.attention_fp64(inp.q, inp.k, inp.v, inp.cu_seqlens, causal, None, rows=rows)
    o8 = o_fp8.float().cpu().numpy()[rows].astype(np.float64)
    obb = ob.float().cpu().numpy()[rows].astype(np.float64)
    r8 = float(np.sqrt(np.mean((o8 - o1) ** 2)))
    rb = float(np.sqrt(np.mean((obb - o1) ** 2)))
    cos = float(np.sum(o8 * o1) / (np.linalg.norm(o8) * np.linalg.norm(o1)))
    return {"rows_sampled": int(len(rows)), "rmse_fp8_vs_fp64": r8, "rmse_bf16_vs_fp64": rb,
            "ratio_fp8_over_bf16": r8 / rb if rb > 0 else None, "cosine_fp8_vs_fp64": cos}


# ---------------------------------------------------------------------------
def cpu_sample(args, inp=None, budget_s=15.0, rows=None):
    """Time the oracle (quantiser + quantised-operand emulation) on whole heads
    of the workload's first document until about `budget_s` of CPU work.
    rows: evaluate only the first `rows` query rows of the document (all keys)."""
    import oracle
    oracle.build()
    w = workloads.WORKLOADS[args.workload]
    if inp is None:
        inp = workloads.make(args.workload, heads=args.heads, seqlen=args.seqlen, batch=args.batch)
    cu = inp.cu_seqlens
    L0 = int(cu[1] - cu[0])
    R = L0 if rows is None else min(rows, L0)
    row_idx = None if R == L0 else np.arange(R, dtype=np.int32)
    flops = 0.0
    t_total = 0.0
    heads_done = 0
    H = inp.q.shape[1]
    d = inp.q.shape[2]
    c1 = np.array([0, L0], np.int32)
    for h in range(H):
        q = np.ascontiguousarray(inp.q[:L0, h:h + 1])
        k = np.ascontiguousarray(inp.k[:L0, h:h + 1])
        v = np.ascontiguousarray(inp.v[:L0, h:h + 1])
        t0 = time.perf_counter()
        if w.mx:
            Q = oracle.quantize_tensor(q, c1, ROW, 32, not args.no_rotate, w.hadamard_seed)
            K = oracle.quantize_tensor(k, c1, ROW, 32, not args.no_rotate, w.hadamard_seed)
            V = (oracle.quantize_tensor(v, c1, oracle.MX_TOKEN, 1, False, 0) if args.exact
                 else oracle.quantize_tensor(v, c1, COL, 32, False, 0))
        else:
            b = 1 if args.exact else w.block
            Q = oracle.quantize_tensor(q, c1, E4M3, b, not args.no_rotate, w.hadamard_seed)
            K = oracle.quantize_tensor(k, c1, E4M3, b, not args.no_rotate, w.hadamard_seed)
            V = oracle.quantize_tensor(v, c1, E4M3, b, False, 0)
        oracle.attention_emulate(Q, K, V, c1, w.causal, bool(args.exact), None, rows=row_idx,
                                 rescale_tau=0.75 if d == 128 else 0.0, exp_mode=EXP_MODES[args.exp_mode])
        t_total += time.perf_counter() - t0
        nkeys = np.arange(1, R + 1) if w.causal else np.full(R, L0)
        flops += float(4.0 * d * nkeys.sum())
        heads_done += 1
        if t_total >= budget_s:
            break
    return {"value": flops / t_total / 1e12, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "sample": f"document 0 ({L0} tokens), {heads_done} of {H} heads, {R} query rows each over all "
                      f"visible keys: oracle quantiser (Q, K, V of the head) + quantised-operand emulation; "
                      f"{t_total:.1f} s of host time",
            "seconds": t_total}


def reference_arm(args, rank, world):
    if rank != 0:
        return
    w = workloads.WORKLOADS[args.workload]
    inp = workloads.make(args.workload, heads=args.heads, seqlen=args.seqlen, batch=args.batch)
    samples = []
    for _ in range(args.warmup):
        cpu_sample(args, inp, budget_s=0.0, rows=64)
    for _ in range(args.steps):
        samples.append(cpu_sample(args, inp, budget_s=0.0, rows=1024))
    secs = sum(s["seconds"] for s in samples)
    val = float(np.median([s["value"] for s in samples]))
    line = {"metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * secs / len(samples), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle emulation of e4m3 / fp32)",
            "data": "synthetic", "impl": "reference", "config": config_of(args, w),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": samples[0]["cores"], "kind": "oracle",
                             "sample": samples[0]["sample"]},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# the probabilities' exponential (include/attn.h attn_exp_mode)
EXP_MODES = {"hw": 0, "schraudolph": 1, "mitchell_p": 2}


def config_of(args, w):
    return {"workload": f"{w.name} (workload {w.wid})", "batch": args.batch or w.batch,
            "heads": args.heads or w.heads, "seq_len": args.seqlen or w.seqlen or None, "head_dim": w.head_dim,
            "causal": w.causal, "causal_exact": bool(args.exact), "exp_mode": args.exp_mode, "schedule": args.sched,
            "quant": ("NVFP4 Q, K (E2M1, E4M3 per 16 channels, fp32 per 128 tokens); V E4M3 blocks of 128 tokens"
                      if args.nvfp4 else
                      ("MXFP8 (E8M0 per 32; V one E8M0 per token, causal-exact)" if args.exact else "MXFP8 (E8M0 per 32)")
                      if w.mx else
                      ("E4M3 one scale per token (causal-exact)" if args.exact else f"E4M3 blocks of {w.block} tokens")) +
            (" + Hadamard rotation of Q, K" if not args.no_rotate else ", no rotation"), "input_dtype": w.in_dtype,
            "l2": "inputs larger than L2 (bf16 Q, K, V and their codes each exceed 129 MB)" if (
                args.heads is None and args.seqlen is None) else "reduced size"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--heads", type=int, default=None)
    ap.add_argument("--seqlen", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-accuracy", action="store_true")
    ap.add_argument("--no-rotate", action="store_true", help="quantise Q and K without the Hadamard rotation")
    ap.add_argument("--sched", default="static", choices=["static", "ticket"],
                    help="the pair kernel's work order: static longest-first rounds or just-in-time tickets")
    ap.add_argument("--quant-split", action="store_true",
                    help="quantise Q, K and V in three launches instead of one")
    ap.add_argument("--exact", action="store_true", help="causal-exact mode (one E4M3 scale per token)")
    ap.add_argument("--nvfp4", action="store_true",
                    help="the mixed NVFP4/FP8 path: NVFP4 Q and K (Q K^T on the FP4 tensor cores), E4M3 V")
    ap.add_argument("--exp-mode", default="hw", choices=sorted(EXP_MODES),
                    help="the probabilities' exponential: the hardware exp2 (default), Schraudolph's, or log-domain P")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the BF16 backward (attn_bf16_bwd) on --batch/--heads/--seqlen "
                         "(default B2 H32 N8192), --steps calls after --warmup, and print its JSON")
    ap.add_argument("--causal", action="store_true", help="with --backward-only: the causal backward only")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip timing the other benchmark configurations in the same process")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        reference_arm(args, rank, world)
        return

    if args.backward_only:
        import torch
        from precision_attention_gb300 import build as pbuild
        pbuild.build()
        import precision_attention_gb300 as pa
        torch.cuda.set_device(0)
        res = time_bwd(pa, torch, torch.device("cuda"), n=args.steps, B=args.batch or 2, H=args.heads or 32,
                       N=args.seqlen or 8192, causals=(True,) if args.causal else (False,), warmup=args.warmup)
        print(json.dumps({"backward": res}), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    from precision_attention_gb300 import build as pbuild
    if rank == 0 or world == 1:
        pbuild.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    r = gpu_arm(args, rank, world, local_rank)
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    w = workloads.WORKLOADS[args.workload]
    value = job_throughput(world, r["flops"], r["ms_step"])
    e2e = job_throughput(world, r["flops"], r["e2e_ms"])
    peak, peak_basis = fp8_peak()
    hbm, hbm_basis = hbm_peak()
    achieved = r["flops"] / (r["attn_ms"] * 1e-3) / 1e12
    clk = r["clocks"] or {}
    # the tensor cores' own e4m3 rate at the clock seen (128 x 128 x 32 MMA in 64
    # cycles: 16,384 FLOP per cycle per SM, measured on this part)
    mma_rate = None
    if clk.get("sm_mhz"):
        import torch
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        mma_rate = 16384.0 * sms * clk["sm_mhz"] * 1e6 / 1e12
    fp8m = r.get("fp8_peak_measured")
    kernel = "attn_pair_kernel" if r["d"] == 128 else "attn_fwd_kernel"
    qbytes = r["quant_bytes"]
    quant_gbs = qbytes / (r["quant_ms"] * 1e-3) / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3" if not w.mx else "mxfp8 (e4m3 + e8m0)", "data": "synthetic",
            "config": config_of(args, w),
            "e2e": {"value": e2e, "unit": UNIT, "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                    "ms_per_step": r["e2e_ms"], "windows_ms": r["e2e_windows_ms"], "window_steps": r["e2e_steps"],
                    "reported": "median of three windows"},
            # per step: the quantiser (one launch, or three with --quant-split; each
            # after the document-table kernel above 1,024 documents), the work list,
            # the V references (E4M3, NVFP4 and causal-exact MX), the attention kernel
            "gpu_launches": ((3 if args.quant_split else 1) * (2 if r["nd"] > 1024 else 1) +
                             (2 if (w.mx and not args.exact) else 3)) * args.steps,
            "roofline": {"bound": "tensor", "kernel": kernel + " (FP8 forward call)", "achieved": achieved,
                         "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "traffic": attn_traffic(args),
                         "peak_basis": peak_basis + " (of measured)",
                         "frac_incl_quant": value / world / peak,
                         "peak_fp8_measured": fp8m, "frac_vs_fp8_measured": (achieved / fp8m) if fp8m else None,
                         "peak_fp8_measured_basis": "dense e4m3 GEMM of the vendor library (torch._scaled_mm), "
                                                    "8192^3, best of 10, this process",
                         "mma_rate_at_clock": mma_rate,
                         "frac_vs_mma_rate": (achieved / mma_rate) if mma_rate else None},
            "quant_roofline": {"bound": "hbm", "kernel": ("quant_tile_kernel (three launches: Q, K, V)" if args.quant_split
                                                      else "quant_tile_kernel (one launch: Q, K, V)"),
                               "achieved": quant_gbs, "peak": hbm, "unit": "GB/s", "frac": quant_gbs / hbm,
                               "bytes_per_step": qbytes, "peak_basis": hbm_basis, "traffic": quant_traffic(args)},
            "attn_ms": r["attn_ms"], "quant_ms": r["quant_ms"], "timing_stats": r["stats"],
            "clocks": r["clocks"], "accuracy": r["acc"], "bf16_path": r.get("bf16"),
            "per_workload": r.get("per_workload"), "bit_level_exp": r.get("bit_level_exp"),
            "backward": r.get("backward")}
    if not args.no_cpu_baseline and world >= 1:
        line["cpu_baseline"] = cpu_sample(args, r.get("inp"))
        line["cpu_baseline"].pop("seconds", None)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
