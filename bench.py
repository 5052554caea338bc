"""Attn-QAT benchmark: backward (and forward) TFLOP/s on one GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c2] [--impl ours|reference]

A step is one pass of the whole path over one batch of synthetic input:
quantize Q/K/V + forward (O, O', LSE), then preprocess + backward (dQ, dK,
dV) on that forward's O' and LSE. The L2 cache is flushed (256 MiB write)
between steps, outside the timed kernels. FLOPs are nominal: forward
4*B*H*Sq*Sk*D, backward 10*B*H*Sq*Sk*D, halved for causal.

`value` is the backward TFLOP/s (CUDA events around the backward API calls);
`roofline` reports the backward main kernel alone against the measured dense
BF16 peak; `e2e` repeats the backward through the C ABI with pinned host
buffers, host<->device copies inside the timed region; `cpu_baseline` times
the float64 CPU oracle on whole heads of the same workload (about 10 s).

With --gpus N (launched by torchrun) every rank runs the full workload on its
own GPU (independent problems, no collective on the data path) and `value` is
the sum over ranks divided by the slowest rank's time (weak scaling). With
--shard heads the ranks instead split one workload's B*H heads into
contiguous, balanced slices (every (b, h) head is independent in both
directions, and a slice of the flattened heads is contiguous in BHSD), each
rank generating and running only its own slice; `value` is the whole
workload's FLOPs over the slowest rank's time (strong scaling). Neither mode
has a collective on the data path: only the timing barrier and the max over
ranks use the process group.

--workload ctx32k (or --path infer) measures the NVFP4 inference forward
instead: a step is NVFP4 packing of Q and K plus the block-scaled FP4 QK /
BF16 PV attention kernel (O and LSE), 4*B*H*Sq*Sk*D FLOPs (halved for
causal). Its roofline is the exp2 (MUFU) bound of the softmax, with the
tensor-pipe bound beside it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp4_quantization_aware_gb300 import synth  # noqa: E402

PROFILE_JSON = os.path.join(ROOT, "profiles", "bwd_main_c2_counters.json")
KERNEL_SOURCES = [os.path.join(ROOT, "fp4_quantization_aware_gb300", "csrc", f)
                  for f in ("bwd.cu", "fp4_mma.cuh", "attn_common.cuh", "nvfp4.cuh", "ptx.cuh")]


METRIC = "QAT attn bwd TFLOP/s on 1 GB300 (fwd in fwd_tflops); % of dense BF16 peak in roofline"
METRIC_INFER = "NVFP4 inference attn fwd TFLOP/s on 1 GB300 (pack Q/K + FP4 QK / BF16 PV kernel)"
INFER_SOURCES = [os.path.join(ROOT, "fp4_quantization_aware_gb300", "csrc", f)
                 for f in ("infer.cu", "fp4_mma.cuh", "attn_common.cuh", "nvfp4.cuh", "ptx.cuh")]
PROFILE_INFER_JSON = os.path.join(ROOT, "profiles", "infer_kernel_ctx32k_counters.json")
# exp2 results per clock per SM of the MUFU unit (ex2.approx), as measured on
# this GPU by a throughput probe (16 lanes x 4 sub-partitions x 2 on the
# Blackwell Ultra SFU, whose exp throughput is twice Blackwell's).
MUFU_EX2_PER_CLK_SM = 32
# `chunks` of attnqat_bwd_host in the end-to-end measurement: head groups of
# ceil(B*H / 4) heads, the first and last of half that (c2: 2, 4, 4, 4, 2)
E2E_CHUNKS = 4
FP4_OVER_BF16 = 6.0        # nominal dense FP4 / BF16 tensor ratio of GB300 (13.5 / 2.25 PFLOP/s)


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings over all ranks (the slowest rank
    sets the job's time). Returns the values unchanged without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tflops(flops_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: `world` ranks each doing `flops_per_rank_step`
    (pass world = 1 with the whole job's FLOPs when the ranks split one
    workload); the job takes as long as its slowest rank."""
    return world * flops_per_rank_step * steps / (max_ms * 1e-3) / 1e12


def head_slice(n_heads: int, world: int, rank: int) -> tuple[int, int]:
    """The heads [h0, h1) of the flattened (b, h) order that rank `rank` of
    `world` takes in the data-parallel mode: contiguous, sizes differing by at
    most one, every head in exactly one rank's slice."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    return rank * n_heads // world, (rank + 1) * n_heads // world


def shard_heads(w, world: int, rank: int) -> list:
    """The (b, h) pairs of this rank's slice, in BHSD memory order."""
    n = w.B * w.H
    if world > n:
        raise ValueError(f"--shard heads needs at most B*H = {n} ranks, got {world}")
    h0, h1 = head_slice(n, world, rank)
    return [divmod(i, w.H) for i in range(h0, h1)]


def shard_byte_offsets(w, rank_heads: list) -> dict:
    """Byte offset of a slice's first head in each full BHSD tensor (and in
    the (B, H, Sq) LSE), for a caller that keeps the whole tensors and hands
    each rank a view: the slice is contiguous there."""
    b, h = rank_heads[0]
    i = b * w.H + h
    return {"q": i * w.Sq * w.D * 2, "do": i * w.Sq * w.D * 2, "o": i * w.Sq * w.D * 2,
            "k": i * w.Sk * w.D * 2, "v": i * w.Sk * w.D * 2, "lse": i * w.Sq * 4}


def rank_workload(w, heads):
    """The workload one rank runs: the whole one, or its slice of heads as a
    (len(heads), 1) batch (each head is an independent problem)."""
    if heads is None:
        return w
    return synth.workload(w.name, B=len(heads), H=1, Sq=w.Sq, Sk=w.Sk)


def kernel_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in (sources or KERNEL_SOURCES):
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16": d["bf16_tflops"], "bf16_sustained": d.get("bf16_tflops_sustained"), "hbm": d["hbm_gbs"],
                "sm_max_mhz": d.get("sm_max_mhz", 2070.0), "src": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "sm_max_mhz": 2070.0, "src": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------- ours
def run_ours(args, w, rank, world, local_rank, heads=None):
    """Time the QAT step on the whole workload, or on `heads` (this rank's
    slice, generated head by head exactly as in the whole workload)."""
    import torch
    from fp4_quantization_aware_gb300 import attnqat
    import ctypes

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = attnqat.load()
    x = synth.inputs(w, heads=heads)
    w = rank_workload(w, heads)
    t = {n: torch.from_numpy(a).to(torch.bfloat16).to(dev) for n, a in x.items()}
    p = attnqat.problem(w.B, w.H, w.Sq, w.Sk, w.D, w.causal, w.scale)
    pp = ctypes.byref(p)
    ws_f = attnqat.workspace(lib.attnqat_fwd_workspace_bytes(pp), dev)
    ws_b = attnqat.workspace(lib.attnqat_bwd_workspace_bytes(pp), dev)
    o, o_hp = torch.empty_like(t["q"]), torch.empty_like(t["q"])
    lse = torch.empty(w.shape_q[:3], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    P = lambda a: a.data_ptr()  # noqa: E731

    # the forward is the one API call a user makes: attnqat_fwd (quantize, then
    # the two passes) or, in recipe R2, attnqat_fwd_r2_p with its P format
    fmt = attnqat.P_FORMATS[args.recipe[3:] if args.recipe.startswith("r2-") else "nvfp4"]

    def fwd():
        if args.recipe == "standard":
            attnqat.check(lib.attnqat_fwd(pp, P(t["q"]), P(t["k"]), P(t["v"]), P(o), P(o_hp), P(lse), P(ws_f),
                                          ws_f.numel(), sp), "fwd")
        else:
            attnqat.check(lib.attnqat_fwd_r2_p(pp, P(t["q"]), P(t["k"]), P(t["v"]), P(o), P(o_hp), P(lse), fmt,
                                               P(ws_f), ws_f.numel(), sp), "fwd r2")

    def bwd(ev=None):
        attnqat.check(lib.attnqat_bwd_preprocess(pp, P(t["do"]), P(t["q"]), P(t["k"]), P(t["v"]), P(o_hp),
                                                 P(ws_b), ws_b.numel(), sp), "prep")
        if ev:
            ev[0].record(stream)
        attnqat.check(lib.attnqat_bwd_main(pp, P(t["do"]), P(lse), P(dk), P(dv), P(ws_b), ws_b.numel(), sp), "bwd")
        if ev:
            ev[1].record(stream)
        attnqat.check(lib.attnqat_bwd_dq_convert(pp, P(dq), P(ws_b), ws_b.numel(), sp), "dqc")

    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for _ in range(args.warmup):
        flush.zero_()
        fwd()
        bwd()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    evs = [(E(), E(), E(), E(), E()) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for e in evs:
            flush.zero_()
            e[0].record(stream)
            fwd()
            e[1].record(stream)
            bwd(ev=(e[2], e[3]))
            e[4].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = sum(e[1].elapsed_time(e[4]) for e in evs)
    main_ms = [e[2].elapsed_time(e[3]) for e in evs]
    step_ms = (fwd_ms + bwd_ms) / args.steps
    launches = 5 * args.steps
    assert attnqat.device_status() == 0, "a device wait timed out during the bench"

    # end to end through the C ABI with pinned host buffers (backward step):
    # attnqat_bwd_host copies head groups in and out while other groups compute
    host_in = {n: t[n].cpu().pin_memory() for n in ("do", "q", "k", "v")}
    host_in["o_hp"] = o_hp.cpu().pin_memory()
    host_in["lse"] = lse.cpu().pin_memory()
    host_out = [torch.empty_like(a, device="cpu").pin_memory() for a in (dq, dk, dv)]
    ws_h = attnqat.workspace(lib.attnqat_bwd_host_workspace_bytes(pp, args.e2e_chunks), dev)
    e2e_evs = [(E(), E()) for _ in range(args.steps)]
    for i in range(args.warmup + args.steps):
        flush.zero_()
        if i >= args.warmup:
            e2e_evs[i - args.warmup][0].record(stream)
        attnqat.check(lib.attnqat_bwd_host(pp, P(host_in["do"]), P(host_in["q"]), P(host_in["k"]), P(host_in["v"]),
                                           P(host_in["o_hp"]), P(host_in["lse"]), P(host_out[0]), P(host_out[1]),
                                           P(host_out[2]), args.e2e_chunks, P(ws_h), ws_h.numel(), sp), "bwd e2e")
        if i >= args.warmup:
            e2e_evs[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    del ws_h
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_evs) / args.steps
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out)

    res = {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "main_ms": main_ms, "step_ms": step_ms, "wall": wall,
           "launches": launches, "e2e_ms": e2e_ms, "h2d": h2d, "d2h": d2h, "clocks": clk.summary()}
    res["bwd_ms"], res["fwd_ms"], res["step_ms"], res["e2e_ms"] = max_over_ranks([bwd_ms, fwd_ms, step_ms, e2e_ms], dev)
    return res


def run_infer(args, w, rank, world, local_rank):
    """Time the NVFP4 inference forward (pack Q, pack K, attention kernel)."""
    import torch
    from fp4_quantization_aware_gb300 import attnqat
    import ctypes

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = attnqat.load()
    x = synth.inputs(w)
    t = {n: torch.from_numpy(x[n]).to(torch.bfloat16).to(dev) for n in ("q", "k", "v")}
    del x
    p = attnqat.problem(w.B, w.H, w.Sq, w.Sk, w.D, w.causal, w.scale)
    pp = ctypes.byref(p)
    need = lib.attnqat_infer_fwd_workspace_bytes(pp)
    if need == 0:
        attnqat.check(lib.attnqat_check_support(pp), "check_support")
        raise SystemExit("the inference forward needs D == 128")
    bh = w.B * w.H
    qp = torch.empty(bh * w.Sq * 64, dtype=torch.uint8, device=dev)
    qs = torch.empty(bh * w.Sq * 8, dtype=torch.uint8, device=dev)
    kp = torch.empty(bh * w.Sk * 64, dtype=torch.uint8, device=dev)
    ks = torch.empty(bh * w.Sk * 8, dtype=torch.uint8, device=dev)
    ws = attnqat.workspace(need, dev)
    o = torch.empty_like(t["q"])
    lse = torch.empty(w.shape_q[:3], dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    P = lambda a: a.data_ptr()  # noqa: E731

    def step(ev=None):
        attnqat.check(lib.attnqat_nvfp4_pack(P(t["q"]), P(qp), P(qs), bh * w.Sq, w.D, sp), "pack q")
        attnqat.check(lib.attnqat_nvfp4_pack(P(t["k"]), P(kp), P(ks), bh * w.Sk, w.D, sp), "pack k")
        if ev:
            ev[0].record(stream)
        attnqat.check(lib.attnqat_infer_fwd_packed(pp, P(qp), P(qs), P(kp), P(ks), P(t["v"]), P(o), P(lse), sp),
                      "infer")
        if ev:
            ev[1].record(stream)

    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    evs = [(E(), E(), E(), E()) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        torch.cuda.synchronize()
        for e in evs:
            flush.zero_()
            e[0].record(stream)
            step(ev=(e[1], e[2]))
            e[3].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    step_ms = sum(e[0].elapsed_time(e[3]) for e in evs) / args.steps
    kern_ms = [e[1].elapsed_time(e[2]) for e in evs]
    assert attnqat.device_status() == 0, "a device wait timed out during the bench"

    # end to end: pinned host Q, K, V in, O and LSE out, through attnqat_infer_fwd
    host_in = {n: t[n].cpu().pin_memory() for n in ("q", "k", "v")}
    dev_in = {n: torch.empty_like(v, device=dev) for n, v in host_in.items()}
    host_out = [torch.empty_like(a, device="cpu").pin_memory() for a in (o, lse)]
    e2e_evs = [(E(), E()) for _ in range(args.steps)]
    for i in range(args.warmup + args.steps):
        flush.zero_()
        if i >= args.warmup:
            e2e_evs[i - args.warmup][0].record(stream)
        for n in dev_in:
            dev_in[n].copy_(host_in[n], non_blocking=True)
        attnqat.check(lib.attnqat_infer_fwd(pp, P(dev_in["q"]), P(dev_in["k"]), P(dev_in["v"]), P(o), P(lse), P(ws),
                                            ws.numel(), sp), "infer e2e")
        for h, d in zip(host_out, (o, lse)):
            h.copy_(d, non_blocking=True)
        if i >= args.warmup:
            e2e_evs[i - args.warmup][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_evs) / args.steps
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out)
    res = {"step_ms": step_ms, "kern_ms": kern_ms, "e2e_ms": e2e_ms, "h2d": h2d, "d2h": d2h,
           "launches": 3 * args.steps, "clocks": clk.summary(),
           "n_sm": torch.cuda.get_device_properties(dev).multi_processor_count}
    res["step_ms"], res["e2e_ms"] = max_over_ranks([step_ms, e2e_ms], dev)
    return res


def infer_line(args, w, world, r, peaks, l2) -> dict:
    flops = w.fwd_flops()
    kern_ms = statistics.mean(r["kern_ms"])
    exps = w.B * w.H * w.Sq * w.Sk / (2 if w.causal else 1)
    sm_mhz = peaks["sm_max_mhz"]
    n_sm = r["n_sm"]
    mufu_peak = MUFU_EX2_PER_CLK_SM * n_sm * sm_mhz * 1e6 / 1e9           # G exp2/s at the maximum SM clock
    achieved = exps / (kern_ms * 1e-3) / 1e9
    # tensor-pipe bound: half the FLOPs (QK) at the FP4 rate, half (PV) at the BF16 rate
    tensor_peak = 2.0 / (1.0 / peaks["bf16"] + 1.0 / (FP4_OVER_BF16 * peaks["bf16"]))
    tensor_achieved = flops / (kern_ms * 1e-3) / 1e12
    traffic = None
    if os.path.exists(PROFILE_INFER_JSON):
        prof = json.load(open(PROFILE_INFER_JSON))
        if prof.get("kernel_hash") == kernel_hash(INFER_SOURCES) and prof.get("workload") == w.name:
            traffic = prof.get("dram_bytes_per_launch")
    cfg = workload_config(w, l2)
    cfg["step"] = "NVFP4 pack of Q and K, then the FP4 QK / BF16 PV attention kernel (O, LSE)"
    return {
        "metric": METRIC_INFER, "value": job_tflops(flops, 1, world, r["step_ms"]), "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["step_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 QK, bf16 PV, f32 softmax",
        "data": "synthetic", "config": cfg,
        "kernel_tflops": tensor_achieved, "kernel_ms": kern_ms,
        "roofline": {"bound": "alu", "kernel": "infer_kernel (attnqat_infer_fwd_packed)", "achieved": achieved,
                     "peak": mufu_peak, "unit": "Gexp2/s", "frac": achieved / mufu_peak, "traffic": traffic,
                     "launch_ms": kern_ms,
                     "peak_note": f"MUFU ex2: {MUFU_EX2_PER_CLK_SM}/clk/SM x {n_sm} SMs (device) x {sm_mhz:.0f} MHz "
                                  f"(sm_max_mhz, {peaks['src']}): derived",
                     "tensor": {"achieved": tensor_achieved, "peak": tensor_peak, "unit": "TFLOP/s",
                                "frac": tensor_achieved / tensor_peak,
                                "note": f"QK at {FP4_OVER_BF16:g}x and PV at 1x the {peaks['src']} BF16 peak "
                                        f"{peaks['bf16']}"}},
        "e2e": {"value": world * flops / (r["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms": r["e2e_ms"],
                "what": "attnqat_infer_fwd with pinned host Q, K, V in and O, LSE out"},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }


def infer_oracle_rows(w, budget_s):
    """Time the float64 oracle's inference forward on growing query-row blocks
    of head (0, 0) until about budget_s; returns (seconds, flops, rows)."""
    import oracle
    x = synth.head_inputs(w, 0, 0)
    rows, flops = 0, 0.0
    blk = 256
    t0 = time.perf_counter()
    kh = oracle.fake_nvfp4(x["k"].astype(np.float64))          # K once per head
    vv = x["v"].astype(np.float64)
    spent = time.perf_counter() - t0
    while spent < budget_s and rows < w.Sq:
        r1 = min(w.Sq, rows + blk)
        t0 = time.perf_counter()
        # fwd_rows slices rows [rows, r1) of its first argument (the causal mask
        # needs the absolute row index)
        qh = np.zeros((r1, w.D))
        qh[rows:r1] = oracle.fake_nvfp4(x["q"][rows:r1].astype(np.float64))
        oracle.fwd_rows(qh, kh, vv, w.scale, w.causal, rows, r1, quantize=False)
        spent += time.perf_counter() - t0
        keys = np.minimum(np.arange(rows, r1) + 1, w.Sk).sum() if w.causal else (r1 - rows) * w.Sk
        flops += 4.0 * keys * w.D
        rows = r1
    return spent, flops, rows


# ---------------------------------------------------------------------------- CPU oracle
def oracle_heads(w, heads):
    """Time the float64 CPU oracle's forward and backward on the listed heads."""
    import oracle
    fwd_s = bwd_s = 0.0
    for bh in heads:
        x = synth.inputs(w, heads=[bh])
        t0 = time.perf_counter()
        o, o_hp, lse = oracle.attn_qat_fwd(x["q"], x["k"], x["v"], w.scale, w.causal)
        t1 = time.perf_counter()
        oracle.attn_qat_bwd(x["do"], x["q"], x["k"], x["v"], o_hp, lse, w.scale, w.causal)
        fwd_s += t1 - t0
        bwd_s += time.perf_counter() - t1
    n = len(heads)
    return {"fwd_s": fwd_s, "bwd_s": bwd_s, "fwd_flops": n * w.fwd_flops() / (w.B * w.H),
            "bwd_flops": n * w.bwd_flops() / (w.B * w.H)}


def cpu_baseline(w, budget_s: float = 10.0) -> dict:
    """Oracle backward on whole heads, in order, until about budget_s of CPU work."""
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    r = oracle_heads(w, heads[:1])
    n = max(1, min(len(heads), int(budget_s / max(r["fwd_s"] + r["bwd_s"], 1e-3))))
    if n > 1:
        r = oracle_heads(w, heads[:n])
    return {"value": r["bwd_flops"] / r["bwd_s"] / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "sample": f"{n} of {len(heads)} heads of the workload, each full {w.Sq}x{w.Sk}: "
            f"backward {r['bwd_s']:.2f} s, forward {r['fwd_s']:.2f} s, float64 NumPy (BLAS on all cores)"}


def workload_config(w, l2, recipe="standard") -> dict:
    return {"workload": f"{w.name}: B={w.B} H={w.H} Sq={w.Sq} Sk={w.Sk} D={w.D} "
            f"{'causal' if w.causal else 'non-causal'}, {w.structure} N(0,1) BF16, scale={w.scale:.6g}",
            "B": w.B, "H": w.H, "Sq": w.Sq, "Sk": w.Sk, "D": w.D, "causal": w.causal, "l2": l2,
            "step": "quantize+fwd, then preprocess+bwd+dQ convert", "fwd_recipe": recipe}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="c2", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default=None, choices=["qat", "infer"],
                    help="qat: the QAT forward+backward step; infer: the NVFP4 inference forward "
                         "(default: infer for ctx32k, qat otherwise)")
    ap.add_argument("--seq", type=int, default=None, help="override Sq = Sk of the workload (smaller captures)")
    ap.add_argument("--e2e-chunks", type=int, default=E2E_CHUNKS,
                    help="head groups of the end-to-end (host-buffer) backward")
    ap.add_argument("--shard", default="none", choices=["none", "heads"],
                    help="with --gpus N: none = every rank runs the whole workload (weak scaling); heads = the "
                         "ranks split its B*H heads into contiguous slices (strong scaling)")
    ap.add_argument("--recipe", default="standard", choices=["standard", "r2", "r2-e5m2", "r2-e4m3"],
                    help="forward recipe of the QAT step: standard (two passes, P^ of the normalised P) or r2 "
                         "(one pass, P^ of each key tile's unnormalised P: NVFP4, or the FP8-P variant in E5M2 / "
                         "E4M3)")
    args = ap.parse_args()
    w = synth.workload(args.workload) if args.seq is None else synth.workload(args.workload, Sq=args.seq,
                                                                               Sk=args.seq)
    path = args.path or ("infer" if args.workload == "ctx32k" else "qat")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    peaks = measured_peaks()
    l2 = "flushed: 256 MiB write between steps"

    if args.impl == "reference" and path == "infer":
        if rank != 0:
            return
        t0 = time.perf_counter()
        per = []
        for _ in range(args.warmup + args.steps):
            per.append(infer_oracle_rows(w, 5.0))
        per = per[args.warmup:]
        val = sum(f for _, f, _ in per) / sum(s_ for s_, _, _ in per) / 1e12
        rows = per[0][2]
        sample = (f"query rows [0, {rows}) of head (b=0, h=0) of {w.B * w.H} per step against all {w.Sk} keys, "
                  "float64 NumPy")
        cfg = workload_config(w, l2)
        cfg["step"] = "NVFP4 pack of Q and K, then the FP4 QK / BF16 PV attention kernel (O, LSE)"
        print(json.dumps({"impl": "reference", "metric": METRIC_INFER, "value": val, "unit": "TFLOP/s",
                          "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": 1e3 * sum(s_ for s_, _, _ in per) / args.steps,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": cfg,
                          "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": os.cpu_count(),
                                           "kind": "oracle", "sample": sample},
                          "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0},
                          "wall_s": time.perf_counter() - t0}))
        return

    if args.impl == "reference":
        if rank != 0:
            return
        t0 = time.perf_counter()
        per = []
        for _ in range(args.warmup + args.steps):
            per.append(oracle_heads(w, [(0, 0)]))
        per = per[args.warmup:]
        bwd_s = sum(r["bwd_s"] for r in per)
        val = sum(r["bwd_flops"] for r in per) / bwd_s / 1e12
        sample = f"backward of head (b=0, h=0) of {w.B * w.H} per step (full {w.Sq}x{w.Sk}), float64 NumPy"
        line = {"impl": "reference", "metric": METRIC, "value": val,
                "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": 1e3 * (bwd_s + sum(r["fwd_s"] for r in per)) / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": workload_config(w, l2),
                "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "wall_s": time.perf_counter() - t0}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if path == "infer":
        r = run_infer(args, w, rank, world, local_rank)
        if rank != 0:
            torch.distributed.destroy_process_group()
            return
        line = infer_line(args, w, world, r, peaks, l2)
        if not args.no_cpu_baseline and world == 1:
            secs, fl, rows = infer_oracle_rows(w, 10.0)
            line["cpu_baseline"] = {"value": fl / secs / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
                                    "kind": "oracle",
                                    "sample": f"query rows [0, {rows}) of head (0, 0) against all {w.Sk} keys: "
                                              f"{secs:.2f} s, float64 NumPy (BLAS on all cores)"}
        print(json.dumps(line))
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    heads = shard_heads(w, world, rank) if args.shard == "heads" else None
    r = run_ours(args, w, rank, world, local_rank, heads)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    wr = rank_workload(w, heads)               # what rank 0 ran
    # whole-job FLOPs per step: the one workload split over the ranks, or one
    # copy of it per rank
    job = 1 if heads is not None else world
    flops_b, flops_f = job * w.bwd_flops(), job * w.fwd_flops()
    value = job_tflops(flops_b, args.steps, 1, r["bwd_ms"])
    main_ms = statistics.mean(r["main_ms"])
    achieved = wr.bwd_flops() / (main_ms * 1e-3) / 1e12
    traffic = None
    if os.path.exists(PROFILE_JSON):
        prof = json.load(open(PROFILE_JSON))
        if prof.get("kernel_hash") == kernel_hash() and prof.get("workload") == w.name and heads is None:
            traffic = prof.get("dram_bytes_per_launch")
    cfg = workload_config(w, l2, args.recipe)
    if world > 1:
        cfg["parallelism"] = (f"data parallel over B*H heads: {world} contiguous slices, rank 0 "
                              f"heads {heads[0]}..{heads[-1]}" if heads is not None
                              else f"{world} replicas of the whole workload")
    line = {
        "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["step_ms"], "higher_is_better": True,
        "scaling": "strong" if heads is not None else "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": cfg,
        "fwd_tflops": job_tflops(flops_f, args.steps, 1, r["fwd_ms"]),
        "step_tflops": (flops_f + flops_b) / (r["step_ms"] * 1e-3) / 1e12,
        "bwd_ms": r["bwd_ms"] / args.steps, "fwd_ms": r["fwd_ms"] / args.steps,
        "roofline": {"bound": "tensor", "kernel": "bwd_fp4_kernel (attnqat_bwd_main, D = 128)", "achieved": achieved,
                     "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16"],
                     "traffic": traffic, "launch_ms": main_ms,
                     "peak_note": f"{peaks['src']} dense BF16 burst (cuBLAS); sustained {peaks['bf16_sustained']}"},
        "e2e": {"value": flops_b / (r["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms": r["e2e_ms"],
                "what": ("attnqat_bwd_host with pinned host inputs (dO, Q, K, V, O', LSE) and outputs (dQ, dK, dV); "
                         f"chunks={args.e2e_chunks}: head groups of ceil(B*H/{args.e2e_chunks}) heads, the first and "
                         "last of half that, copies overlapping the kernels")},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
