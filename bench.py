"""GPTQ seconds per layer on one B300: Hessian + damping/factor + sweep (+ deferred GEMMs) + packing.

One step = one pass of the whole path over one synthetic layer:
    H = 0; gptq_hessian_accumulate(H, X); gptq_quantize_layer(W, H, ...)
(+ gptq_weight_error and eora_compensate on the EoRA workloads, + cycles of
eora_compensate and gptq_bidup on the refinement workloads; on the
GPTQ-intrinsic LoRA workloads gptq_lora_basis and gptq_intrinsic_lora in place
of gptq_quantize_layer; the packed-layer workloads time gptq_packed_linear)
with X and W resident in HBM.  X (2.15 GB for the default workload) is larger
than the 126 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line.  Under torchrun (N > 1) every rank quantizes its own copy
of the layer (independent replicas, no collective on the data path) and
rank 0 prints the aggregate: layers processed by all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import datetime
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

from synthetic import CHUNK_ROWS, LAYERS, generate, generate_rows  # noqa: E402

METRIC = "GPTQ sec per layer (Hessian+Cholesky+sweep+pack) at 1 B300; % of roofline"
# The largest single-GPU quantization workload: the widest layer (11008 inputs), the largest X (5.77 GB),
# Hessian and factor.
DEFAULT_WORKLOAD = "llama7b_down_proj_4096x11008"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}, "fallback"


# Token slices of X in the end-to-end leg (copy of slice i+1 overlaps the Hessian of slice i).
E2E_CHUNKS = 8


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def mark(self, which: str):
        """Record the wall-clock start or end of the timed region."""
        setattr(self, which, datetime.datetime.now())

    def summary(self):
        """Median SM clock and active throttle reasons over the samples taken inside the timed region."""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "start", None), getattr(self, "stop", None)
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f")
                if t0 is not None and t1 is not None and not (t0 <= ts <= t1):
                    continue
                sm.append(float(p[2]))
                mx.append(float(p[3]))
            except ValueError:
                continue
            for name, v in zip(names, p[6:10]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def describe_inputs(spec) -> str:
    """The synthetic recipe of the workload, for the JSON line."""
    x = spec.X
    dist = {"t": f"Student-t({x.nu:g})", "normal": "N(0,1)", "absnormal_x_normal": "|N(0,1)|*N(0,1)"}[x.dist]
    out = f" with {x.n_outliers} outlier channels x{x.outlier_scale:g}" if x.n_outliers else ""
    return (f"synthetic, seeded: X {x.rows}x{x.cols} {x.dtype} {dist}{out}; "
            f"W {spec.rows}x{spec.cols} {spec.W.dtype} N(0,{spec.W.std:g}^2)")


def max_over_ranks(ms_local: float, world: int, device=None) -> float:
    """The slowest rank's time: every rank quantizes its own layer, the job ends with the last."""
    if world <= 1:
        return ms_local
    import torch
    import torch.distributed as dist

    on_cpu = dist.get_backend() == "gloo"
    t = torch.tensor([ms_local], dtype=torch.float64, device="cpu" if on_cpu else device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def seconds_per_layer(ms_per_step: float, world: int) -> float:
    """Whole-job value: world ranks each finish one layer per step, so the job spends
    ms_per_step / world per layer."""
    return ms_per_step / 1e3 / world


# --------------------------------------------------------------------------- ours
def run_ours(args, rank: int, world: int):
    import torch

    import post_weight_quantization_30_b300 as gq

    spec = LAYERS[args.workload]
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    # --split tokens (N > 1): one layer for the whole job.  Each rank accumulates H over its own
    # range of tokens, one NCCL all-reduce sums H, and each rank quantizes its own range of rows.
    split = args.split == "tokens" and world > 1
    if split and (spec.eora_rank or spec.lora_rank or spec.refine_cycles):
        raise SystemExit("--split tokens runs the plain GPTQ workloads")
    from post_weight_quantization_30_b300 import sharding

    t_lo, t_hi = sharding.token_range(spec.n, world, rank, CHUNK_ROWS) if split else (0, spec.n)
    r_lo, r_hi = sharding.row_range(spec.rows, world, rank) if split else (0, spec.rows)

    # Inputs: seeded host generation (spawn pool), then resident in HBM.
    t0 = time.time()
    def host_tensor(ts, r0=0, r1=None):
        # Rows [r0, r1) of the tensor; bf16 tensors travel as their raw 16-bit patterns, float32 as is.
        r1 = ts.rows if r1 is None else r1
        if ts.dtype == "bf16":
            h = torch.empty((r1 - r0, ts.cols), dtype=torch.int16, pin_memory=True)
            generate_rows(ts, r0, r1, out=h.numpy().view(np.uint16))
        else:
            h = torch.empty((r1 - r0, ts.cols), dtype=torch.float32, pin_memory=True)
            generate_rows(ts, r0, r1, out=h.numpy())
        return h

    def to_dev(h, dst=None):
        if h.dtype == torch.int16:
            if dst is None:
                return h.to(dev).view(torch.bfloat16)
            dst.view(torch.int16).copy_(h, non_blocking=True)
            return dst
        if dst is None:
            return h.to(dev)
        dst.copy_(h, non_blocking=True)
        return dst

    x_host = host_tensor(spec.X, t_lo, t_hi)
    w_host = host_tensor(spec.W)[r_lo:r_hi] if split else host_tensor(spec.W)
    gen_s = time.time() - t0
    X = to_dev(x_host)
    W = to_dev(w_host)
    R, C, N = r_hi - r_lo, spec.cols, t_hi - t_lo  # this rank's rows and tokens
    H = torch.zeros((C, C), dtype=torch.float32, device=dev)
    ws = torch.empty(gq.lib.gptq_quantize_layer_workspace_size(R, C, spec.block), dtype=torch.uint8, device=dev)
    r = spec.eora_rank
    rl = spec.lora_rank
    rc = spec.refine_cycles
    # Ŵ is an output only when EoRA or the intrinsic LoRA needs it (the error they compensate is W - Ŵ);
    # the refinement also needs the codes.
    out = gq._lib._sweep_outputs(R, C, spec.bits, spec.group, dev, codes=rc > 0, W_hat=(r or rl) > 0,
                                 row_err=False)
    if rc:
        bu_ws = torch.empty(gq.lib.gptq_bidup_workspace_size(R, C), dtype=torch.uint8, device=dev)
    if rl:
        ws = torch.empty(gq.lib.gptq_intrinsic_lora_workspace_size(R, C, rl, spec.block), dtype=torch.uint8,
                         device=dev)
        bws = torch.empty(gq.lib.gptq_lora_basis_workspace_size(C, rl), dtype=torch.uint8, device=dev)
        bout = dict(Lt=torch.empty((rl, C), dtype=torch.float32, device=dev),
                    lam=torch.empty(rl, dtype=torch.float32, device=dev))
        out["R"] = torch.empty((R, rl), dtype=torch.float32, device=dev)
    if r:
        dW = torch.empty((R, C), dtype=torch.float32, device=dev)
        ews = torch.empty(gq.lib.eora_compensate_workspace_size(R, C, r), dtype=torch.uint8, device=dev)
        eout = dict(A=torch.empty((r, C), dtype=torch.float32, device=dev),
                    B=torch.empty((R, r), dtype=torch.float32, device=dev),
                    sigma=torch.empty(r, dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream(dev)

    def eora_part(Wsrc):
        gq.gptq_weight_error(Wsrc, out["W_hat"], out=dW)
        gq.eora_compensate(dW, H, r, workspace=ews, out=eout)

    def refine_part(Wsrc):
        # rc cycles of OLrC (EoRA of W - Ŵ) then Bid-Up against W - B A; codes, Ŵ and qweight refined in place
        for _ in range(rc):
            eora_part(Wsrc)
            gq.gptq_bidup(Wsrc, H, out["codes"], out["scales"], out["qzeros"], spec.bits, spec.group, eout["A"],
                          eout["B"], W_hat=out["W_hat"], qweight=out["qweight"], workspace=bu_ws)

    def quantize(Wsrc):
        if rl:
            gq.gptq_lora_basis(H, rl, workspace=bws, out=bout)
            gq.gptq_intrinsic_lora(Wsrc, H, bout["Lt"], spec.bits, spec.group, spec.block, spec.damp, workspace=ws,
                                   out=out)
            return
        gq.gptq_quantize_layer(Wsrc, H, spec.bits, spec.group, spec.block, spec.damp, workspace=ws, out=out)
        if rc:
            refine_part(Wsrc)
        elif r:
            eora_part(Wsrc)

    def reduce_h():
        if split:
            sharding.reduce_hessian(H)  # NCCL all-reduce (sum) on the current stream

    def step(ev=None):
        H.zero_()
        if ev is not None:
            ev[0].record(stream)
        gq.gptq_hessian_accumulate(H, X)
        if ev is not None:
            ev[1].record(stream)
        reduce_h()
        quantize(W)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    import torch.distributed as dist

    hev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clocks:
        time.sleep(0.3)  # let the sampler start before the timed region
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        launches0 = gq.lib.gq_kernel_launches()
        clocks.mark("start")
        start.record(stream)
        for k in range(args.steps):
            step(hev[k])
        stop.record(stream)
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()
        clocks.mark("stop")
        launches = gq.lib.gq_kernel_launches() - launches0
        time.sleep(0.15)
    ms_total = start.elapsed_time(stop)
    h_ms = [a.elapsed_time(b) for a, b in hev]
    ms_total = max_over_ranks(ms_total, world, dev)
    ms_per_step = ms_total / args.steps

    # Per-phase breakdown (untimed for the headline): factor and sweep separately.
    phase = {}
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    F = torch.empty((C, C), dtype=torch.float32, device=dev)
    dead = torch.empty(C, dtype=torch.uint8, device=dev)
    fws = torch.empty(max(256, gq.lib.gptq_factor_workspace_size(C)), dtype=torch.uint8, device=dev)
    sws = torch.empty(gq.lib.gptq_sweep_workspace_size(R, C, spec.block), dtype=torch.uint8, device=dev)
    import ctypes

    reps = 3
    acc = {"hessian": 0.0, "factor": 0.0, "sweep": 0.0}
    if rl:
        acc = {"hessian": 0.0, "basis": 0.0, "intrinsic_lora": 0.0}
        for _ in range(reps):
            H.zero_()
            e[0].record(stream)
            gq.gptq_hessian_accumulate(H, X)
            e[1].record(stream)
            gq.gptq_lora_basis(H, rl, workspace=bws, out=bout)
            e[2].record(stream)
            gq.gptq_intrinsic_lora(W, H, bout["Lt"], spec.bits, spec.group, spec.block, spec.damp, workspace=ws,
                                   out=out)
            e[3].record(stream)
            torch.cuda.synchronize(dev)
            acc["hessian"] += e[0].elapsed_time(e[1])
            acc["basis"] += e[1].elapsed_time(e[2])
            acc["intrinsic_lora"] += e[2].elapsed_time(e[3])
        reps_done = True
    else:
        reps_done = False
    if r:
        acc["eora" if not rc else "refine"] = 0.0
        e.append(torch.cuda.Event(enable_timing=True))
    for _ in range(0 if reps_done else reps):
        H.zero_()
        e[0].record(stream)
        gq.gptq_hessian_accumulate(H, X)
        e[1].record(stream)
        info = ctypes.c_int64(-1)
        st = gq.lib.gptq_factor(ctypes.c_void_p(H.data_ptr()), C, spec.damp, ctypes.c_void_p(F.data_ptr()),
                                ctypes.c_void_p(dead.data_ptr()), ctypes.c_void_p(fws.data_ptr()), fws.numel(),
                                ctypes.c_void_p(stream.cuda_stream), ctypes.byref(info))
        assert st == 0, st
        e[2].record(stream)
        so = gq.gptq_sweep(W, F, dead, spec.bits, spec.group, spec.block, codes=rc > 0, W_hat=r > 0, row_err=False,
                           workspace=sws)
        e[3].record(stream)
        if rc:
            for kk in ("codes", "W_hat"):
                out[kk].copy_(so[kk])
            refine_part(W)
            e[4].record(stream)
        elif r:
            gq.gptq_weight_error(W, so["W_hat"], out=dW)
            gq.eora_compensate(dW, H, r, workspace=ews, out=eout)
            e[4].record(stream)
        torch.cuda.synchronize(dev)
        acc["hessian"] += e[0].elapsed_time(e[1])
        acc["factor"] += e[1].elapsed_time(e[2])
        acc["sweep"] += e[2].elapsed_time(e[3])
        if r:
            acc["eora" if not rc else "refine"] += e[3].elapsed_time(e[4])
    phase = {k: v / reps for k, v in acc.items()}

    # One more untimed step with the library's per-launch CUDA events on (a breakdown by
    # kernel class: summed time, launches and useful flops each launcher declares).
    torch.cuda.synchronize(dev)
    with gq.kernel_timing() as kt:
        step()
    torch.cuda.synchronize(dev)

    # End to end through the public API from pinned host buffers, every step:
    # H2D of X and W, the whole path, D2H of the packed result.  X arrives in
    # E2E_CHUNKS slices of tokens on a copy stream, and H accumulates each slice
    # as soon as it has landed (H is a sum over tokens), so the host link and the
    # tensor cores overlap, as when calibration batches stream in.
    results = {k: v for k, v in out.items() if v is not None and k != "W_hat"}
    if rl:
        results.update(lora_Lt=bout["Lt"])
    if r:
        results.update(eora_A=eout["A"], eora_B=eout["B"])
    res_host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in results.items()}
    h2d = x_host.numel() * x_host.element_size() + w_host.numel() * w_host.element_size()
    d2h = sum(v.numel() * v.element_size() for v in res_host.values())
    Xd = torch.empty_like(X)
    Wd = torch.empty_like(W)
    torch.cuda.synchronize(dev)
    e2e_steps = max(2, min(args.steps, 5))
    copy_stream = torch.cuda.Stream(dev)
    bounds = [N * i // E2E_CHUNKS for i in range(E2E_CHUNKS + 1)]
    landed = [torch.cuda.Event() for _ in range(E2E_CHUNKS + 1)]
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        copy_stream.wait_stream(stream)  # the previous step's reads of Xd and Wd are done
        with torch.cuda.stream(copy_stream):
            for i in range(E2E_CHUNKS):
                to_dev(x_host[bounds[i]:bounds[i + 1]], Xd[bounds[i]:bounds[i + 1]])
                landed[i].record(copy_stream)
            to_dev(w_host, Wd)
            landed[E2E_CHUNKS].record(copy_stream)
        H.zero_()
        for i in range(E2E_CHUNKS):
            stream.wait_event(landed[i])
            gq.gptq_hessian_accumulate(H, Xd[bounds[i]:bounds[i + 1]])
        reduce_h()
        stream.wait_event(landed[E2E_CHUNKS])
        quantize(Wd)
        for k, v in res_host.items():
            v.copy_(results[k], non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t0) / e2e_steps

    peaks, peak_kind = _peaks()
    flops = float(N) * C * (C + 1)  # symmetric work of H += 2 X^T X
    h_avg_s = statistics.mean(h_ms) / 1e3
    achieved = flops / h_avg_s / 1e12
    # The Hessian runs for milliseconds inside a step of tens of milliseconds, at the maximum
    # clock: the burst peak (a seconds-long loop settles at the sustained one).
    peak = peaks["bf16_tflops"]
    bound, peak_kind = "tensor", f"{peak_kind} bf16 dense burst"
    if spec.X.dtype != "bf16":
        # float32 X runs the float32 SIMT product: 148 SMs x 128 FMA/clk x 2 flops x 2.032 GHz.
        bound, peak, peak_kind = "alu", round(148 * 128 * 2 * peaks.get("sm_max_mhz", 2032.0) * 1e6 / 1e12, 1), \
            "float32 FMA issue rate from SM count and maximum clock"
    traffic = _read_traffic(args.workload)
    rooflines = phase_rooflines(spec, phase, kt, peaks, _peaks()[1], codes=rc > 0, w_hat=(r or rl) > 0)

    result = {
        "metric": METRIC,
        "value": round(ms_per_step / 1e3 if split else seconds_per_layer(ms_per_step, world), 6),
        "unit": "s/layer",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": False,
        "scaling": "strong" if split else "weak",
        "vs_baseline": None,
        "dtype": "bf16 x bf16 -> f32 (Hessian); f32 (factor, sweep, 3xTF32 GEMMs" +
                 (", OLrC + Bid-Up)" if rc else ", EoRA)" if r else ", intrinsic LoRA)" if rl else ")"),
        "data": describe_inputs(spec),
        "config": {
            "workload": args.workload, "rows": spec.rows, "cols": C, "tokens": spec.n, "bits": spec.bits,
            "group": spec.group,
            "block": spec.block, "damp": spec.damp, "x_dtype": spec.X.dtype, "w_dtype": spec.W.dtype,
            "l2": "inputs larger than L2 (X %.2f GB > 126 MB), no flush" % (spec.X.nbytes / 1e9),
            "parallelism": (f"tokens split for H ({N} of {spec.n} on rank {rank}) + one NCCL all-reduce of H, rows "
                            f"split for the factor-and-sweep ({R} of {spec.rows})" if split else
                            "replicas" if world > 1 else "single GPU"),
        },
        "phases_ms": {k: round(v, 4) for k, v in phase.items()},
        "roofline": {
            "kernel": "hessian_pair_kernel (H += 2 X^T X)",
            "bound": bound, "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
            "flops_per_launch": flops, "traffic": traffic,
        },
        "rooflines": rooflines,
        "kernel_classes": {k: {"ms": round(kt.ms[k], 4), "launches": kt.count[k], "flops": kt.flops[k]}
                           for k in kt.ms if kt.count[k]},
        "e2e": {"value": round(e2e_s, 6), "unit": "s/layer", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
        "input_generation_s": round(gen_s, 1),
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        result["cpu_baseline"] = cpu_baseline(spec, **ORACLE_SAMPLE)
    return result


def sweep_pack_bytes(spec, codes: bool, w_hat: bool) -> float:
    """Algorithmic HBM bytes of the sweep + packing: W read once, the packed codes, the per-group
    scales (float32) and zero points, the diagonal of the factor, and the optional codes (1 byte)
    and Ŵ (float32) outputs."""
    R, C, b, g = spec.rows, spec.cols, spec.bits, spec.group
    wbytes = 2 if spec.W.dtype == "bf16" else 4
    byt = R * C * wbytes + R * C * b / 8 + (C // g) * R * (4 + b / 8) + C * 4
    if codes:
        byt += R * C
    if w_hat:
        byt += R * C * 4
    return float(byt)


def phase_rooflines(spec, phase: dict, kt, peaks: dict, peak_kind: str, codes: bool, w_hat: bool) -> dict:
    """Roofline of each phase of the step and of the 3xTF32 GEMMs as a class.

    * factor: one Cholesky of the cols x cols damped H, cols^3 / 3 useful flops, against the useful
      float32 rate of 3xTF32 on the tensor cores (the measured bf16 burst x 1.1 / 2.25, the nominal
      dense tf32 : bf16 ratio, x 1/3 for the three TF32 products per useful product);
    * sweep_pack: the algorithmic bytes of sweep_pack_bytes against the measured HBM copy rate; the
      phase also runs the in-block updates and the deferred trailing GEMMs, and its floor is the
      chain of cols dependent column steps, reported as chain_floor_ms = cols x the measured time of
      one column step of the block kernel;
    * gemm3: every 3xTF32 GEMM launch of one step, the useful flops they declare over their summed
      CUDA-event time, against the same 3xTF32 rate.
    """
    C = spec.cols
    tf32x3 = peaks["bf16_tflops"] * (1.1 / 2.25) / 3
    tf32_kind = (f"{peak_kind} bf16 dense burst x 1.1/2.25 (nominal dense tf32 : bf16) x 1/3 (three TF32 products "
                 f"per useful product)")
    out = {}
    if phase.get("factor"):
        fl = C ** 3 / 3
        a = fl / (phase["factor"] / 1e3) / 1e12
        out["factor"] = {"bound": "tensor", "achieved": round(a, 2), "peak": round(tf32x3, 1), "unit": "TFLOP/s",
                         "frac": round(a / tf32x3, 4), "peak_kind": tf32_kind, "flops_per_call": fl,
                         "phase_ms": round(phase["factor"], 4),
                         "diagonal_block_chain_ms": round(kt.ms["diag"], 4), "diagonal_blocks": kt.count["diag"],
                         "traffic": None}
    if phase.get("sweep"):
        byt = sweep_pack_bytes(spec, codes, w_hat)
        a = byt / (phase["sweep"] / 1e3) / 1e9
        n_sw = kt.count["sweep"]
        # Every column is one step of the block kernels (a launch sweeps one or two blocks).
        t_step_ns = kt.ms["sweep"] * 1e6 / C if n_sw else None
        out["sweep_pack"] = {"bound": "hbm", "achieved": round(a, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(a / peaks["hbm_gbs"], 4), "peak_kind": f"{peak_kind} HBM copy",
                             "bytes_per_call": byt, "phase_ms": round(phase["sweep"], 4),
                             "block_kernel_ms": round(kt.ms["sweep"], 4), "block_launches": n_sw,
                             "column_step_ns": round(t_step_ns, 2) if t_step_ns else None,
                             "chain_floor_ms": round(C * t_step_ns / 1e6, 4) if t_step_ns else None,
                             "traffic": None}
    if kt.count["gemm3"]:
        a = kt.flops["gemm3"] / (kt.ms["gemm3"] / 1e3) / 1e12
        out["gemm3"] = {"bound": "tensor", "achieved": round(a, 2), "peak": round(tf32x3, 1), "unit": "TFLOP/s",
                        "frac": round(a / tf32x3, 4), "peak_kind": tf32_kind, "launches": kt.count["gemm3"],
                        "ms": round(kt.ms["gemm3"], 4), "useful_flops": kt.flops["gemm3"], "traffic": None}
    if kt.count["hessian"]:
        a = kt.flops["hessian"] / (kt.ms["hessian"] / 1e3) / 1e12
        out["hessian"] = {"bound": "tensor", "achieved": round(a, 2), "peak": peaks["bf16_tflops"],
                          "unit": "TFLOP/s", "frac": round(a / peaks["bf16_tflops"], 4),
                          "peak_kind": f"{peak_kind} bf16 dense burst", "ms": round(kt.ms["hessian"], 4),
                          "launches": kt.count["hessian"]}
    return out


def _read_traffic(workload: str):
    """DRAM bytes per launch of the Hessian kernel from the committed ncu summary,
    if it was taken on this workload and the kernel source is unchanged since."""
    import hashlib

    p = os.path.join(ROOT, "profiles", "hessian_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        src = b"".join(open(os.path.join(ROOT, "post_weight_quantization_30_b300", "csrc", n), "rb").read()
                       for n in ("hessian_tc.cu", "tc_common.cuh"))
    except (OSError, ValueError):
        return None
    if hashlib.sha256(src).hexdigest() != rec.get("kernel_source_sha256"):
        return None
    if not str(rec.get("workload", "")).startswith(workload):
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------- packed layer (inference)
PACKED_METRIC = "packed quantized linear Y = X What^T (+ (X A^T) B^T): seconds per call at 1 B300; % of roofline"


def _packed_bytes(spec, n, r) -> float:
    """Bytes one call must move at least: packed weights, scales, zeros, X, Y (and the adapter)."""
    R, C, b = spec.rows, spec.cols, spec.bits
    byt = R * C * b / 8 + (C // spec.group) * R * 4 + (C // spec.group) * R * b / 8 + n * C * 2 + n * R * 4
    if r:
        byt += (r * C + R * r) * 4
    return float(byt)


def run_packed(args, rank: int, world: int):
    """The quantized layer applied from its packed form to n tokens.  Setup (untimed): the layer is
    quantized by the library from a calibration set; the adapter (if any) is seeded random.  A step
    is one gptq_packed_linear call; the K timed steps are captured as one CUDA graph and replayed
    (no host launch cost between calls, as in a serving loop); e2e calls the API eagerly with the
    tokens copied in and Y copied out every step."""
    from dataclasses import replace

    import torch

    import post_weight_quantization_30_b300 as gq

    spec = LAYERS[args.workload]
    n, r = spec.packed_tokens, spec.eora_rank
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    R, C = spec.rows, spec.cols

    def host(ts):
        h = torch.empty((ts.rows, ts.cols), dtype=torch.int16, pin_memory=True)
        generate(ts, out=h.numpy().view(np.uint16))
        return h

    t0 = time.time()
    calib = replace(spec.X, rows=8192, key=spec.X.key + (7,))
    x_host = host(spec.X)
    Xc = host(calib).to(dev).view(torch.bfloat16)
    W = host(spec.W).to(dev).view(torch.bfloat16)
    X = x_host.to(dev).view(torch.bfloat16)
    gen_s = time.time() - t0
    H = torch.zeros((C, C), dtype=torch.float32, device=dev)
    gq.gptq_hessian_accumulate(H, Xc)
    q = gq.gptq_quantize_layer(W, H, spec.bits, spec.group, spec.block, spec.damp, codes=False, W_hat=False,
                               row_err=False)
    del Xc, H
    g = torch.Generator(device=dev).manual_seed(0)
    A = (torch.randn((r, C), device=dev, generator=g) * 0.01) if r else None
    B = (torch.randn((R, r), device=dev, generator=g) * 0.01) if r else None
    Y = torch.empty((n, R), dtype=torch.float32, device=dev)
    wsb = gq.lib.gptq_packed_linear_workspace_size(n, R, C, spec.group, r)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)

    def call(Xin):
        gq.gptq_packed_linear(Xin, q["qweight"], q["scales"], q["qzeros"], R, C, spec.bits, spec.group, A, B, out=Y,
                              workspace=ws)

    for _ in range(max(1, args.warmup)):
        call(X)
    torch.cuda.synchronize(dev)
    l0 = gq.lib.gq_kernel_launches()
    call(X)
    torch.cuda.synchronize(dev)
    launches_per_call = gq.lib.gq_kernel_launches() - l0
    # The K timed steps as one CUDA graph (K calls), replayed once untimed (warm-up, K >= W calls)
    # and once timed.
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for _ in range(args.steps):
                call(X)
    graph.replay()
    torch.cuda.synchronize(dev)
    gq.gq_check_device()
    stream = torch.cuda.current_stream(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # A call can take microseconds, far below the 100 ms clock-sampling period, so the clocks are
    # sampled over a window of >= 0.3 s of the same replays on each side of the timed region.
    def soak(seconds):
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            graph.replay()
            torch.cuda.synchronize(dev)

    with ClockSampler(dev.index) as clocks:
        time.sleep(0.3)
        clocks.mark("start")
        soak(0.3)
        start.record(stream)
        graph.replay()
        stop.record(stream)
        torch.cuda.synchronize(dev)
        soak(0.3)
        clocks.mark("stop")
        time.sleep(0.15)
    gq.gq_check_device()
    ms = max_over_ranks(start.elapsed_time(stop), world, dev) / args.steps

    # End to end: tokens in from pinned host memory, the eager API call, Y out, every step.
    y_host = torch.empty((n, R), dtype=torch.float32, pin_memory=True)
    Xd = torch.empty_like(X)
    e2e_steps = max(3, min(args.steps, 20))
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    for _ in range(e2e_steps):
        Xd.view(torch.int16).copy_(x_host, non_blocking=True)
        call(Xd)
        y_host.copy_(Y, non_blocking=True)
        torch.cuda.synchronize(dev)
    e2e_s = (time.perf_counter() - t1) / e2e_steps

    peaks, peak_kind = _peaks()
    flops = 2.0 * n * R * C + (2.0 * n * r * (R + C) if r else 0.0)
    if n > 32:
        roof = {"kernel": "packed_linear_kernel (tensor cores)", "bound": "tensor",
                "achieved": round(flops / (ms / 1e3) / 1e12, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "peak_kind": f"{peak_kind} bf16 dense burst (kernel timed alone)",
                "flops_per_launch": flops}
        roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    else:
        byt = _packed_bytes(spec, n, r)
        roof = {"kernel": "packed_gemv_kernel + packed_reduce_kernel (decode path)", "bound": "hbm",
                "achieved": round(byt / (ms / 1e3) / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "peak_kind": f"{peak_kind} HBM copy", "bytes_per_launch": byt}
        roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = None
    result = {
        "metric": PACKED_METRIC,
        "value": round(ms / 1e3 / world, 9),
        "unit": "s/call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 X x exact (q - z) integers -> f32, per-group f32 scale" + ("; f32 adapter" if r else ""),
        "data": (f"synthetic, seeded: {describe_inputs(spec)}; W quantized by gptq_quantize_layer with H from 8192 "
                 f"calibration tokens of the same distribution"
                 + (f"; adapter A {r}x{C}, B {R}x{r} seeded N(0,0.01^2)" if r else "")),
        "config": {"workload": args.workload, "rows": R, "cols": C, "tokens": n, "bits": spec.bits,
                   "group": spec.group, "adapter_rank": r, "graph_replay": True,
                   "l2": "no flush; packed weights fit in L2 across calls" if n <= 32 else "no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tokens_per_s": round(n * world / (ms / 1e3), 1),
        "roofline": roof,
        "e2e": {"value": round(e2e_s, 9), "unit": "s/call", "h2d_bytes_per_step": n * C * 2,
                "d2h_bytes_per_step": n * R * 4},
        "gpu_launches": launches_per_call * args.steps,
        "clocks": dict(clocks.summary(), window="the timed region plus 0.3 s of the same graph replays on each side"),
        "input_generation_s": round(gen_s, 1),
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        result["cpu_baseline"] = cpu_baseline(spec, **ORACLE_SAMPLE)
    return result


def cpu_baseline_packed(spec) -> dict:
    """The float64 oracle of the packed layer on a sample of the tokens, scaled to the call."""
    from oracle import pack as opk
    from oracle import packed_linear as pl
    from synthetic import bf16_bits_to_f32

    n = spec.packed_tokens
    n_s = min(n, 64)
    cores = len(os.sched_getaffinity(0))
    rng = np.random.default_rng(0)
    R, C, b, g = spec.rows, spec.cols, spec.bits, spec.group
    codes = rng.integers(0, 2 ** b, (R, C)).astype(np.uint8)
    zeros = rng.integers(0, 2 ** b, (C // g, R)).astype(np.uint8)
    scales = rng.uniform(0.005, 0.05, (C // g, R)).astype(np.float32)
    qw, qz = opk.pack_qweight(codes, b), opk.pack_qzeros(zeros, b)
    x = bf16_bits_to_f32(generate_rows(spec.X, 0, n_s, workers=1)).astype(np.float64)
    r = spec.eora_rank
    A = rng.standard_normal((r, C)) * 0.01 if r else None
    B = rng.standard_normal((R, r)) * 0.01 if r else None
    t0 = time.perf_counter()
    W_hat = pl.dequantize(qw, scales, qz, b, g, R, C)
    t1 = time.perf_counter()
    Y = x @ W_hat.T
    if r:
        Y = Y + (x @ A.T) @ B.T
    t2 = time.perf_counter()
    assert Y.shape == (n_s, R)
    per_call = (t1 - t0) + (t2 - t1) * n / n_s
    return {"value": round(per_call, 4), "unit": "s/call", "cores": cores, "kind": "oracle",
            "sample": f"unpack + dequantize the whole layer once, then the float64 product on {n_s} of {n} tokens "
                      f"(x{n / n_s:g})", "sample_s": round(t2 - t0, 2)}


# ----------------------------------------------------------------- oracle (CPU)
def cpu_baseline(spec, n_s: int = 4096, r_s: int = 16, factor_cols: int | None = None) -> dict:
    """The float64 oracle, as it stands, on a bounded sample of the same layer,
    extrapolated to seconds per layer: H on n_s tokens (scaled by N / n_s); damping
    + inverse + Cholesky of the whole cols x cols H, or of its leading
    factor_cols x factor_cols block scaled by (cols / factor_cols)^3 (the work is
    cubic); the eager sweep on r_s rows (scaled by rows / r_s, and by
    (cols / factor_cols)^2 when the sweep runs on the leading block: its work per
    row is quadratic in cols); packing of those rows (scaled by rows / r_s and
    cols / factor_cols)."""
    if spec.packed_tokens:
        return cpu_baseline_packed(spec)
    from oracle import gptq as og
    from oracle import pack as opk
    from synthetic import bf16_bits_to_f32

    cores = len(os.sched_getaffinity(0))
    n_s = min(n_s, spec.n)
    r_s = min(r_s, spec.rows)
    k = spec.cols if factor_cols is None or spec.lora_rank else min(factor_cols, spec.cols)
    k -= k % spec.group
    key = (spec.X, spec.W, n_s, r_s)
    if key not in _SAMPLES:  # the sampled inputs, generated once per process (not timed)
        x = bf16_bits_to_f32(generate_rows(spec.X, 0, n_s, workers=1)) if spec.X.dtype == "bf16" else \
            generate_rows(spec.X, 0, n_s, workers=1)
        w = generate_rows(spec.W, 0, r_s, workers=1)
        _SAMPLES.clear()
        _SAMPLES[key] = (x, (bf16_bits_to_f32(w) if spec.W.dtype == "bf16" else w).astype(np.float64))
    x, w = _SAMPLES[key]
    t0 = time.perf_counter()
    H = og.hessian(x.astype(np.float64)) * (spec.n / n_s)
    t1 = time.perf_counter()
    if spec.lora_rank:
        # GPTQ-intrinsic LoRA: basis by a full eigendecomposition, augmented Hessian, partial sweep.
        from oracle import intrinsic_lora as il

        L, _ = il.top_right_singular_vectors(H, spec.lora_rank)
        Hd, dead = og.prepare_hessian(il.augmented_hessian(H, L), spec.damp)
        U = og.inverse_cholesky_upper(Hd)
        t2 = time.perf_counter()
        res = il.sweep_partial(np.hstack([w, np.zeros((r_s, spec.lora_rank))]), U, spec.bits, spec.group, spec.cols,
                               dead=dead)
    else:
        Hd, dead = og.prepare_hessian(H[:k, :k], spec.damp)
        U = og.inverse_cholesky_upper(Hd)
        t2 = time.perf_counter()
        res = og.sweep(w[:, :k], U, spec.bits, spec.group, dead=dead)
    t3 = time.perf_counter()
    opk.pack_qweight(res["codes"], spec.bits)
    t4 = time.perf_counter()
    c = spec.cols / k
    ph = {"hessian": (t1 - t0) * spec.n / n_s, "factor": (t2 - t1) * c ** 3,
          "sweep": (t3 - t2) * spec.rows / r_s * c ** 2, "pack": (t4 - t3) * spec.rows / r_s * c}
    per_layer = sum(ph.values())
    if spec.lora_rank:
        fac = (f"full float64 eigendecomposition for the rank-{spec.lora_rank} basis, inverse + Cholesky of the "
               f"augmented {spec.cols + spec.lora_rank}x{spec.cols + spec.lora_rank} Hessian; ")
    elif k == spec.cols:
        fac = f"full float64 inverse + Cholesky of {spec.cols}x{spec.cols}; "
    else:
        fac = (f"float64 inverse + Cholesky of the leading {k}x{k} block of H (x{c ** 3:.4g}, cubic in cols); "
               f"the sweep on those {k} columns (x{c ** 2:.4g}, quadratic in cols); ")
    return {
        "value": round(per_layer, 3), "unit": "s/layer", "cores": cores, "kind": "oracle",
        "sample": f"H on {n_s} of {spec.n} tokens (x{spec.n / n_s:g}); " + fac +
                  f"eager sweep + pack on {r_s} of {spec.rows} rows (x{spec.rows / r_s:g})" +
                  ("; the OLrC + Bid-Up cycles not included" if spec.refine_cycles else
                   "; EoRA not included" if spec.eora_rank else ""),
        "sample_s": round(t4 - t0, 2),
        "phases_s": {k_: round(v, 3) for k_, v in ph.items()},
    }


# The sample of the oracle timing, in the bench line's cpu_baseline and in each step of the reference
# arm: bounded so that a reference run of --steps 20 --warmup 5 ends within a few minutes.
ORACLE_SAMPLE = dict(n_s=4096, r_s=16, factor_cols=4096)
_SAMPLES = {}


def run_reference(args):
    spec = LAYERS[args.workload]
    for _ in range(args.warmup):
        cpu_baseline(spec, **ORACLE_SAMPLE)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(spec, **ORACLE_SAMPLE))
    wall = time.perf_counter() - t0
    v = statistics.mean(x["value"] for x in vals)
    packed = bool(spec.packed_tokens)
    cb = dict(vals[-1])
    cb["value"] = round(v, 4 if packed else 3)
    return {
        "impl": "reference",
        "metric": PACKED_METRIC if packed else METRIC, "value": round(v, 4 if packed else 3),
        "unit": "s/call" if packed else "s/layer", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 1), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": args.workload, "rows": spec.rows, "cols": spec.cols, "tokens": spec.n,
                   "bits": spec.bits, "group": spec.group, "block": spec.block},
        "cpu_baseline": cb,
        "e2e": {"value": round(v, 4 if packed else 3), "unit": "s/call" if packed else "s/layer",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(LAYERS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--split", default="replicas", choices=["replicas", "tokens"],
                    help="N > 1: independent replicas (default) or one layer split over the ranks")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    res = run_packed(args, rank, world) if LAYERS[args.workload].packed_tokens else run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
