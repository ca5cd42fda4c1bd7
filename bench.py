"""Benchmark of the GB300 dense GEMM library.

Default workload: the projection GEMMs of one training step of the 6-layer,
d_model = 384 character GPT of "bare-metal-bard" (second paragraph) at batch
64 x context 256 (16384 token rows): for each of the five projections (QKV,
attention out, MLP up, MLP down, LM head) the forward Y = X W, the input
gradient dX = dY W^T and the weight gradient dW = X^T dY, each in FP32 (CUDA
cores) and in TF32 (tensor cores): 30 GEMMs per step.  Activations and
gradients are N(0, 1), weights N(0, 0.02^2), drawn from seeded generators
(seeded_inputs.py); there is no dataset.

One JSON line on rank 0: whole-job TFLOP/s over the timed steps (CUDA events
on the launching stream), the end-to-end figure through the C ABI with the
inputs copied from pinned host memory and the outputs copied back inside the
timed region, the roofline of the dominant kernel, the per-shape breakdown,
and the oracle timed on a bounded sample on the host cores.

`--impl reference` times the CPU oracle (the only reference arm there is:
the pages publish no code) on a bounded sample of the same workload.
`--gpus N` under torchrun runs N independent replicas (GEMM shards with no
exchange), one per rank; value = all ranks' FLOPs / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import seeded_inputs as si  # noqa: E402

METRIC = "GEMM TFLOP/s per shape & % of GB300 roofline (tensor peak or HBM BW), 1 GPU"
SMS = 152
FP32_LANES_PER_SM = 128
SM_MAX_MHZ = 2070.0
# Nominal dense rates (recipe): tf32 1.1 PF, bf16 2.25 PF, fp8 4.5 PF.
TF32_OVER_BF16 = 1.1 / 2.25
FP8_OVER_BF16 = 4.5 / 2.25
FP4_OVER_FP8 = 3.0     # nominal dense FP4 / FP8 tensor rate of this GPU (13.5 / 4.5 PFLOP/s)


# DRAM bytes (read + write) per launch of the dominant kernel, from one ncu
# capture of the step's 15 FP32 GEMM launches (cold L2).  The figure belongs
# to the kernel source it was measured on: if the source's SHA-256 differs,
# "traffic" is reported as null.
PROFILED_TRAFFIC = {
    "fp32": {"source": "dense_gemm_transformer_gb300/csrc/simt.cu", "sha256": "3328d0a225eb74b4",
             "bytes_per_launch": 92.43e6},
}


def profiled_traffic(family):
    import hashlib
    rec = PROFILED_TRAFFIC.get(family)
    if not rec or rec["sha256"] is None:
        return None
    with open(os.path.join(ROOT, rec["source"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != rec["sha256"]:
            return None
    return rec["bytes_per_launch"]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    src = "measured"
    try:
        with open(path) as f:
            p = json.load(f)
        hbm, bf16, bf16_s = p["hbm_gbs"], p["bf16_tflops"], p["bf16_tflops_sustained"]
    except Exception:
        hbm, bf16, bf16_s, src = 6800.0, 1900.0, 1700.0, "fallback"
    fp32_alu = SMS * FP32_LANES_PER_SM * 2 * SM_MAX_MHZ * 1e6 / 1e12
    return {"hbm_gbs": hbm, "bf16_tflops": bf16, "bf16_tflops_sustained": bf16_s,
            "tf32_tflops": bf16 * TF32_OVER_BF16, "tf32_tflops_sustained": bf16_s * TF32_OVER_BF16,
            "fp8_tflops": bf16 * FP8_OVER_BF16, "fp8_tflops_sustained": bf16_s * FP8_OVER_BF16,
            "fp32_alu_tflops": fp32_alu, "source": src}


def measure_fp32_peak(dev, sample_ms=20.0, samples=3):
    """The FP32 FMA roof of this GPU, measured: gemm_launch_fma_peak (16
    independent FMA chains per thread, 4 CTAs of 256 threads per SM) timed
    with CUDA events, in its scalar and packed (fma.rn.f32x2) forms, each the
    median of `samples` launches of >= sample_ms; the roof is the faster
    form.  No clock or other setting of the GPU is touched."""
    import ctypes

    import dense_gemm_transformer_gb300 as dg
    fn = dg.load().gemm_launch_fma_peak
    fn.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    grid = 4 * sms
    out = torch.empty(grid * 256, device=dev)
    stream = torch.cuda.Stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(packed, iters):
        e0.record(stream)
        st = fn(packed, grid, iters, out.data_ptr(), stream.cuda_stream)
        e1.record(stream)
        stream.synchronize()
        if st != 0:
            raise RuntimeError(f"gemm_launch_fma_peak: status {st}")
        return e0.elapsed_time(e1)

    res = {}
    with ClockSampler(dev.index) as clk:
        for packed, name in ((0, "scalar"), (1, "packed")):
            timed(packed, 1000)
            ms = timed(packed, 20000)
            iters = int(20000 * sample_ms / max(ms, 1e-3)) + 1
            runs = sorted(timed(packed, iters) for _ in range(samples))
            med = runs[len(runs) // 2]
            res[name] = grid * 256 * iters * 32 / (med * 1e-3) / 1e12
    res["tflops"] = max(res["scalar"], res["packed"])
    res["clocks"] = clk.summary()
    res["how"] = (f"gemm_launch_fma_peak: {grid} CTAs x 256 threads x 16 FMA chains, median of {samples} "
                  f"launches of >= {sample_ms:g} ms, scalar fma.rn.f32 and packed fma.rn.f32x2; the faster form")
    return res


class Call:
    """One GEMM of the step with its buffers."""

    def __init__(self, case: si.GemmCase, mode: str, A, B, C):
        self.case, self.mode, self.A, self.B, self.C = case, mode, A, B, C

    @property
    def name(self):
        return f"{self.mode}.{self.case.name}"

    def bytes(self):
        es = 2 if self.mode == "bf16" else 4
        c = self.case
        return es * (c.M * c.K + c.K * c.N) + 4 * c.M * c.N


def gpt_workload(device):
    """Inputs X, W, dY of every projection and one output per (mode, GEMM)."""
    inputs = []
    for p, (name, kin, nout) in enumerate(si.GPT_PROJECTIONS):
        X, W, dY = si.gpt_tensors(p, kin, nout)
        inputs += [X, W, dY]
    dev_inputs = [t.to(device) for t in inputs]
    return gpt_calls(dev_inputs, device), inputs, dev_inputs


def gpt_calls(dev_inputs, device):
    """The 30 GEMMs of a step on the given device inputs, each with its own C."""
    calls = []
    cases = si.gpt_cases()
    for mode in ("fp32", "tf32"):
        for p in range(len(si.GPT_PROJECTIONS)):
            X, W, dY = dev_inputs[3 * p: 3 * p + 3]
            fwd, dx, dw = cases[3 * p: 3 * p + 3]
            calls.append(Call(fwd, mode, X, W, torch.empty((fwd.M, fwd.N), device=device)))
            calls.append(Call(dx, mode, dY, W, torch.empty((dx.M, dx.N), device=device)))
            calls.append(Call(dw, mode, X, dY, torch.empty((dw.M, dw.N), device=device)))
    return calls


def run_call(h, c: Call, stream):
    h.run(c.A, c.B, c.C, mode=c.mode, transA=c.case.transA, transB=c.case.transB, stream=stream)


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"dgt_clocks_{os.getpid()}_{id(self)}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
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
        try:
            self.fh.close()
        except Exception:
            pass

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


def oracle_sample(calls_meta, budget_macs):
    """Time the oracle on the first rows of every GEMM; returns (flops, seconds, rows)."""
    import numpy as np

    import oracle
    cores = os.cpu_count() or 1
    flops, secs, desc = 0, 0.0, []
    per_call = budget_macs / max(len(calls_meta), 1)
    cache = {}
    for mode, case, (a_t, b_t) in calls_meta:
        key = (id(a_t), id(b_t))
        if key not in cache:
            cache[key] = (a_t.numpy(), b_t.numpy())
        a, b = cache[key]
        rows = int(max(cores, min(case.M, per_call // max(case.N * case.K, 1))))
        rows = min(rows, case.M)
        t0 = time.perf_counter()
        oracle.gemm(mode, a, b, transA=case.transA, transB=case.transB, rows=(0, rows))
        secs += time.perf_counter() - t0
        flops += 2 * rows * case.N * case.K
        desc.append(rows)
    return flops, secs, desc


def cpu_meta():
    """The (mode, case, host tensors) list of the GPT workload, host side only."""
    cases = si.gpt_cases()
    meta = []
    host = []
    for p, (name, kin, nout) in enumerate(si.GPT_PROJECTIONS):
        host.append(si.gpt_tensors(p, kin, nout))
    for mode in ("fp32", "tf32"):
        for p in range(len(si.GPT_PROJECTIONS)):
            X, W, dY = host[p]
            fwd, dx, dw = cases[3 * p: 3 * p + 3]
            meta += [(mode, fwd, (X, W)), (mode, dx, (dY, W)), (mode, dw, (X, dY))]
    return meta


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl != "reference" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def bench_reference(args, world, rank):
    """The CPU oracle as the reference arm, on a bounded sample per step."""
    if rank != 0:
        return
    meta = cpu_meta()
    total_flops = sum(2 * c.M * c.N * c.K for _, c, _ in meta)
    for _ in range(args.warmup):
        oracle_sample(meta[:2], 1e7)
    flops = secs = 0.0
    rows = None
    for _ in range(args.steps):
        f, s, rows = oracle_sample(meta, args.ref_macs)
        flops += f
        secs += s
    value = flops / secs / 1e12
    sample = (f"first rows of each of the 30 GEMMs ({min(rows)}..{max(rows)} rows, "
              f"{flops / args.steps / total_flops * 100:.3f}% of a step's FLOPs per step)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights)",
            "config": {"workload": "gpt_projections_fp32_tf32", "tokens": si.GPT_TOKENS, "d_model": 384,
                       "gemms_per_step": 30, "parallelism": f"replicas{world}",
                       "l2": "host memory (the oracle runs on the CPU cores)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def bench_ours(args, world, rank, local):
    import dense_gemm_transformer_gb300 as dg
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    dg.load(build_if_missing=True)
    h = dg.Gemm()
    if args.tile_n:
        h.set_option("tile_n", args.tile_n)
    stream = torch.cuda.Stream(dev)
    calls, host_inputs, dev_inputs = gpt_workload(dev)
    if args.only:
        import re
        calls = [c for c in calls if re.fullmatch(args.only, c.name)]
        if not calls:
            raise SystemExit(f"--only {args.only!r} matches no GEMM of the step")
    step_flops = sum(c.case.flops for c in calls)
    pk = peaks()
    fp32_peak = None
    if not args.no_fp32_peak:
        fp32_peak = measure_fp32_peak(dev)
        pk["fp32_alu_tflops_derived"] = pk["fp32_alu_tflops"]
        pk["fp32_alu_tflops"] = fp32_peak["tflops"]

    def step():
        for c in calls:
            run_call(h, c, stream)

    # Launch counts per call (deterministic plans).
    launches = 0
    with torch.cuda.stream(stream):
        for c in calls:
            run_call(h, c, stream)
            launches += h.plan()["kernels"]
    stream.synchronize()
    assert h.check_device(stream) == 0

    for _ in range(args.warmup):
        step()
    stream.synchronize()

    # Timed region: K whole steps, CUDA events around every call on the stream.
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in calls]
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        time.sleep(0.4)
        t_start.record(stream)
        for s in range(args.steps):
            for i, c in enumerate(calls):
                ev[s][i][0].record(stream)
                run_call(h, c, stream)
                ev[s][i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world, dev)
    assert h.check_device(stream) == 0
    per_call_ms = [statistics.mean(ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps))
                   for i in range(len(calls))]
    ms_per_step = total_ms / args.steps
    value = world * step_flops / (ms_per_step * 1e-3) / 1e12

    # Per-shape breakdown against each mode's roof.
    shapes = []
    for c, ms in zip(calls, per_call_ms):
        peak = pk["fp32_alu_tflops"] if c.mode == "fp32" else pk["tf32_tflops_sustained"]
        t_roof = max(c.case.flops / (peak * 1e12), c.bytes() / (pk["hbm_gbs"] * 1e9))
        bound = ("alu" if c.mode == "fp32" else "tensor") if c.case.flops / (peak * 1e12) >= c.bytes() / (
            pk["hbm_gbs"] * 1e9) else "hbm"
        shapes.append({"gemm": c.name, "M": c.case.M, "N": c.case.N, "K": c.case.K, "ms": round(ms, 4),
                       "tflops": round(c.case.flops / (ms * 1e-3) / 1e12, 2), "bound": bound,
                       "roofline_frac": round(t_roof / (ms * 1e-3), 3)})

    # Dominant kernel family = the mode with the larger share of the step.
    fam_ms = {m: sum(ms for c, ms in zip(calls, per_call_ms) if c.mode == m) for m in ("fp32", "tf32")
              if any(c.mode == m for c in calls)}
    dom = max(fam_ms, key=fam_ms.get)
    dom_flops = sum(c.case.flops for c in calls if c.mode == dom)
    n_launch = sum(1 for c in calls if c.mode == dom)
    achieved = dom_flops / (fam_ms[dom] * 1e-3) / 1e12
    if dom == "fp32":
        roof = {"bound": "alu", "kernel": "simt_gemm_kernel (FP32 FFMA)", "achieved": achieved,
                "peak": pk["fp32_alu_tflops"], "unit": "TFLOP/s",
                "peak_source": ("measured on this GPU in this run: " + fp32_peak["how"]) if fp32_peak else
                               "derived: 152 SMs x 128 FP32 lanes x 2 flop x 2070 MHz"}
    else:
        roof = {"bound": "tensor", "kernel": "tc_gemm_kernel (tcgen05 kind::tf32)", "achieved": achieved,
                "peak": pk["tf32_tflops_sustained"], "unit": "TFLOP/s",
                "peak_source": f"{pk['source']} bf16 sustained x 1.1/2.25 (nominal tf32/bf16)"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profiled_traffic(dom)
    roof["algorithmic_bytes_per_launch"] = sum(c.bytes() for c in calls if c.mode == dom) / max(n_launch, 1)
    roof["launches_per_step"] = n_launch
    roof["share_of_step"] = fam_ms[dom] / sum(per_call_ms)

    # End to end through the C ABI: pinned host inputs -> device, the 30 GEMMs,
    # every output -> pinned host, all inside the timed region.  Inputs and
    # outputs are double-buffered on the device so that step s+1's uploads
    # (one copy stream) run while step s computes, and each output goes down
    # on another copy stream as soon as its GEMM has finished.
    e2e = None
    if not args.no_e2e:
        pinned_in = [t.pin_memory() for t in host_inputs]
        h2d = sum(t.numel() * t.element_size() for t in pinned_in)
        dev_inputs2 = [torch.empty_like(t) for t in dev_inputs]
        bufs = [(dev_inputs, calls), (dev_inputs2, gpt_calls(dev_inputs2, dev))]
        if args.only:
            import re
            bufs[1] = (dev_inputs2, [c for c in bufs[1][1] if re.fullmatch(args.only, c.name)])
        pinned_out = [torch.empty(c.C.shape, dtype=c.C.dtype, pin_memory=True) for c in calls]
        d2h = sum(t.numel() * t.element_size() for t in pinned_out)
        # Several copy streams per direction, so that transfers can use more
        # than one copy engine at a time.
        nq = max(1, args.copy_streams)
        ups = [torch.cuda.Stream(dev) for _ in range(nq)]
        downs = [torch.cuda.Stream(dev) for _ in range(nq)]
        done = [torch.cuda.Event() for _ in calls]
        up_done = [[torch.cuda.Event(), torch.cuda.Event()] for _ in range(nq)]
        comp_done = [torch.cuda.Event(), torch.cuda.Event()]
        down_done = [[torch.cuda.Event(), torch.cuda.Event()] for _ in range(nq)]

        def e2e_step(s):
            b = s % 2
            ins, cls = bufs[b]
            for i, up in enumerate(ups):
                up.wait_event(comp_done[b])  # the GEMMs that last read these inputs are done
                with torch.cuda.stream(up):
                    for src, dst in list(zip(pinned_in, ins))[i::nq]:
                        dst.copy_(src, non_blocking=True)
                up_done[i][b].record(up)
                stream.wait_event(up_done[i][b])
            for i in range(nq):
                stream.wait_event(down_done[i][b])  # these outputs have been downloaded
            for j, (c, dst, ev) in enumerate(zip(cls, pinned_out, done)):
                run_call(h, c, stream)
                ev.record(stream)
                down = downs[j % nq]
                down.wait_event(ev)
                with torch.cuda.stream(down):
                    dst.copy_(c.C, non_blocking=True)
            comp_done[b].record(stream)
            for i, down in enumerate(downs):
                down_done[i][b].record(down)

        def run_steps(n):
            for q in ups + downs:
                q.wait_stream(stream)
            for s in range(n):
                e2e_step(s)
            for q in ups + downs:
                stream.wait_stream(q)

        run_steps(2)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(stream)
        run_steps(args.steps)
        e1.record(stream)
        stream.synchronize()
        e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
        e2e = {"value": world * step_flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms}

    configs = None
    if rank == 0 and not args.no_configs:
        configs = bench_configs(args, h, dev, pk)
        # the whole 6-layer projection step (75 GEMMs) in each mode, eager
        # and as one CUDA graph
        with ClockSampler(dev.index) as fclk:
            configs["full_step"] = [time_full_step(h, dev, m, 5, 3) for m in ("tf32", "bf16", "fp32")]
        configs["full_step_clocks"] = fclk.summary()
        # the fused attention forward (the GPT's attention and two longer
        # contexts), a shorter sample than --workload attention takes
        with ClockSampler(dev.index) as aclk:
            configs["attention"] = attention_shapes(h, dev, stream, pk, samples=3, sample_ms=10.0)
        configs["attention_clocks"] = aclk.summary()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, s, rows = oracle_sample(cpu_meta(), args.cpu_macs)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"first {min(rows)}..{max(rows)} rows of each of the 30 GEMMs "
                         f"({f / step_flops * 100:.3f}% of a step's FLOPs, {s:.1f} s)"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32+tf32",
                "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights)",
                "config": {"workload": "gpt_projections_fp32_tf32", "tokens": si.GPT_TOKENS, "d_model": 384,
                           "gemms_per_step": len(calls), "parallelism": f"replicas{world}",
                           "l2": "inputs larger than L2: a step touches %.2f GB; no tensor is re-read "
                                 "before >4x L2 of other traffic" % (sum(c.bytes() for c in calls) / 1e9)},
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches * args.steps,
                "clocks": clk.summary(), "shapes": shapes, "peaks": pk, "fp32_peak": fp32_peak,
                "configs": configs}
        print(json.dumps(line), flush=True)
    h.close()


def sweep_cases(workload):
    """(label, mode, case, alpha, beta, weight_std) of a per-shape sweep."""
    out = []
    if workload == "square":
        for n in si.SQUARE_SWEEP:
            for mode in ("fp32", "tf32", "bf16"):
                for alpha, beta in ((1.0, 0.0), (0.5, 1.0)):
                    out.append((f"{mode}.square{n}.a{alpha}b{beta}", mode, si.square_case(n), alpha, beta, 1.0))
    elif workload == "large":
        for M, N, K in si.LARGE_BF16:
            out.append((f"bf16.{M}x{N}x{K}", "bf16", si.GemmCase(f"{M}x{N}x{K}", False, False, M, N, K),
                        1.0, 0.0, 1.0))
    elif workload == "skinny":
        for tB in (False, True):
            for c in si.skinny_cases():
                case = si.GemmCase(c.name + (".T" if tB else ""), False, tB, c.M, c.N, c.K)
                out.append((f"bf16.{case.name}", "bf16", case, 1.0, 0.0, 0.02))
    elif workload == "large_fp8":
        # E4M3 operands, both K-major (B stored N x K), N(0, 1) codes
        for M, N, K in ((4096, 4096, 4096),) + si.LARGE_BF16:
            out.append((f"fp8.{M}x{N}x{K}.T", "fp8", si.GemmCase(f"{M}x{N}x{K}.T", False, True, M, N, K),
                        1.0, 0.0, 1.0))
    elif workload == "large_bs":
        # block-scaled operands with M > 16, both stored K-major (B N x K):
        # random finite codes and scales, as for the decode shapes below
        for mode in ("mxfp8_e4m3", "nvfp4"):
            for M, N, K in ((4096, 4096, 4096),) + si.LARGE_BF16:
                out.append((f"{mode}.{M}x{N}x{K}.T", mode, si.GemmCase(f"{M}x{N}x{K}.T", False, True, M, N, K),
                            1.0, 0.0, 1.0))
    elif workload in ("skinny_nvfp4", "skinny_mxfp8"):
        # block-scaled weights stored N x K (the form the kernels read): random
        # finite codes and scales (a quantiser would only change their values)
        mode = "nvfp4" if workload == "skinny_nvfp4" else "mxfp8_e4m3"
        for c in si.skinny_cases():
            case = si.GemmCase(c.name + ".T", False, True, c.M, c.N, c.K)
            out.append((f"{mode}.{case.name}", mode, case, 1.0, 0.0, 1.0))
    elif workload == "skinny_fp8":
        # E4M3 weights stored N x K (the form the FP8 mode takes), N(0, 1)
        # codes: a per-tensor scale would only change alpha
        for c in si.skinny_cases():
            case = si.GemmCase(c.name + ".T", False, True, c.M, c.N, c.K)
            out.append((f"fp8.{case.name}", "fp8", case, 1.0, 0.0, 1.0))
    return out


GATE = 0.70  # the configurations' roofline targets: tensor peak (large squares, 8192-class), HBM (decode)


def config_cases():
    """(config, gate, label, mode, case, alpha, beta, weight_std) of every
    configuration other than the GPT step, for the default benchmark line:
    0: FP32 256^3; 2: the square sweep, every mode, both alpha/beta pairs;
    3: the large BF16 shapes; 4: the decode shapes, weights K x N and N x K.
    The gates: the tensor peak for TF32/BF16 squares of 4096 and the large
    BF16 shapes, HBM bandwidth for the decode shapes (graph timing)."""
    out = [(0, None, "fp32.square256", "fp32", si.square_case(256), 1.0, 0.0, 1.0)]
    for label, mode, c, alpha, beta, wstd in sweep_cases("square"):
        gate = "tensor" if mode != "fp32" and c.M >= 4096 else None
        out.append((2, gate, label, mode, c, alpha, beta, wstd))
    for label, mode, c, alpha, beta, wstd in sweep_cases("large"):
        out.append((3, "tensor", label, mode, c, alpha, beta, wstd))
    for label, mode, c, alpha, beta, wstd in sweep_cases("skinny"):
        out.append((4, "hbm", label, mode, c, alpha, beta, wstd))
    return out


def bench_configs(args, h, dev, pk, samples=3, sample_ms=10.0):
    """Every other configuration's shapes, timed in this process as the
    per-shape sweeps time them (operands rotated over > 3x L2, R launches
    per sample for >= sample_ms, back to back, as one CUDA graph, and the
    identity null), with fewer, shorter samples so that the default run
    stays within minutes; gated shapes say whether they meet 0.70."""
    stream = torch.cuda.Stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    meta = config_cases()
    shapes = []
    h.set_option("tile_n", 0)
    with ClockSampler(dev.index) as clk:
        _sweep_shapes(args, h, stream, pk, l2, dev, shapes, cases=[m[2:] for m in meta], samples=samples,
                      sample_ms=sample_ms)
    by_label = {m[2]: m for m in meta}
    met = total = 0
    for x in shapes:
        cfg, gate = by_label[x["gemm"]][0], by_label[x["gemm"]][1]
        x["config"] = cfg
        x["gate"] = None if gate is None else f"{gate} >= {GATE}"
        if gate is not None:
            x["gate_met"] = bool(x["roofline_frac"] >= GATE and x["bound"] in (("hbm",) if gate == "hbm"
                                                                               else ("tensor",)))
            met += x["gate_met"]
            total += 1
    return {"shapes": shapes, "gates_met": met, "gates": total, "clocks": clk.summary(),
            "timing": f"one process, median of {samples} samples of >= {sample_ms:g} ms per shape; decode shapes "
                      "gated on the CUDA-graph timing; operands rotated over > 3x L2",
            "roofline": "roofline_frac against the burst peaks (tensor: MEASURED_PEAKS bf16 x the nominal "
                        "tf32/bf16 ratio for TF32), HBM: MEASURED_PEAKS copy bandwidth; FP32 against the "
                        "measured FMA roof"}


def _elem_bytes(mode):
    return {"bf16": 2, "fp8": 1, "mxfp8_e4m3": 1, "nvfp4": 0.5}.get(mode, 4)


def _scale_bytes(mode, rows, K):
    """Bytes of the block scales of a rows x K block-scaled operand."""
    if mode not in ("nvfp4", "mxfp8_e4m3"):
        return 0
    bs = 16 if mode == "nvfp4" else 32
    return rows * -(-K // bs)


def _block_scaled_set(mode, c, dev, g):
    """Codes and tiled scales of a block-scaled case (A M x K, B N x K)."""
    import dense_gemm_transformer_gb300 as dg
    per = 2 if mode == "nvfp4" else 1
    bs = 16 if mode == "nvfp4" else 32
    nb = -(-c.K // bs)

    def codes(rows):
        if mode == "nvfp4":
            return torch.randint(0, 256, (rows, c.K // per), generator=g, dtype=torch.uint8).to(dev)
        mag = torch.randint(0x20, 0x50, (rows, c.K), generator=g, dtype=torch.uint8)
        return (mag | (torch.randint(0, 2, (rows, c.K), generator=g, dtype=torch.uint8) << 7)).to(dev)

    def scales(rows):
        lo, hi = (120, 131) if mode != "nvfp4" else (0x28, 0x48)
        return dg.tile_block_scales(torch.randint(lo, hi, (rows, nb), generator=g, dtype=torch.uint8).to(dev))

    return codes(c.M), scales(c.M), codes(c.N), scales(c.N)


def _operand_dtype(mode):
    return {"bf16": torch.bfloat16, "fp8": torch.float8_e4m3fn}.get(mode, torch.float32)


SAMPLES = 5          # timed samples per shape (median and spread)
SAMPLE_MS = 20.0     # each sample covers at least this much device time
MAX_REPS = 4000      # launches per sample at most
QUEUE_CALLS = 600    # launches held behind one spin kernel at a time


def _timed_back_to_back(fn, reps, stream, chunk):
    """Device time per call of fn(0..reps-1), enqueued in chunks that each sit
    behind a spin kernel while the host enqueues them, so the timed calls run
    back to back with no host gaps; the chunk's events bracket only the calls."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total, done = 0.0, 0
    while done < reps:
        n = min(chunk, reps - done)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(max(4e6, n * 1e5)))  # ~50 us of spin per queued call
            e0.record(stream)
            for r in range(done, done + n):
                fn(r)
            e1.record(stream)
        stream.synchronize()
        total += e0.elapsed_time(e1)
        done += n
    return total / reps


def _stats(xs):
    xs = sorted(xs)
    return {"median": xs[len(xs) // 2], "min": xs[0], "max": xs[-1]}


def bench_sweep(args):
    """Per-shape TFLOP/s and roofline fractions for the other configurations.

    Each shape, after warm-up, with the operands rotated over enough copies
    that one rotation's working set exceeds 3x the L2 (every launch reads its
    weights from HBM), and R launches per sample, R chosen so that a sample
    covers >= 20 ms:
      * "ms": calls back to back on the device (held behind a spin kernel
        while the host enqueues them), median of 5 samples, with the spread;
      * "ms_graph": the same R calls captured once in a CUDA graph, median of
        5 replays (small-M shapes are gated on this one);
      * "ms_stream": the calls as the host issues them (includes the host's
        per-call cost whenever it exceeds the kernel time);
      * "null_ms": gemm_launch_null -- an empty kernel with the launch
        configuration of the call's main kernel -- timed like "ms".
    """
    import dense_gemm_transformer_gb300 as dg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dg.load(build_if_missing=True)
    h = dg.Gemm()
    if args.tile_n:
        h.set_option("tile_n", args.tile_n)
    if args.pair is not None:
        h.set_option("pair", args.pair)
    if args.split_k:
        h.set_option("split_k", args.split_k)
    stream = torch.cuda.Stream(dev)
    pk = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    shapes = []
    with ClockSampler(dev.index) as clk:
        _sweep_shapes(args, h, stream, pk, l2, dev, shapes)
    h.close()
    return shapes, clk.summary()


def _sweep_shapes(args, h, stream, pk, l2, dev, shapes, cases=None, samples=SAMPLES, sample_ms=SAMPLE_MS):
    for label, mode, c, alpha, beta, wstd in (cases if cases is not None else sweep_cases(args.workload)):
        if args.only:
            import re
            if not re.fullmatch(args.only, label):
                continue
        es = _elem_bytes(mode)
        sf_bytes = _scale_bytes(mode, c.M, c.K) + _scale_bytes(mode, c.N, c.K)
        per_set = int(es * (c.M * c.K + c.K * c.N)) + sf_bytes + 4 * c.M * c.N
        copies = max(1, min(32, -(-3 * l2 // per_set)))
        g = torch.Generator(device="cpu")
        g.manual_seed(si.BASE_SEED)
        sets = []
        if sf_bytes:
            A0, SA0, B0, SB0 = _block_scaled_set(mode, c, dev, g)
            for i in range(copies):
                cl = (lambda t: t) if i == 0 else (lambda t: t.clone())
                sets.append((cl(A0), cl(SA0), cl(B0), cl(SB0), torch.randn((c.M, c.N), generator=g).to(dev)))

            def call(r):
                A, SA, B, SB, C = sets[r % copies]
                h.run_block_scaled(A, SA, B, SB, C, mode=mode, alpha=alpha, beta=beta, stream=stream)
        else:
            dt = _operand_dtype(mode)
            A0 = torch.randn(c.a_shape, generator=g).to(dt).to(dev)
            B0 = (torch.randn(c.b_shape, generator=g) * wstd).to(dt).to(dev)
            for i in range(copies):
                A = A0 if i == 0 else A0.clone()
                B = B0 if i == 0 else B0.clone()
                C = torch.randn((c.M, c.N), generator=g).to(dev)
                sets.append((A, B, C))

            def call(r):
                A, B, C = sets[r % copies]
                h.run(A, B, C, mode=mode, transA=c.transA, transB=c.transB, alpha=alpha, beta=beta, stream=stream)

        with torch.cuda.stream(stream):
            for r in range(copies):
                call(r)
        stream.synchronize()
        plan = h.plan()
        chunk = max(copies, QUEUE_CALLS // max(plan["kernels"], 1))
        # R: enough launches that one sample covers SAMPLE_MS of device time.
        t_est = _timed_back_to_back(call, max(2 * copies, 10), stream, chunk)
        reps = int(min(MAX_REPS, max(10, math.ceil(sample_ms / max(t_est, 1e-4)))))
        reps = max(reps, copies)
        dev_ms = [_timed_back_to_back(call, reps, stream, chunk) for _ in range(samples)]
        # As the host issues them.
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for r in range(reps):
                call(r)
            e1.record(stream)
        stream.synchronize()
        stream_ms = e0.elapsed_time(e1) / reps
        # One CUDA graph of the R calls, replayed.
        graph_ms, graph_err = None, None
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for r in range(reps):
                    call(r)
            graph.replay()
            stream.synchronize()
            gm = []
            for _ in range(samples):
                with torch.cuda.stream(stream):
                    e0.record(stream)
                    graph.replay()
                    e1.record(stream)
                stream.synchronize()
                gm.append(e0.elapsed_time(e1) / reps)
            graph_ms = _stats(gm)
            del graph
        except Exception as exc:  # reported, not fatal: the stream timings stand
            graph_err = f"{type(exc).__name__}: {exc}"[:200]
            stream.synchronize()
        assert h.check_device(stream) == 0
        # The identity null of this configuration.
        call(0)
        null_ms = _stats([_timed_back_to_back(lambda r: h.launch_null(stream), reps, stream, QUEUE_CALLS)
                          for _ in range(samples)])
        stream.synchronize()
        byts = int(es * (c.M * c.K + c.K * c.N)) + sf_bytes + 4 * c.M * c.N * (2 if beta != 0 else 1)
        # block-scaled: the dense rate of the element type (FP4: FP8's x the nominal ratio)
        peak = {"fp32": pk["fp32_alu_tflops"], "tf32": pk["tf32_tflops"], "bf16": pk["bf16_tflops"],
                "fp8": pk["fp8_tflops"], "mxfp8_e4m3": pk["fp8_tflops"],
                "nvfp4": FP4_OVER_FP8 * pk["fp8_tflops"]}[mode]
        peak_s = {"fp32": pk["fp32_alu_tflops"], "tf32": pk["tf32_tflops_sustained"],
                  "bf16": pk["bf16_tflops_sustained"], "fp8": pk["fp8_tflops_sustained"],
                  "mxfp8_e4m3": pk["fp8_tflops_sustained"],
                  "nvfp4": FP4_OVER_FP8 * pk["fp8_tflops_sustained"]}[mode]
        t_c, t_m = c.flops / (peak * 1e12), byts / (pk["hbm_gbs"] * 1e9)
        t_cs = c.flops / (peak_s * 1e12)
        st = _stats(dev_ms)
        gate_graph = plan["family"] == "skinny" or (c.M <= 16 and graph_ms is not None)
        t = graph_ms["median"] if (gate_graph and graph_ms is not None) else st["median"]
        shapes.append({"gemm": label, "M": c.M, "N": c.N, "K": c.K, "ms": round(t, 5),
                       "timing": "graph" if (gate_graph and graph_ms is not None) else "back_to_back",
                       "ms_back_to_back": {k: round(v, 5) for k, v in st.items()},
                       "ms_graph": None if graph_ms is None else {k: round(v, 5) for k, v in graph_ms.items()},
                       "graph_error": graph_err,
                       "ms_stream": round(stream_ms, 5),
                       "null_ms": {k: round(v, 5) for k, v in null_ms.items()},
                       "samples": samples, "reps": reps,
                       "tflops": round(c.flops / (t * 1e-3) / 1e12, 2),
                       "gbs": round(byts / (t * 1e-3) / 1e9, 1), "bound": "hbm" if t_m > t_c else
                       ("alu" if mode == "fp32" else "tensor"), "roofline_frac": round(max(t_c, t_m) / (t * 1e-3), 3),
                       "roofline_frac_sustained": round(max(t_cs, t_m) / (t * 1e-3), 3),
                       "plan": plan, "copies": copies})
        del sets, A0, B0
        torch.cuda.empty_cache()


def sweep_line(args, shapes, processes, clocks):
    pk = peaks()
    total_flops = sum(2 * x["M"] * x["N"] * x["K"] for x in shapes)
    total_s = sum(x["ms"] for x in shapes) * 1e-3
    return {"metric": METRIC, "value": total_flops / total_s / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
            "higher_is_better": True, "dtype": "see shapes", "data": "synthetic",
            "config": {"workload": args.workload, "l2": "operands rotated over copies > 3x L2",
                       "samples": f"median of {SAMPLES} samples of >= {SAMPLE_MS:g} ms per process, "
                                  f"median over {processes} process(es)"},
            "processes": processes, "clocks": clocks, "shapes": shapes, "peaks": pk,
            "roofline_note": "roofline_frac against the burst tensor peak (a kernel timed alone); "
                             "roofline_frac_sustained against the sustained one (samples of >= 20 ms "
                             "back to back run under the power cap)"}


def bench_sweep_processes(args):
    """The sweep in `args.processes` separate processes; per shape, the median
    over the processes of their medians, with the spread across processes."""
    if args.processes <= 1:
        shapes, clocks = bench_sweep(args)
        print(json.dumps(sweep_line(args, shapes, 1, clocks)), flush=True)
        return
    runs, clocks = [], []
    for _ in range(args.processes):
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", args.workload, "--processes", "1"]
        if args.only:
            cmd += ["--only", args.only]
        if args.tile_n:
            cmd += ["--tile-n", str(args.tile_n)]
        if args.pair is not None:
            cmd += ["--pair", str(args.pair)]
        if args.split_k:
            cmd += ["--split-k", str(args.split_k)]
        out = subprocess.run(cmd, capture_output=True, text=True, check=True).stdout
        line = json.loads(out.strip().splitlines()[-1])
        runs.append(line["shapes"])
        clocks.append(line.get("clocks"))
    print(json.dumps(sweep_line(args, merge_process_runs(runs), args.processes, clocks)), flush=True)


def merge_process_runs(runs):
    """Per shape (the same order in every run): the record of the process
    whose time is the median across processes, with every process's time in
    "ms_processes" (the spread)."""
    shapes = []
    for per in zip(*runs):
        labels = {x["gemm"] for x in per}
        if len(labels) != 1:
            raise ValueError(f"processes timed different shapes: {sorted(labels)}")
        ms = sorted(x["ms"] for x in per)
        med = ms[len(ms) // 2]
        rec = dict(next(x for x in per if x["ms"] == med))
        rec["ms_processes"] = ms
        shapes.append(rec)
    return shapes


def bench_epilogue(args):
    """The fused epilogue on the GPT products that carry one: the MLP-up
    forward with bias + GELU (C = GELU(X W + b)) and the MLP-down dX with
    GELU' (dH = (dY W^T) * GELU'(Z), Z the kept pre-activation), in FP32 and
    TF32.  Each is timed as the plain GEMM and as the fused call (median of 5
    samples of >= 20 ms, operands rotated over > 3x L2); "pass_ms" is what a
    separate elementwise pass would take at the measured HBM bandwidth
    (read and write C, and read Z for GELU'), the least the unfused form
    adds."""
    import dense_gemm_transformer_gb300 as dg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dg.load(build_if_missing=True)
    h = dg.Gemm()
    stream = torch.cuda.Stream(dev)
    pk = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    T, D, F = si.GPT_TOKENS, 384, 1536
    shapes = []
    with ClockSampler(dev.index) as clk:
        for mode in ("fp32", "tf32"):
            for name, M, N, K, tB, act in (("mlp_up.fwd+bias+gelu", T, F, D, False, "gelu"),
                                           ("mlp_down.dX*dgelu", T, F, D, True, "dgelu")):
                if args.only and not re.fullmatch(args.only, f"{mode}.{name}"):
                    continue
                g = torch.Generator(device="cpu")
                g.manual_seed(si.BASE_SEED)
                per_set = 4 * (M * K + K * N + M * N * (2 if act == "dgelu" else 1))
                copies = max(1, min(8, -(-3 * l2 // per_set)))
                sets = []
                for _ in range(copies):
                    A = torch.randn((M, K), generator=g).to(dev)
                    B = (torch.randn((N, K) if tB else (K, N), generator=g) * 0.02).to(dev)
                    C = torch.empty((M, N), device=dev)
                    Z = torch.randn((M, N), generator=g).to(dev) if act == "dgelu" else None
                    sets.append((A, B, C, Z))
                bias = (torch.randn((N,), generator=g) * 0.02).to(dev) if act == "gelu" else None

                def plain(r):
                    A, B, C, _ = sets[r % copies]
                    h.run(A, B, C, mode=mode, transB=tB, stream=stream)

                def fused(r):
                    A, B, C, Z = sets[r % copies]
                    h.run(A, B, C, mode=mode, transB=tB, stream=stream, act=act, bias=bias, aux=Z)

                res = {}
                for label, fn in (("plain", plain), ("fused", fused)):
                    with torch.cuda.stream(stream):
                        for r in range(copies):
                            fn(r)
                    stream.synchronize()
                    t_est = _timed_back_to_back(fn, max(2 * copies, 10), stream, 300)
                    reps = int(min(MAX_REPS, max(10, math.ceil(SAMPLE_MS / max(t_est, 1e-4)))))
                    res[label] = _stats([_timed_back_to_back(fn, reps, stream, 300) for _ in range(SAMPLES)])
                assert h.check_device(stream) == 0
                flops = 2 * M * N * K
                pass_bytes = 4 * M * N * (3 if act == "dgelu" else 2)
                pass_ms = pass_bytes / (pk["hbm_gbs"] * 1e9) * 1e3
                byts = 4 * (M * K + K * N + M * N) + (4 * M * N if act == "dgelu" else 4 * N)
                peak = pk["fp32_alu_tflops"] if mode == "fp32" else pk["tf32_tflops_sustained"]
                t_roof = max(flops / (peak * 1e12), byts / (pk["hbm_gbs"] * 1e9))
                fm = res["fused"]["median"]
                shapes.append({"gemm": f"{mode}.{name}", "M": M, "N": N, "K": K,
                               "ms_plain": round(res["plain"]["median"], 5), "ms_fused": round(fm, 5),
                               "fused_overhead_ms": round(fm - res["plain"]["median"], 5),
                               "pass_ms": round(pass_ms, 5),
                               "unfused_floor_ms": round(res["plain"]["median"] + pass_ms, 5),
                               "tflops_fused": round(flops / (fm * 1e-3) / 1e12, 2),
                               "roofline_frac_fused": round(t_roof / (fm * 1e-3), 3),
                               "plan": h.plan()})
                del sets
                torch.cuda.empty_cache()
    h.close()
    if not shapes:
        raise SystemExit(f"--only {args.only!r} matches no epilogue product")
    total_flops = sum(2 * x["M"] * x["N"] * x["K"] for x in shapes)
    line = {"metric": METRIC, "value": total_flops / (sum(x["ms_fused"] for x in shapes) * 1e-3) / 1e12,
            "unit": "TFLOP/s", "n_gpus": 1, "higher_is_better": True, "dtype": "f32+tf32", "data": "synthetic",
            "config": {"workload": "epilogue", "l2": "operands rotated over copies > 3x L2",
                       "samples": f"median of {SAMPLES} samples of >= {SAMPLE_MS:g} ms"},
            "clocks": clk.summary(), "shapes": shapes, "peaks": pk}
    print(json.dumps(line), flush=True)


def attention_flops_bytes(P, T, D, causal):
    """Algorithmic work of one attention forward: 4 D flops per (query, visible
    key) pair (the score dot product and the P V product); bytes: Q, K and V
    read once (bf16) and O written once (fp32)."""
    pairs = T * (T + 1) // 2 if causal else T * T
    return 4 * D * pairs * P, P * T * D * (3 * 2 + 4)


def attention_shapes(h, dev, stream, pk, samples=SAMPLES, sample_ms=SAMPLE_MS, only=None):
    """The fused attention forward (gemm_attention_forward) on the GPT's
    attention (64 sequences x 6 heads of 64, context 256) and on the same
    16384 tokens at contexts 1024 and 2048, causal: median of `samples`
    samples of >= sample_ms of calls back to back, inputs rotated over copies
    > 3x L2; the roofline is the larger of the tensor time (bf16 burst peak)
    and the HBM time of the algorithmic bytes.  only: a regex on the
    workload names (gpt_ctx256, ctx1024, ctx2048), or None for all."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    D = si.ATTN_HEAD_DIM
    shapes = []
    for idx, (name, P, T) in enumerate(si.ATTN_WORKLOADS):
        if only and not re.search(only, name):
            continue
        flops, byts = attention_flops_bytes(P, T, D, True)
        copies = max(1, min(8, -(-3 * l2 // byts)))
        Q, K, V = (t.to(dev) for t in si.attention_qkv(P, T, shape=idx))
        sets = [(Q, K, V, torch.empty(Q.shape, dtype=torch.float32, device=dev))]
        for _ in range(copies - 1):
            sets.append((Q.clone(), K.clone(), V.clone(), torch.empty(Q.shape, dtype=torch.float32, device=dev)))

        def call(r):
            q, k, v, o = sets[r % copies]
            h.attention(q, k, v, o, causal=True, stream=stream)

        with torch.cuda.stream(stream):
            for r in range(copies):
                call(r)
        stream.synchronize()
        t_est = _timed_back_to_back(call, max(2 * copies, 10), stream, 300)
        reps = int(min(MAX_REPS, max(10, math.ceil(sample_ms / max(t_est, 1e-4)))))
        st = _stats([_timed_back_to_back(call, reps, stream, 300) for _ in range(samples)])
        assert h.check_device(stream) == 0
        ms = st["median"]
        t_tensor = flops / (pk["bf16_tflops"] * 1e12)
        t_hbm = byts / (pk["hbm_gbs"] * 1e9)
        shapes.append({"attention": name, "problems": P, "T": T, "Dh": D, "causal": True,
                       "ms": round(ms, 5), "ms_min": round(st["min"], 5), "ms_max": round(st["max"], 5),
                       "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
                       "gbs": round(byts / (ms * 1e-3) / 1e9, 1),
                       "bound": "tensor" if t_tensor >= t_hbm else "hbm",
                       "roofline_frac": round(max(t_tensor, t_hbm) / (ms * 1e-3), 3),
                       "scores_bytes_not_written": 4 * P * T * T, "plan": h.plan()})
        del sets, Q, K, V
        torch.cuda.empty_cache()
    return shapes


def bench_attention(args):
    """The fused attention forward on its three workloads (attention_shapes),
    median of 5 samples of >= 20 ms each."""
    import dense_gemm_transformer_gb300 as dg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dg.load(build_if_missing=True)
    h = dg.Gemm()
    stream = torch.cuda.Stream(dev)
    pk = peaks()
    D = si.ATTN_HEAD_DIM
    with ClockSampler(dev.index) as clk:
        shapes = attention_shapes(h, dev, stream, pk, only=args.only)
    h.close()
    total_flops = sum(attention_flops_bytes(x["problems"], x["T"], D, True)[0] for x in shapes)
    line = {"metric": "fused attention forward TFLOP/s and fraction of the roofline, 1 GPU",
            "value": total_flops / (sum(x["ms"] for x in shapes) * 1e-3) / 1e12,
            "unit": "TFLOP/s", "n_gpus": 1, "higher_is_better": True, "dtype": "bf16 in, fp32 accumulate and out",
            "data": "synthetic",
            "config": {"workload": "attention", "l2": "inputs rotated over copies > 3x L2",
                       "samples": f"median of {SAMPLES} samples of >= {SAMPLE_MS:g} ms"},
            "clocks": clk.summary(), "shapes": shapes, "peaks": pk}
    print(json.dumps(line), flush=True)


def time_full_step(h, dev, mode, steps, warmup):
    """The full projection step of the GPT (six layers of QKV, attention-out,
    MLP-up and MLP-down, each forward, dX and dW, plus the LM head: 75 GEMMs,
    1046 GFLOP), timed as the host issues it and as one CUDA graph of the
    whole step replayed.  Each layer has its own weights and activations
    (seeded, drawn on the device); one mode for the whole step."""
    stream = torch.cuda.Stream(dev)
    dt = torch.bfloat16 if mode == "bf16" else torch.float32
    T, layers = si.GPT_TOKENS, 6
    g = torch.Generator(device=dev)
    g.manual_seed(si.BASE_SEED + 4000)
    calls = []
    shapes = []
    projs = [(name, kin, nout) for name, kin, nout in si.GPT_PROJECTIONS if name != "lm_head"]
    head = [(name, kin, nout) for name, kin, nout in si.GPT_PROJECTIONS if name == "lm_head"]
    for layer in range(layers + 1):
        for name, kin, nout in (projs if layer < layers else head):
            X = torch.randn((T, kin), generator=g, device=dev).to(dt)
            W = (torch.randn((kin, nout), generator=g, device=dev) * 0.02).to(dt)
            dY = torch.randn((T, nout), generator=g, device=dev).to(dt)
            for A, B, tA, tB, M, N, K in ((X, W, False, False, T, nout, kin), (dY, W, False, True, T, kin, nout),
                                          (X, dY, True, False, kin, nout, T)):
                calls.append((A, B, torch.empty((M, N), device=dev), tA, tB))
                shapes.append((M, N, K))
    flops = sum(2 * M * N * K for M, N, K in shapes)

    def step():
        for A, B, C, tA, tB in calls:
            h.run(A, B, C, mode=mode, transA=tA, transB=tB, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 1)):
            step()
    stream.synchronize()
    launches = 0
    with torch.cuda.stream(stream):
        for A, B, C, tA, tB in calls:
            h.run(A, B, C, mode=mode, transA=tA, transB=tB, stream=stream)
            launches += h.plan()["kernels"]
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    stream.synchronize()
    eager_ms = e0.elapsed_time(e1) / steps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    graph.replay()
    stream.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    graph_ms = e0.elapsed_time(e1) / steps
    assert h.check_device(stream) == 0
    del graph, calls
    torch.cuda.empty_cache()
    return {"mode": mode, "gemms": len(shapes), "gflop": round(flops / 1e9, 1), "eager_ms": eager_ms,
            "graph_ms": graph_ms, "eager_tflops": flops / (eager_ms * 1e-3) / 1e12,
            "graph_tflops": flops / (graph_ms * 1e-3) / 1e12, "launches_per_step": launches}


def bench_gpt_full(args):
    """The full projection step in one mode (--mode), eager and as one graph."""
    import dense_gemm_transformer_gb300 as dg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    dg.load(build_if_missing=True)
    h = dg.Gemm()
    mode = args.mode
    with ClockSampler(dev.index) as clk:
        r = time_full_step(h, dev, mode, args.steps, args.warmup)
    h.close()
    line = {"metric": METRIC, "value": r["graph_tflops"], "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["graph_ms"], "higher_is_better": True,
            "dtype": {"fp32": "f32", "tf32": "tf32", "bf16": "bf16"}[mode], "data": "synthetic (seeded, drawn on the device)",
            "config": {"workload": f"gpt_full_step_{mode}", "layers": 6, "tokens": si.GPT_TOKENS, "d_model": 384,
                       "gemms_per_step": r["gemms"], "gflop_per_step": r["gflop"],
                       "timing": "one CUDA graph of the step, replayed; eager = as the host issues it"},
            "eager": {"value": r["eager_tflops"], "ms_per_step": r["eager_ms"]},
            "gpu_launches_per_step": r["launches_per_step"], "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--copy-streams", type=int, default=2, help="copy streams per direction in the end-to-end step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-shape timing of the other configurations in the default line")
    ap.add_argument("--no-fp32-peak", action="store_true",
                    help="take the derived FP32 roof instead of measuring it with the FMA kernel")
    ap.add_argument("--cpu-macs", type=float, default=4.5e10,
                    help="oracle multiply-adds in the CPU baseline (about 10 s on 16 host cores)")
    ap.add_argument("--ref-macs", type=float, default=3e8, help="oracle multiply-adds per reference step")
    ap.add_argument("--tile-n", type=int, default=0, help="sweeps: force the tensor-core tile width (128/256)")
    ap.add_argument("--only", default=None,
                    help="regex: time only the matching GEMMs of the step, sweep shapes, epilogue products or "
                         "attention workloads (profiling)")
    ap.add_argument("--pair", type=int, default=None,
                    help="sweeps: CTA pairs issuing one 256-row MMA (0 wherever allowed, 1 never)")
    ap.add_argument("--split-k", type=int, default=0, help="sweeps: force this many K slices (0: planner)")
    ap.add_argument("--workload", default="gpt", choices=["gpt", "square", "large", "large_fp8", "large_bs", "skinny",
                                                          "skinny_fp8",
                                                          "skinny_nvfp4", "skinny_mxfp8", "epilogue", "gpt_full",
                                                          "attention"],
                    help="gpt: the timed step; the others print a per-shape sweep")
    ap.add_argument("--mode", default="tf32", choices=["fp32", "tf32", "bf16"],
                    help="gpt_full: the mode of the whole step")
    ap.add_argument("--processes", type=int, default=3,
                    help="sweeps: separate processes to run the sweep in (median and spread across them)")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        bench_reference(args, world, rank)
    elif args.workload == "epilogue":
        bench_epilogue(args)
    elif args.workload == "attention":
        bench_attention(args)
    elif args.workload == "gpt_full":
        bench_gpt_full(args)
    elif args.workload != "gpt":
        bench_sweep_processes(args)
    else:
        bench_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
