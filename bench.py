#!/usr/bin/env python
"""Forward+backward benchmark of the routed MoE SwiGLU expert FFN with rank-128
side-LoRA at the production shape of "feat(mega): add fused shared side-LoRA
kernels" (DeepGEMM PR #9, Matched production-shape performance): 65,536 tokens,
H=4096, I=2048, E=256, top-6, rank 128, s=1, BF16 with FP32 accumulation, on one
GB300 (the pages measured 65,536 tokens per rank on 4 GPUs with expert
parallelism; this path has no expert parallelism).

One step = routing plan + forward + backward over one batch.  Inputs are seeded
synthetic tensors of the pages' shapes and distributions (synth.make_inputs),
resident in HBM; the working set (12.9 GB of frozen weights alone) is far larger
than the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  `value` is algorithmic TFLOP/s of the whole job (N GPUs,
max-over-ranks time); `e2e` repeats the measurement through the public Python
API with the inputs copied from pinned host memory and every result read back,
inside the timed region.  `--impl reference` times the CPU oracle (the method
written plainly in C) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from synth import Shape, make_inputs, make_router_inputs, shape  # noqa: E402

METRIC = "fwd+bwd ms & TFLOP/s (% BF16 peak), 64K tok H4096 I2048 E256 top6 r128"
ADAPTER_GRADS = ("dA1", "dA3", "dB1", "dB3", "dA2", "dB2")
WEIGHTS = ("W1", "W3", "W2", "A1", "A3", "B1", "B3", "A2", "B2")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sus": d.get("bf16_tflops_sustained",
                                                                                  d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sus": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ algorithmic work
def step_flops(T, R, H, I, r):
    """Forward + backward FLOPs over live routes R (no padding, no per-route
    re-expansion of the shared factors): 12RHI + 18THr + 18RIr."""
    return 12.0 * R * H * I + 18.0 * T * H * r + 18.0 * R * I * r


def kernel_work(T, R, H, I, r, k, E=256):
    """Per-launch algorithmic FLOPs (tensor kernels) or bytes (HBM kernels)."""
    E_I_H = float(E) * I * H
    fl = {
        "shrink_x_A13": 2.0 * T * H * 2 * r,
        "w13_lora_swiglu": 4.0 * R * H * I + 4.0 * R * I * r,
        "w13_native": 4.0 * R * H * I + 4.0 * R * I * r,
        "w2_a2": 2.0 * R * I * H + 2.0 * R * I * r,
        "w2_native": 2.0 * R * I * H + 2.0 * R * I * r,
        "b2_expand": 2.0 * T * r * H,
        "dy_b2": 2.0 * T * H * r,
        "dB2": 2.0 * T * H * r,
        "w2_dgrad_swiglu_bwd": 2.0 * R * H * I + 2.0 * R * r * I,
        "dA2": 2.0 * R * r * I,
        "w13_dgrad_b13": 4.0 * R * I * H + 4.0 * R * I * r,
        "dB13": 4.0 * R * I * r,
        "a13_expand": 4.0 * T * r * H,
        "dA13": 4.0 * T * r * H,
    }
    by = {
        "gather_fwd": 2.0 * (T * H + R * H + 2 * R * 2 * r),
        "z2_combine": 2.0 * (R * r + T * r),
        "gather_bwd": 2.0 * (T * H + R * H + 3 * R * r),
        "dw_reduce": 4.0 * (R * (I // 128) + T * k),
        "dw_native": 2.0 * (R * H + R * H + R * r) + 4.0 * T * k,
        "dy13_combine": 4.0 * R * 2 * r + 2.0 * T * 2 * r,
        "dequant_mxfp4": (2.0 + 0.5 + 1.0 / 32) * E_I_H,
        "combine_y": 2.0 * (R * H + 2 * T * H),
        "combine_dx": 2.0 * (R * H + 2 * T * H),
        "plan_count": 4.0 * T * k, "plan_scan": 0.0, "plan_scatter": 4.0 * T * k * 3, "plan_finish": 0.0, "plan_wide": 0.0,
    }
    return fl, by


def dominant_kernel(fl, native):
    """The roofline's kernel: the largest algorithmic FLOPs per launch among the kernels
    the configuration launches (W13 and the W13 dgrad tie; the forward's W13 comes
    first).  The native FP4 forward launches w13_native / w2_native in place of
    w13_lora_swiglu / w2_a2."""
    if native:
        names = [n for n in fl if n not in NATIVE_TWINS.values()]
    else:
        names = [n for n in fl if n not in NATIVE_TWINS]
    return max(names, key=lambda n: fl[n])


# the native FP4 forward's kernels and the ones they replace (the same work)
NATIVE_TWINS = {"w13_native": "w13_lora_swiglu", "w2_native": "w2_a2"}


# The committed DRAM-traffic counters (profiles/traffic.json) are keyed, per kernel,
# to the code that defines it: the GEMM engine and its helpers (shared by every
# problem), the kernel's own problem type in gemm_problems.cuh, and the host block
# that builds and launches it.  A change to another problem type leaves the record
# valid; comments and blank lines do not count.
ENGINE_SOURCES = ("sm100_ptx.cuh", "common.cuh", "gemm_engine.cuh", "gemm_pair.cuh")
PROBLEM_OF = {"shrink_x_A13": ("ProbShrink", "K_SHRINK"), "w13_lora_swiglu": ("ProbW13T", "K_W13"),
              "w2_a2": ("ProbW2T", "K_W2"), "b2_expand": ("ProbB2Expand", "K_B2_EXPAND"),
              "dy_b2": ("ProbDyB2", "K_DYB2"), "dB2": ("ProbDB2", "K_DB2"),
              "w2_dgrad_swiglu_bwd": ("ProbW2DgradT", "K_W2_DGRAD"), "dA2": ("ProbDA2", "K_DA2"),
              "w13_dgrad_b13": ("ProbW13DgradT", "K_W13_DGRAD"), "dB13": ("ProbDB13", "K_DB13"),
              "a13_expand": ("ProbA13Expand", "K_A13_EXPAND"), "dA13": ("ProbDA13", "K_DA13")}


def _csrc(f):
    with open(os.path.join(ROOT, "moe_expert_ffn_top_gb300", "csrc", f)) as fh:
        return fh.read()


def _code(text):
    """Source text without comments and blank lines."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def problem_source(prob, slot):
    """The section of gemm_problems.cuh that defines `prob` (sections are delimited by
    '// ====' lines; the file's preamble, shared helpers included, comes with every
    problem) and the host block of forward.cu / backward.cu that builds and launches
    it: from the step's comment line above the first launch with profiler slot `slot`
    to the last such launch."""
    text = _csrc("gemm_problems.cuh")
    parts = re.split(r"^// =+$", text, flags=re.M)
    mine = [p for p in parts if re.search(r"\bstruct\s+" + prob + r"\b(?!\w)", p)]
    host = []
    for f in ("forward.cu", "backward.cu"):
        lines = _csrc(f).splitlines()
        hits = [i for i, line in enumerate(lines) if re.search(r"\b" + slot + r"\b", line)]
        if not hits:
            continue
        i = hits[0]
        while i > 0 and not re.match(r"^  // \S", lines[i]):
            i -= 1
        host.append("\n".join(lines[i:hits[-1] + 1]))
    return parts[0] + "".join(mine) + "".join(host)


def src_hash(kernel):
    """Hash of the code behind `kernel` (see above)."""
    h = hashlib.sha256()
    for f in ENGINE_SOURCES:
        h.update(f.encode())
        h.update(_code(_csrc(f)).encode())
    prob, slot = PROBLEM_OF[kernel]
    h.update(prob.encode())
    h.update(_code(problem_source(prob, slot)).encode())
    return h.hexdigest()[:16]


def traffic_for(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it was
    captured on the kernel's current code (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("src_hash") != src_hash(kernel):
        return None
    return e.get("bytes_per_launch")


# ------------------------------------------------------------------ multi-rank timing
def max_over_ranks(dist, v, device):
    """The slowest rank's value (every rank gets it); v itself on a single process."""
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_rank, ms):
    """Whole-job throughput: the units every rank processed over the max-over-ranks time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        self.dev = device_index

    def start(self):
        # 20 ms: the clock under a power cap moves within one 30 ms step
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "20"]
        try:
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [l.strip().split(", ") for l in self.f.read().splitlines() if l.strip()]
        os.unlink(self.f.name)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        for r in rows:
            if len(r) < 9:
                continue
            try:
                samples.append((float(r[1]), float(r[2]), float(r[3]),
                                [n for n, v in zip(names, r[5:9]) if v.strip().lower().startswith("active")]))
            except ValueError:
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # "under load": samples drawing at least 40% of the window's peak power
        # (the sampler also sees the gaps around the timed region)
        pmax = max(p for _, _, p, _ in samples)
        load = [s for s in samples if s[2] >= 0.4 * pmax] or samples
        reasons = sorted({n for s in load for n in s[3]})
        return {"sm_mhz": statistics.median(s[0] for s in load), "sm_max_mhz": max(s[1] for s in samples),
                "reasons": reasons, "samples": len(samples), "samples_under_load": len(load),
                "power_w_median": statistics.median(s[2] for s in load), "power_w_max": pmax}


# ------------------------------------------------------------------ timed regions
def timed_region(fn, steps, stream, local_rank, dist, sample_clocks=True):
    """Runs fn() `steps` times between CUDA events on `stream` (barrier and
    synchronize on both sides), sampling the SM clocks meanwhile.  Returns
    (max-over-ranks ms per call, clock record)."""
    clocks = ClockSampler(local_rank) if sample_clocks else None
    if clocks:
        clocks.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    return max_over_ranks(dist, e0.elapsed_time(e1) / steps, "cuda"), clk


def per_kernel_pass(m, fn, steps, only=None):
    """Per-kernel CUDA-event times of `steps` calls of fn(): {name: (total ms, launches)}.
    only: time just that kernel's launches (no events around any other launch)."""
    m.moe_lora_profile_select(only)
    m.moe_lora_profile_enable(True)
    for _ in range(steps):
        fn()
    torch.cuda.synchronize()
    prof = m.moe_lora_profile_read()
    m.moe_lora_profile_enable(False)
    m.moe_lora_profile_select(None)
    return prof


def base_fmt_of(shp, mx_once=False):
    """The library's base_fmt for a synthetic shape: bf16 0, MXFP4 decoded in the
    GEMMs 1 (or once per pass 2), the native FP4 forward with the rest as 1 (3) or as 2 (4)."""
    if shp.base_fmt == "mxfp4":
        return 2 if mx_once else 1
    if shp.base_fmt == "mxfp4_native":
        return 4 if mx_once else 3
    return 0


def measure_workload(m, name, seed, args, local_rank, dist, world, mx_once=False):
    """A compact record of one more workload (the same step: plan + forward +
    backward), measured after the headline: step time with its own clock record,
    the per-kernel times, the workspace sizes and, for several adapters, the same
    work as standalone single-adapter passes back to back.  mx_once: an MXFP4 base
    decoded once per pass (base_fmt 2) instead of inside the GEMMs (1)."""
    shp = shape(name)
    inp = make_inputs(shp, seed=seed, device="cuda")
    T, H, I, E, k, r, A = shp.T, shp.H, shp.I, shp.E, shp.k, shp.r, shp.A
    R = int((inp["topk_ids"] >= 0).sum())
    d = m.make_dims(T, H, I, E, k, r, A, shp.scale, base_fmt=base_fmt_of(shp, mx_once))
    offs = inp["adapter_offsets"].tolist() if A > 1 else None
    ws = m.Workspaces.allocate(d)
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    dx, dw = torch.empty_like(y), torch.empty(T, k, dtype=torch.float32, device="cuda")
    g = m.alloc_grads(d)
    wts = {n: inp[n] for n in WEIGHTS + ("S1", "S3", "S2") if n in inp}
    x, ids, tw, dy = inp["x"], inp["topk_ids"], inp["topk_w"], inp["dy"]
    stream = torch.cuda.current_stream()

    def step():
        m.moe_lora_plan(d, ids, offs, ws.plan)
        m.moe_lora_forward(d, ws.plan, x, tw, wts, y, ws.saved, ws.fwd)
        m.moe_lora_backward(d, ws.plan, ws.saved, x, tw, dy, wts, dx, dw, g, ws.bwd)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert m.moe_lora_get_error(d, ws.plan) == 0, "device error word set"
    m.moe_lora_launch_count(reset=True)
    ms, clk = timed_region(step, args.steps, stream, local_rank, dist)
    launches = m.moe_lora_launch_count(reset=True) // args.steps
    flops = step_flops(T, R, H, I, r)
    pk = peaks()
    prof = per_kernel_pass(m, step, args.steps)
    value = job_tflops(world, flops, ms)
    base = shp.base_fmt + ((" decoded once per pass" if mx_once else " decoded in the GEMMs")
                           if shp.base_fmt == "mxfp4" else "")
    if shp.base_fmt == "mxfp4_native":
        base = ("mxfp4, gate/up products native (MXFP8 x MXFP4 on block-scaled FP4 tensor cores), "
                "the rest decoded " + ("once per pass" if mx_once else "in the GEMMs"))
    rec = {"workload": f"{name}: T={T} H={H} I={I} E={E} top{k} r={r} A={A} s={shp.scale} base={base}",
           "ms_per_step": round(ms, 3), "value": round(value, 2), "unit": "TFLOP/s",
           "pct_of_bf16_peak": round(100 * value / world / pk["bf16"], 2), "live_routes": R,
           "tflop_per_step": round(flops / 1e12, 4), "launches_per_step": launches, "clocks": clk,
           "kernels_ms": {n: round(t / c, 4) for n, (t, c) in prof.items()},
           "workspace_gb": {w_: round(m.moe_lora_workspace_bytes(d, i_) / 1e9, 3)
                            for w_, i_ in (("plan", 0), ("saved", 1), ("fwd_scratch", 2), ("bwd_scratch", 3))}}
    if shp.base_fmt == "mxfp4_native" and "w13_native" in prof:
        t, c = prof["w13_native"]
        kms = t / c
        f13 = 4.0 * R * H * I + 4.0 * R * I * r   # gate/up base products + the B1/B3 expand
        fp8 = 2.0 * pk["bf16"]                    # dense FP8 peak: measured BF16 x the nominal 4.5 / 2.25
        rec["w13_native"] = {"ms": round(kms, 4), "tflops": round(f13 / kms / 1e9, 1),
                             "peak_fp8_tflops": round(fp8, 1), "frac_of_fp8_peak": round(f13 / kms / 1e9 / fp8, 4),
                             "frac_of_bf16_peak": round(f13 / kms / 1e9 / pk["bf16"], 4),
                             "note": "kind::mxf8f6f4 runs E4M3 x E2M1 at the FP8 rate; the FP8 peak is the "
                                     "measured BF16 burst x 2 (nominal dense ratio), not measured"}
    if A > 1:
        ms_sa, clk_sa = standalone_time(m, inp, shp, offs, args, stream, local_rank, dist)
        rec["standalone"] = {"ms_per_step": round(ms_sa, 3), "value": round(job_tflops(world, flops, ms_sa), 2),
                             "fused_speedup": round(ms_sa / ms, 3), "clocks": clk_sa,
                             "note": f"{A} standalone single-adapter passes of {offs[1] - offs[0]} tokens back "
                                     f"to back (same total work); results equal the fused pass bit for bit "
                                     f"(GPU tests)"}
    del inp, ws, y, dx, dw, g, wts
    torch.cuda.empty_cache()
    return rec


def standalone_time(m, inp, shp, offs, args, stream, local_rank, dist):
    """Several adapters: the fused pass's work as one standalone pass per adapter
    (each its own plan, forward and backward over its token range), back to back."""
    A, H, I, E, k, r = shp.A, shp.H, shp.I, shp.E, shp.k, shp.r
    n = offs[1] - offs[0]
    assert all(offs[a + 1] - offs[a] == n for a in range(A)), "equal token ranges"
    d1 = m.make_dims(n, H, I, E, k, r, 1, shp.scale)
    ws1 = m.Workspaces.allocate(d1)
    y1 = torch.empty(n, H, dtype=torch.bfloat16, device="cuda")
    dx1, dw1 = torch.empty_like(y1), torch.empty(n, k, dtype=torch.float32, device="cuda")
    g1 = m.alloc_grads(d1)
    args_dev = (inp["x"], inp["topk_ids"], inp["topk_w"], inp["dy"])

    def standalone_step():
        for a in range(A):
            sl = slice(offs[a], offs[a + 1])
            wa = {nm: (inp[nm] if nm in ("W1", "W3", "W2") else inp[nm][a:a + 1]) for nm in WEIGHTS}
            x_, ids_, tw_, dy_ = (t[sl] for t in args_dev)
            m.moe_lora_plan(d1, ids_, None, ws1.plan)
            m.moe_lora_forward(d1, ws1.plan, x_, tw_, wa, y1, ws1.saved, ws1.fwd)
            m.moe_lora_backward(d1, ws1.plan, ws1.saved, x_, tw_, dy_, wa, dx1, dw1, g1, ws1.bwd)

    for _ in range(args.warmup):
        standalone_step()
    torch.cuda.synchronize()
    ms, clk = timed_region(standalone_step, args.steps, stream, local_rank, dist)
    assert m.moe_lora_get_error(d1, ws1.plan) == 0, "device error word set"
    del ws1, y1, dx1, dw1, g1
    torch.cuda.empty_cache()
    return ms, clk


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(inp_cpu, shp, seconds_target, max_tokens=512):
    """Times the CPU oracle (forward + backward) on the first tokens of the
    workload, sized to take about `seconds_target`.  Returns (TFLOP/s, info)."""
    import oracle
    oracle.build()
    cores = os.cpu_count()

    def run(n):
        toks = list(range(n))
        R = int((inp_cpu["topk_ids"][:n] >= 0).sum())
        t0 = time.perf_counter()
        oracle.forward(inp_cpu, shp, tokens=toks)
        oracle.backward(inp_cpu, shp, tokens=toks)
        dt = time.perf_counter() - t0
        return dt, step_flops(n, R, shp.H, shp.I, shp.r), R

    n = 4
    dt, fl, R = run(n)
    while dt < seconds_target / 8 and n < max_tokens:
        n = min(max_tokens, 2 * n)
        dt, fl, R = run(n)
    if dt < seconds_target / 2 and n < max_tokens:
        n = int(min(max_tokens, n * seconds_target / max(dt, 1e-3)))
        dt, fl, R = run(n)
    return fl / dt / 1e12, {"tokens": n, "routes": R, "seconds": dt, "cores": cores, "flops": fl}


def host_inputs(shp, seed):
    """The workload's seeded inputs drawn on the device, copied to host memory."""
    inp = make_inputs(shp, seed=seed, device="cuda")
    out = {n: v.cpu() for n, v in inp.items()}
    del inp
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import moe_expert_ffn_top_gb300 as m
    from moe_expert_ffn_top_gb300 import _build
    _build.build()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    shp = shape(args.workload)
    inp = make_inputs(shp, seed=2 + rank, device="cuda")
    T, H, I, E, k, r = shp.T, shp.H, shp.I, shp.E, shp.k, shp.r
    R = int((inp["topk_ids"] >= 0).sum())
    A = shp.A
    d = m.make_dims(T, H, I, E, k, r, A, shp.scale, base_fmt=base_fmt_of(shp))
    offs = inp["adapter_offsets"].tolist() if A > 1 else None  # token range of each adapter
    ws = m.Workspaces.allocate(d)
    y = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    dx = torch.empty_like(y)
    dw = torch.empty(T, k, dtype=torch.float32, device="cuda")
    g = m.alloc_grads(d)
    wts = {n: inp[n] for n in WEIGHTS + ("S1", "S3", "S2") if n in inp}
    stream = torch.cuda.current_stream()

    def step(x, ids, tw, dy):
        m.moe_lora_plan(d, ids, offs, ws.plan)
        m.moe_lora_forward(d, ws.plan, x, tw, wts, y, ws.saved, ws.fwd)
        m.moe_lora_backward(d, ws.plan, ws.saved, x, tw, dy, wts, dx, dw, g, ws.bwd)

    def barrier():
        if dist is not None:
            dist.barrier()

    args_dev = (inp["x"], inp["topk_ids"], inp["topk_w"], inp["dy"])
    # pinned host buffers of the end-to-end leg, allocated before any other host-side
    # work and filled without pageable intermediates (host memory churn makes the
    # kernel compact memory, which stalls copies to and from pinned pages)
    h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in args_dev]
    for hd, t in zip(h_in, args_dev):
        hd.copy_(t)
    h_out = [torch.zeros(t.shape, dtype=t.dtype, pin_memory=True) for t in [y, dx, dw] + [g[n] for n in ADAPTER_GRADS]]
    for _ in range(args.warmup):
        step(*args_dev)
    torch.cuda.synchronize()
    assert m.moe_lora_get_error(d, ws.plan) == 0, "device error word set"

    # ---- device-resident timing.  The roofline's kernel (the largest algorithmic FLOPs
    # per launch; W13 and the W13 dgrad tie and W13 comes first) is timed inside this
    # same region, with CUDA events around its launches only.
    fl, by = kernel_work(T, R, H, I, r, k, E)
    native = shp.base_fmt == "mxfp4_native"
    dom = dominant_kernel(fl, native)
    m.moe_lora_launch_count(reset=True)
    m.moe_lora_profile_select(dom)
    m.moe_lora_profile_enable(True)
    ms, clk = timed_region(lambda: step(*args_dev), args.steps, stream, local_rank, dist)
    live = m.moe_lora_profile_read()
    m.moe_lora_profile_enable(False)
    m.moe_lora_profile_select(None)
    launches = m.moe_lora_launch_count(reset=True)
    flops = step_flops(T, R, H, I, r)
    value = job_tflops(world, flops, ms)

    # ---- forward (plan + forward) and backward timed on their own, as the pages
    # report them (separate passes after the headline region)
    def timed(fn):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(args.steps):
            fn()
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / args.steps

    x_, ids_, tw_, dy_ = args_dev
    ms_fwd = timed(lambda: (m.moe_lora_plan(d, ids_, offs, ws.plan),
                            m.moe_lora_forward(d, ws.plan, x_, tw_, wts, y, ws.saved, ws.fwd)))
    ms_bwd = timed(lambda: m.moe_lora_backward(d, ws.plan, ws.saved, x_, tw_, dy_, wts, dx, dw, g, ws.bwd))

    # ---- per-kernel event timing: one pass with an event pair around every launch
    # (the kernels table and shares), then one pass timing the dominant kernel
    # alone, so no events sit between the other launches (the roofline figure)
    prof = per_kernel_pass(m, lambda: step(*args_dev), args.steps)
    pk = peaks()
    kernels = {}
    for name, (tot, n) in prof.items():
        avg = tot / n
        e = {"ms": round(avg, 4), "launches_per_step": n // args.steps, "share": None}
        if name in fl:
            e["tflops"] = round(fl[name] / (avg * 1e-3) / 1e12, 1)
        elif name in by:
            e["gbs"] = round(by[name] / (avg * 1e-3) / 1e9, 1)
        kernels[name] = e
    tot_all = sum(t for t, _ in prof.values())
    for name, (tot, n) in prof.items():
        kernels[name]["share"] = round(tot / tot_all, 4)
    dom_ms = max_over_ranks(dist, live[dom][0] / live[dom][1], "cuda")
    achieved = fl[dom] / (dom_ms * 1e-3) / 1e12
    gemm_ms = sum(prof[n][0] for n in prof if n in fl) / args.steps
    gemm_flops = sum(fl[n] for n in prof if n in fl)
    # the native W13 runs E4M3 x E2M1 at the FP8 rate: the measured BF16 peak x 2 (the
    # nominal dense ratio), not itself measured
    pscale = 2.0 if native else 1.0
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": pscale * pk["bf16"],
                "unit": "TFLOP/s", "frac": round(achieved / (pscale * pk["bf16"]), 4),
                "traffic": traffic_for(dom) if args.workload == "prod" else None,
                "peak_kind": (f"fp8 dense = bf16 dense burst ({pk['source']}) x 2, " if native else
                              f"bf16 dense, burst ({pk['source']}): ") +
                             f"the timed region is {args.steps} steps of ~{ms:.0f} ms, not a seconds-long loop",
                "frac_of_sustained_peak": round(achieved / (pscale * pk["bf16_sus"]), 4),
                "sustained_peak": pscale * pk["bf16_sus"],
                "kernel_ms": round(dom_ms, 4),
                "timing": "CUDA events on the launch stream around this kernel's launches only, inside the "
                          "headline timed region",
                "grouped_gemms_tflops": round(gemm_flops / (gemm_ms * 1e-3) / 1e12, 1),
                "grouped_gemms_frac_of_burst_peak": round(gemm_flops / (gemm_ms * 1e-3) / 1e12 / pk["bf16"], 4)}
    per_kernel_sum = tot_all / args.steps
    event_pass = {"sum_of_kernels_ms": round(per_kernel_sum, 3), "step_ms": round(ms, 3),
                  "inflation": round(per_kernel_sum / ms, 4),
                  "dominant_kernel_ms_all_events": round(prof[dom][0] / prof[dom][1], 4),
                  "note": "kernels table: a separate pass with an event pair around every launch (each pair "
                          "drains the stream between kernels, so the tails no longer overlap); the sum exceeds "
                          "the step by `inflation`; the roofline times its kernel inside the headline region"}

    # ---- several adapters: the same work as one standalone pass per adapter
    standalone = None
    if A > 1:
        ms_sa, clk_sa = standalone_time(m, inp, shp, offs, args, stream, local_rank, dist)
        standalone = {"ms_per_step": round(ms_sa, 3), "tflops": round(job_tflops(world, flops, ms_sa), 2),
                      "fused_speedup": round(ms_sa / ms, 3), "clocks": clk_sa,
                      "note": f"{A} standalone single-adapter passes of {offs[1] - offs[0]} tokens back to back "
                              f"(same total work); results equal the fused pass bit for bit (GPU tests)"}

    # ---- the routing step ahead of the path (router forward / backward), timed on
    # its own: the headline step takes ids and weights as inputs, as the pages do.
    router = None
    if shp.A == 1 and 16 <= E <= 256 and E % 16 == 0:
        rin = make_router_inputs(T, H, E, k, seed=100 + rank, device="cuda")
        rsc = m.router_scratch(d)
        rids = torch.empty(T, k, dtype=torch.int32, device="cuda")
        rw = torch.empty(T, k, dtype=torch.float32, device="cuda")
        rdWr = torch.empty(E, H, dtype=torch.float32, device="cuda")
        rdx = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
        rf = lambda: m.moe_lora_router_forward(d, rin["x"], rin["Wr"], rids, rw, None, rsc)
        rb = lambda: m.moe_lora_router_backward(d, rin["x"], rin["Wr"], rids, rw, rin["dw"], None, rdWr, rdx, rsc)
        for _ in range(args.warmup):
            rf()
            rb()
        torch.cuda.synchronize()
        rt = []
        for fn in (rf, rb):
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(args.steps):
                fn()
            a1.record(stream)
            torch.cuda.synchronize()
            rt.append(a0.elapsed_time(a1) / args.steps)
        m.moe_lora_profile_enable(True)
        for _ in range(args.steps):
            rf()
            rb()
        torch.cuda.synchronize()
        rprof = m.moe_lora_profile_read()
        m.moe_lora_profile_enable(False)
        assert m.moe_lora_router_get_error(rsc) == 0, "router device error word set"
        rfl = 2.0 * T * E * H
        router = {"ms_forward": round(rt[0], 4), "ms_backward": round(rt[1], 4),
                  "tflops_forward": round(rfl / (rt[0] * 1e-3) / 1e12, 1),
                  "tflops_backward": round(2 * rfl / (rt[1] * 1e-3) / 1e12, 1),
                  "kernels": {n: round(tot / cnt, 4) for n, (tot, cnt) in rprof.items()},
                  "note": "softmax top-k router GEMM (fused epilogue) and its backward "
                          "(dlogits, dx += dlogits W_r, dW_r); not part of the headline step"}
        del rin, rsc, rids, rw, rdWr, rdx
        torch.cuda.empty_cache()

    # ---- end to end through the public API: pinned host inputs in, results out.
    # Every step copies its own inputs host->device and reads all of its results
    # back device->host inside the timed region; copies run on their own streams
    # with double-buffered device inputs/outputs, so step i's read-back and step
    # i+1's upload overlap the compute of their neighbours.  Each copy follows its
    # data: dy goes up while the forward runs (only the backward reads it) and y
    # comes back while the backward runs.
    d_in = [[torch.empty_like(t) for t in args_dev] for _ in range(2)]
    outs_2 = [[y, dx, dw] + [g[n] for n in ADAPTER_GRADS]]
    y2, dx2, dw2, g2 = torch.empty_like(y), torch.empty_like(dx), torch.empty_like(dw), m.alloc_grads(d)
    outs_2.append([y2, dx2, dw2] + [g2[n] for n in ADAPTER_GRADS])
    bi = sum(t.numel() * t.element_size() for t in h_in)
    bo = sum(t.numel() * t.element_size() for t in h_out)
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    fwd_in_ready, bwd_in_ready, in_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    fwd_done, bwd_done, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e_ in in_free + out_free:
        e_.record(stream)

    copy_ev = []  # per timed step: start/end of the forward and backward uploads and read-backs

    def copies(pairs, stream_, ce, j):
        if ce is not None:
            ce[j].record(stream_)
        for src, dst in pairs:
            dst.copy_(src, non_blocking=True)
        if ce is not None:
            ce[j + 1].record(stream_)

    def run_e2e(nsteps, timed=False):
        for i in range(nsteps):
            b_ = i % 2
            ce = [torch.cuda.Event(enable_timing=True) for _ in range(8)] if timed else None
            xi, idsi, twi, dyi = d_in[b_]
            with torch.cuda.stream(up):  # x, ids, weights, then dy
                up.wait_event(in_free[b_])
                copies(zip(h_in[:3], d_in[b_][:3]), up, ce, 0)
                fwd_in_ready[b_].record(up)
                copies([(h_in[3], dyi)], up, ce, 2)
                bwd_in_ready[b_].record(up)
            stream.wait_event(fwd_in_ready[b_])
            stream.wait_event(out_free[b_])
            yo, dxo, dwo = outs_2[b_][0], outs_2[b_][1], outs_2[b_][2]
            go = dict(zip(ADAPTER_GRADS, outs_2[b_][3:]))
            m.moe_lora_plan(d, idsi, offs, ws.plan, stream)
            m.moe_lora_forward(d, ws.plan, xi, twi, wts, yo, ws.saved, ws.fwd, stream)
            fwd_done[b_].record(stream)
            stream.wait_event(bwd_in_ready[b_])
            m.moe_lora_backward(d, ws.plan, ws.saved, xi, twi, dyi, wts, dxo, dwo, go, ws.bwd, stream)
            in_free[b_].record(stream)
            bwd_done[b_].record(stream)
            with torch.cuda.stream(down):  # y, then the backward's results
                down.wait_event(fwd_done[b_])
                copies([(yo, h_out[0])], down, ce, 4)
                down.wait_event(bwd_done[b_])
                copies(zip(outs_2[b_][1:], h_out[1:]), down, ce, 6)
                out_free[b_].record(down)
            if timed:
                copy_ev.append(ce)

    run_e2e(args.warmup)
    torch.cuda.synchronize()
    barrier()
    e2e_clocks = ClockSampler(local_rank)
    e2e_clocks.start()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(up)
    run_e2e(args.steps, timed=True)
    torch.cuda.current_stream(torch.device("cuda")).wait_stream(down)
    s1.record(down)
    torch.cuda.synchronize()
    barrier()
    e2e_clk = e2e_clocks.stop()
    ms_e2e = max_over_ranks(dist, s0.elapsed_time(s1) / args.steps, "cuda")
    # per-step copy times: a host under memory compaction (seen right after a large
    # test run) stalls single pinned copies for ~0.1 s; counted here, not removed
    t_up = [e[0].elapsed_time(e[1]) + e[2].elapsed_time(e[3]) for e in copy_ev]
    t_dn = [e[4].elapsed_time(e[5]) + e[6].elapsed_time(e[7]) for e in copy_ev]
    med_up, med_dn = statistics.median(t_up), statistics.median(t_dn)
    stalls = sum(1 for v in t_up if v > 3 * med_up) + sum(1 for v in t_dn if v > 3 * med_dn)
    e2e = {"value": round(job_tflops(world, flops, ms_e2e), 2), "unit": "TFLOP/s",
           "ms_per_step": round(ms_e2e, 3), "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
           "clocks": e2e_clk,
           "copy_ms": {"upload_median": round(med_up, 2), "upload_max": round(max(t_up), 2),
                       "readback_median": round(med_dn, 2), "readback_max": round(max(t_dn), 2),
                       "stalled_copies": stalls},
           "copies": "pinned host memory, own streams; dy uploaded during the forward and y read back "
                     "during the backward; overlapped with neighbouring steps' compute"}

    # ---- CPU oracle baseline (rank 0, single GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        del ws
        torch.cuda.empty_cache()
        host = {n: v.cpu() for n, v in inp.items()}
        oshp = shp
        if A > 1:  # the oracle takes one adapter: adapter 0's token range and factors
            sl = slice(offs[0], offs[1])
            host = {n: (host[n][sl] if n in ("x", "dy", "topk_ids", "topk_w") else
                        host[n] if n in ("W1", "W3", "W2") else host[n][0:1].contiguous())
                    for n in ("x", "dy", "topk_ids", "topk_w") + WEIGHTS}
            host["adapter_offsets"] = torch.tensor([0, offs[1] - offs[0]], dtype=torch.int64)
            oshp = Shape(T=offs[1] - offs[0], H=H, I=I, E=E, k=k, r=r, A=1, scale=shp.scale)
        v, info = oracle_sample(host, oshp, args.cpu_seconds)
        cpu = {"value": round(v, 6), "unit": "TFLOP/s", "cores": info["cores"], "kind": "oracle",
               "sample": f"first {info['tokens']} tokens ({info['routes']} routes) of the same workload"
                         f"{' (adapter 0)' if A > 1 else ''}, "
                         f"forward+backward, {info['seconds']:.1f} s, plain C FP32 oracle with OpenMP"}

    # ---- the MXFP4-base workload (same shape, E2M1 + UE8M0 frozen base) and the
    # 16-adapter fused pass, each measured after the headline with its own clocks
    subs = {}
    if args.workload == "prod" and world == 1 and not args.no_sub_records:
        subs["mxfp4"] = measure_workload(m, "prod_mxfp4", 3, args, local_rank, dist, world)
        subs["mxfp4_once"] = measure_workload(m, "prod_mxfp4", 3, args, local_rank, dist, world, mx_once=True)
        subs["native"] = measure_workload(m, "prod_native", 3, args, local_rank, dist, world)
        subs["native_once"] = measure_workload(m, "prod_native", 3, args, local_rank, dist, world, mx_once=True)
        subs["multi"] = measure_workload(m, "multi", 4, args, local_rank, dist, world)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; shapes and distributions of the pages' workload)",
            "config": {"workload": f"{args.workload}: T={T} H={H} I={I} E={E} top{k} r={r} s={shp.scale}, "
                                   f"fwd+bwd incl. routing plan",
                       "tokens_per_gpu": T, "live_routes_per_gpu": R, "tflop_per_step_per_gpu": round(flops / 1e12, 3),
                       "pct_of_bf16_peak": round(100 * value / world / pk["bf16"], 2),
                       "parallelism": "replicas only (one independent batch per GPU, no collectives)",
                       "adapters": A,
                       "l2": f"inputs larger than L2 ({3 * E * H * I * 2 / 1e9:.1f} GB frozen weights), no flush"},
            "forward_ms": round(ms_fwd, 3), "backward_ms": round(ms_bwd, 3),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clk, "kernels": kernels, "event_pass": event_pass, "router": router,
            "standalone": standalone, **subs,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------ reference arm
def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores: each step is a bounded sample
    (the first tokens of the same workload) of forward + backward."""
    if rank != 0:
        return
    shp = shape(args.workload)
    host = host_inputs(shp, seed=2)
    per_step = max(1.0, args.cpu_seconds / 3)
    import oracle
    oracle.build()
    # size one step's sample once (calibration is not timed)
    _, info = oracle_sample(host, shp, per_step)
    n = info["tokens"]
    toks = list(range(n))
    R = int((host["topk_ids"][:n] >= 0).sum())
    fl = step_flops(n, R, shp.H, shp.I, shp.r)
    for _ in range(args.warmup):
        oracle.forward(host, shp, tokens=toks[:2])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(host, shp, tokens=toks)
        oracle.backward(host, shp, tokens=toks)
    dt = (time.perf_counter() - t0) / args.steps
    v = fl / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; same inputs as our arm)",
            "config": {"workload": f"{args.workload}: first {n} tokens per step ({R} routes), "
                                   f"T={shp.T} H={shp.H} I={shp.I} E={shp.E} top{shp.k} r={shp.r}"},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"first {n} tokens of the workload per step, forward+backward"},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prod", choices=["prod", "prod_mxfp4", "prod_e16", "prod_e16_mxfp4", "prod_native",
                                                            "prod_e16_native", "tiny", "edge", "multi"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-records", action="store_true",
                    help="skip the MXFP4-base and 16-adapter records that follow the headline")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
