#!/usr/bin/env python3
"""Benchmark of the fused 4-bit AdamW optimizer step on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: the Llama-style 8B parameter set (291 tensors,
8,030,261,248 FP32 master weights, BF16 gradients, 4-bit ZIP-SR state, about
73 GB resident in HBM).  One step = one q4adamw_step over every tensor.  The
timed region holds exactly K steps, bracketed by a barrier and
torch.cuda.synchronize(); each step's working set (113 GB) exceeds the 126 MB
L2, so no flush is needed between steps.  Rank 0 prints one JSON line.

Metric: optimizer-step parameters per second (whole job); the roofline object
reports achieved HBM GB/s of the step kernel against the measured copy peak.
Algorithmic bytes per parameter: 2 (BF16 grad read) + 4 + 4 (FP32 master read
and write) + 2 (BF16 weight write) + 2 x 1.0625 (packed m+v codes and block
scales, read and written) = 14.125.

--impl reference times the CPU oracle (oracle/, single thread) on a bounded
sample of the same workload: it is the reference arm of this benchmark.
Multi-GPU (torchrun, one rank per GPU): every rank runs an independent replica
of the workload on its own GPU (weak scaling; the step has no data-path
collective).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

BYTES_PER_PARAM = 2 + 4 + 4 + 2 + 2 * 1.0625           # packed (non-factored) tensors
BYTES_PER_PARAM_FACTORED = 2 + 4 + 4 + 2 + 2 * 0.53125  # rank >= 2 tensors, factored v (m only)
NOMINAL_HBM_GBS = 8000.0
# rounding-variant call flags (Q4_M_SR_ALL, Q4_V_UPDATE_RTN, Q4_V_NEXT_R)
VARIANT_FLAGS = {"none": 0, "m_sr_all": 0x2, "v_update_rtn": 0x4, "v_next_r": 0x8, "v_next_r_rtn": 0xC}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama8b_zipsr")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle time of the CPU sample")
    ap.add_argument("--variant", default="none", choices=sorted(VARIANT_FLAGS),
                    help="rounding variant (call flag) to time instead of the recipe's own rules")
    ap.add_argument("--max-grad-norm", type=float, default=None,
                    help="time the step with global gradient-norm clipping (sum-of-squares pass + clipped step)")
    ap.add_argument("--tensors", type=int, default=0,
                    help="keep only the first N tensors of the workload (small cases for profiling)")
    ap.add_argument("--tensor-slice", default="",
                    help="keep tensors a:b of the workload (e.g. 1:10 = the first decoder layer of the 8B set)")
    ap.add_argument("--companion", default="auto",
                    help="a second workload timed after the first and reported under 'companion' "
                         "('auto': the 8B ZE-EDEN step beside the default 8B ZIP-SR one; 'none': skip)")
    return ap.parse_args()


def companion_workload(args):
    """The workload timed beside the main one: the 8B model is specified with
    both second-moment recipes, each timed over the same number of steps."""
    if args.companion == "none":
        return None
    if args.companion != "auto":
        return args.companion
    plain = not args.tensors and not args.tensor_slice and args.variant == "none" and args.max_grad_norm is None
    return "llama8b_zeeden" if plain and args.workload == "llama8b_zipsr" else None


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float) -> float:
    """Maximum of a per-rank scalar over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6400.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, mem, power, reasons = [], [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for dst, k in ((power, 3), (mem, 9)):
                try:
                    dst.append(float(parts[k]))
                except (ValueError, IndexError):
                    pass
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "mem_mhz": statistics.median(mem) if mem else None,
                "power_w": statistics.median(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _strip_comments(src: str) -> str:
    """C/C++ source without comments and with whitespace runs collapsed
    (string and character literals kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of every source of the CUDA library, comments and layout ignored
    (a traffic record is valid only for the code it was measured on)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "bit_quantized_adamw_q4adamw_b300", "csrc")
    for name in sorted(os.listdir(d)):
        with open(os.path.join(d, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def traffic_record(workload: str):
    """DRAM bytes per parameter of the step kernel from a committed ncu summary
    (profiles/step_kernel_traffic.json), valid only for the kernel source it was
    taken on."""
    p = os.path.join(ROOT, "profiles", "step_kernel_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(workload)
    if not rec or rec.get("kernel_sha") != kernel_source_hash():
        return None
    return rec


# ---------------------------------------------------------------- workload setup
def build_state(w, device):
    import torch

    import bit_quantized_adamw_q4adamw_b300 as q4
    from bit_quantized_adamw_q4adamw_b300 import workloads as W
    st = q4.Q4State(w.tensors, w.recipe, device=device)
    for i, s in enumerate(w.tensors):
        st.view(i, "param").copy_(W.init_param(s, i, device=device))
        W.draw_grad(w, s, i, w.first_step, device=device, out=st.view(i, "grad"))
    st.init()
    torch.cuda.synchronize()
    return st


def algorithmic_bytes(st, recipe) -> float:
    total = 0.0
    for sl in st.slots:
        if st.is_factored(sl):
            total += sl.numel * BYTES_PER_PARAM_FACTORED + (sl.rows + sl.numel // sl.rows) * 8
        else:
            total += sl.numel * BYTES_PER_PARAM
    return total


def launches_per_step(st, clip: bool = False, flags: int = 0) -> int:
    # step kernel: two launches when one instantiation does not suit every
    # tensor (a factored list with packed 1-D tensors; ZIP-SR / ZE-EDEN with
    # stochastic m rounding on some tensors only); factored statistics (4
    # kernels: the pass over g, rows, columns, mean(R)); clipping's sum of
    # squares (3)
    live = [s for s in st.slots if s.numel > 0]
    fact = [st.is_factored(s) for s in live]
    if st.recipe in ("zip_sr", "ze_eden"):
        msr = [bool(flags & 0x2) or bool((s.flags & 0x1) and (flags & 0x1)) for s in live]
    else:
        msr = [False]
    split = (any(fact) and not all(fact)) or (any(msr) and not all(msr))
    return (2 if split else 1) + (4 if any(fact) else 0) + (3 if clip else 0)


def time_sqnorm(st, stream, iters: int) -> float:
    """Mean duration (ms) of one q4adamw_grad_sqnorm call (its three kernels)."""
    import torch
    st.grad_sqnorm(stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        st.grad_sqnorm(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(w, target_seconds: float, device_gen: str = "cpu"):
    """Time the oracle on a bounded, block-aligned sample of the workload.

    The sample takes whole-tensor prefixes (multiples of 128 elements) in
    workload order, sized from a short probe so that the timed oracle work lasts
    about target_seconds.  Inputs are drawn with the same generators on the CPU.
    Returns (params_per_second, sample_description, params)."""
    import numpy as np
    import torch

    from bit_quantized_adamw_q4adamw_b300 import workloads as W
    from oracle import oracle as O
    h = W.HYPER
    flags = O.LM_HEAD_SR_ACTIVE if w.lm_head_sr else 0

    def run(n_target):
        done, secs, parts = 0, 0.0, []
        for i, s in enumerate(w.tensors):
            if done >= n_target:
                break
            take = min(s.numel, ((n_target - done + 127) // 128) * 128)
            if st_factored(w, s):
                take = s.numel  # factored statistics need the whole tensor
            th = W.init_param(s, i, n=take).numpy()
            g = W.draw_grad(w, s, i, w.first_step, n=take)
            gb = g.view(torch.int16).numpy().view(np.uint16)
            t = O.OracleTensor.zeros_state(th, i, rows=s.rows if take == s.numel else 1, flags=s.flags,
                                           recipe=w.recipe)
            t0 = time.perf_counter()
            t.step(gb, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], w.first_step, 0, w.recipe,
                   flags)
            secs += time.perf_counter() - t0
            done += take
            parts.append(f"{s.name}[:{take}]")
        return done, secs, parts

    def st_factored(w, s):
        return w.recipe == "factored" and bool(s.flags & W.T_FACTORED)

    n0, s0, _ = run(2_000_000)
    rate = n0 / max(s0, 1e-9)
    n_target = int(min(max(rate * target_seconds, 1_000_000), w.numel))
    n, secs, parts = run(n_target)
    desc = (f"first {n} of {w.numel} params of {w.name} in tensor order "
            f"({len(parts)} tensor prefixes), one step t={w.first_step}")
    return n / secs, desc, n, secs


# ---------------------------------------------------------------- arms
def get_workload(args):
    import dataclasses

    from bit_quantized_adamw_q4adamw_b300 import workloads as W
    w = W.WORKLOADS[args.workload]
    if args.tensors > 0:
        w = dataclasses.replace(w, name=f"{w.name}[:{args.tensors}]", tensors=w.tensors[:args.tensors])
    if args.tensor_slice:
        a, b = (int(x) for x in args.tensor_slice.split(":"))
        w = dataclasses.replace(w, name=f"{w.name}[{a}:{b}]", tensors=w.tensors[a:b])
    return w


def workload_config(w, world) -> dict:
    """The workload as both arms name it in their JSON lines."""
    alg = sum(s.numel * (BYTES_PER_PARAM_FACTORED if (w.recipe == "factored" and s.flags & 0x2) else BYTES_PER_PARAM)
              for s in w.tensors)
    return {"workload": w.name, "params": w.numel, "tensors": len(w.tensors), "recipe": w.recipe,
            "lm_head_sr": w.lm_head_sr, "parallelism": f"replicas{world}",
            "l2": f"inputs larger than L2 ({alg / 1e9:.1f} GB per step)"}


def run_reference(args, rank, world):
    """The oracle, single-threaded, each step a bounded sample of the workload.
    Everything reported is measured on that sample: params/s is the sample's
    parameters over the oracle's time, ms_per_step the oracle's time per step
    (sample_params_per_step parameters, not the whole workload)."""
    if rank != 0:
        return
    w = get_workload(args)
    per_step = max(args.cpu_seconds / max(args.steps, 1), 0.5)
    secs_total, desc, n = 0.0, "", 0
    for k in range(args.warmup + args.steps):
        v, desc, n, secs = oracle_sample(w, per_step if k >= args.warmup else 0.2)
        if k >= args.warmup:
            secs_total += secs
    value = args.steps * n / secs_total if secs_total > 0 else 0.0
    cpu = {"value": value, "unit": "params/s", "cores": 1, "host_cores": os.cpu_count(), "kind": "oracle",
           "sample": f"each step: {desc}; {secs_total:.2f} s of oracle time over {args.steps} steps"}
    line = {
        "impl": "reference", "metric": "optimizer-step params/sec", "value": value, "unit": "params/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs_total / args.steps if args.steps else None,
        "sample_params_per_step": n, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": cpu,
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist

    from bit_quantized_adamw_q4adamw_b300 import workloads as W
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = get_workload(args)
    h = W.HYPER
    flags = (1 if w.lm_head_sr else 0) | VARIANT_FLAGS[args.variant]
    st = build_state(w, dev)
    stream = torch.cuda.current_stream(dev)

    mgn = args.max_grad_norm

    def one_step(t):
        st.step(t, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], seed=0, flags=flags, stream=stream,
                max_grad_norm=mgn)

    t = w.first_step
    for _ in range(args.warmup):
        one_step(t)
        t += 1
    torch.cuda.synchronize()
    main_alg = algorithmic_bytes(st, w.recipe)
    main_launches = launches_per_step(st, mgn is not None, flags)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs[0].record(stream)
    for k in range(args.steps):
        one_step(t)
        t += 1
        evs[k + 1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    per = [evs[k].elapsed_time(evs[k + 1]) for k in range(args.steps)]
    total_ms = max_over_ranks(evs[0].elapsed_time(evs[-1]))
    ms_per_step = total_ms / args.steps
    value = world * w.numel * args.steps / (total_ms / 1e3)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        e2e = run_e2e(args, st, w, dev, stream, t)
        t += args.e2e_steps + 1

    sq_ms = time_sqnorm(st, stream, max(3, args.steps)) if mgn is not None else None
    comp = None
    cname = companion_workload(args)
    if cname:
        # the main state is released first: both 8B states do not need to be resident
        st = None
        torch.cuda.empty_cache()
        comp = time_companion(args, W.WORKLOADS[cname], dev, stream, rank, local)
    if rank != 0:
        return
    alg = main_alg + (2.0 * w.numel if mgn is not None else 0.0)
    peak, peak_kind = peaks()
    mean_ms = statistics.mean(per)
    achieved = alg / (mean_ms / 1e3) / 1e9
    tr = traffic_record(w.name)
    line = {
        "metric": "optimizer-step params/sec", "value": value, "unit": "params/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, world),
        "step_ms": {"median": statistics.median(per), "p10": sorted(per)[len(per) // 10],
                    "p90": sorted(per)[min(len(per) - 1, (9 * len(per)) // 10)]},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.4 TB/s",
                     "traffic": (tr["dram_bytes_per_param"] * w.numel) if tr else None,
                     "traffic_source": tr["measured_on"] if tr else "no ncu record for this kernel source",
                     "algorithmic_bytes": alg, "kernel": "step_kernel (one launch per step)",
                     "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS},
        "gpu_launches": main_launches * args.steps,
        "clocks": clocks,
    }
    if args.variant != "none":
        line["config"]["variant"] = args.variant
    if mgn is not None:
        # the timed step is the sum-of-squares pass plus the clipped step: the
        # roofline above covers both (2 more bytes per parameter); the pass is
        # also timed alone here
        line["config"]["max_grad_norm"] = mgn
        line["roofline"]["kernel"] = "sqnorm pass (3 kernels) + step_kernel, per step"
        sq_tr = traffic_record("sqnorm_chunk_kernel")
        line["roofline"]["traffic"] = ((tr["dram_bytes_per_param"] + sq_tr["dram_bytes_per_param"]) * w.numel
                                       if tr and sq_tr else None)
        line["sqnorm_pass"] = {"ms": sq_ms, "bytes": 2.0 * w.numel,
                               "achieved_gbs": 2.0 * w.numel / (sq_ms / 1e3) / 1e9,
                               "frac": 2.0 * w.numel / (sq_ms / 1e3) / 1e9 / peak}
    if e2e:
        line["e2e"] = e2e
    if comp:
        line["companion"] = comp
    if not args.no_cpu_baseline:
        v, desc, n, secs = oracle_sample(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "params/s", "cores": 1, "host_cores": os.cpu_count(),
                                "kind": "oracle", "sample": f"{desc}; {secs:.1f} s single-threaded"}
    print(json.dumps(line), flush=True)


def time_companion(args, w, dev, stream, rank, gpu_index):
    """The companion workload timed like the main one (W warm-up steps, then K
    steps between CUDA events, clocks sampled); its own roofline and launch
    count.  Called on every rank; rank 0's figures are reported."""
    import torch
    h = W_HYPER()
    flags = 1 if w.lm_head_sr else 0
    st = build_state(w, dev)
    t = w.first_step
    for _ in range(args.warmup):
        st.step(t, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 0, flags, stream)
        t += 1
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_index) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for k in range(args.steps):
        st.step(t, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 0, flags, stream)
        t += 1
        evs[k + 1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None
    per = [evs[k].elapsed_time(evs[k + 1]) for k in range(args.steps)]
    mean_ms = statistics.mean(per)
    alg = algorithmic_bytes(st, w.recipe)
    peak, _ = peaks()
    achieved = alg / (mean_ms / 1e3) / 1e9
    tr = traffic_record(w.name)
    out = {"config": workload_config(w, 1), "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": evs[0].elapsed_time(evs[-1]) / args.steps, "value": w.numel / (mean_ms / 1e3),
           "unit": "params/s",
           "step_ms": {"median": statistics.median(per), "p10": sorted(per)[len(per) // 10],
                       "p90": sorted(per)[min(len(per) - 1, (9 * len(per)) // 10)]},
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                        "traffic": (tr["dram_bytes_per_param"] * w.numel) if tr else None,
                        "algorithmic_bytes": alg},
           "gpu_launches": launches_per_step(st, False, flags) * args.steps, "clocks": clocks}
    del st
    torch.cuda.empty_cache()
    return out


def run_e2e(args, st, w, dev, stream, t0):
    """Same metric through the public API with host buffers: per step, copy the
    BF16 gradients from pinned host memory, run q4adamw_step, copy the BF16
    weights back to pinned host memory.  The two copies run on their own
    streams, ordered by events: the upload of step t+1's gradients waits only
    for step t's kernel (which has consumed the gradient buffer), and step
    t+1's kernel waits for the download of step t's weights (which frees the
    BF16 buffer), so the download of step t and the upload of step t+1 share
    the host link in opposite directions."""
    import torch
    h = W_HYPER()
    n = st.grad.numel()
    try:
        g_host = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
        out_host = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
    except RuntimeError as e:
        return {"value": None, "unit": "params/s", "error": f"pinned allocation failed: {e}"[:200]}
    g_host.copy_(st.grad)
    torch.cuda.synchronize()
    flags = (1 if w.lm_head_sr else 0) | VARIANT_FLAGS[args.variant]
    mgn = args.max_grad_norm
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(t, steps):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        s_up.wait_event(ev0)
        s_down.wait_event(ev0)
        kdone = down = None
        for _ in range(steps):
            up = torch.cuda.Event()
            with torch.cuda.stream(s_up):
                if kdone is not None:
                    s_up.wait_event(kdone)
                st.grad.copy_(g_host, non_blocking=True)
                up.record(s_up)
            stream.wait_event(up)
            if down is not None:
                stream.wait_event(down)
            st.step(t, h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], 0, flags, stream,
                    max_grad_norm=mgn)
            kdone = torch.cuda.Event()
            kdone.record(stream)
            down = torch.cuda.Event()
            with torch.cuda.stream(s_down):
                s_down.wait_event(kdone)
                out_host.copy_(st.param_bf16, non_blocking=True)
                down.record(s_down)
            t += 1
        stream.wait_event(down)
        ev1.record(stream)
        torch.cuda.synchronize()
        return t, ev0.elapsed_time(ev1) / steps

    t, _ = run(t0, 1)           # one untimed round trip
    t, ms = run(t, args.e2e_steps)
    return {"value": w.numel / (ms / 1e3), "unit": "params/s", "h2d_bytes_per_step": 2 * n,
            "d2h_bytes_per_step": 2 * n, "ms_per_step": ms, "steps": args.e2e_steps,
            "copies": "upload of step t+1 concurrent with download of step t (separate streams)"}


def W_HYPER():
    from bit_quantized_adamw_q4adamw_b300 import workloads as W
    return W.HYPER


def main():
    args = parse()
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
