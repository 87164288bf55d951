"""Benchmark of the NVFP4 W4A16 MoE layer on GB300 (one JSON line on stdout).

Headline workload: the 2-token MTP decode step of the GLM-5.3-Flash routed-
expert layer (128 experts, hidden 4096, expert intermediate 1536, top-8, 1
token + 1 speculative token), synthetic seeded inputs (synth/).  A step is one
call of nvfp4_moe_forward: route -> permute -> gate/up GEMV + SwiGLU -> down
GEMV -> weighted combine.  The same line carries, under config.secondary, the
16-token decode step and the 1024- and 16384-token prefill workloads, each with
its own step time, tokens/s and dominant-kernel roofline.

Measured:
* value: tokens/s with inputs resident in HBM; each step is one replay of a
  CUDA graph holding one forward, timed with CUDA events on the launching
  stream; L2 is flushed (256 MiB write) before every step, outside the events;
* e2e: the same metric through the C ABI with the step's inputs copied from
  pinned host memory and the output read back, all inside the events;
* roofline: the dominant kernel, its algorithmic work per launch over its
  CUDA-event duration on the library's stream: decode, the fused kernel's
  bytes (the touched experts' NVFP4 weights, logits, x and out) against the
  measured HBM copy bandwidth; prefill, the gate/up GEMM's flops against the
  measured BF16 tensor-core peak;
* cpu_baseline: the float64 CPU oracle on a bounded sample of the step (at
  most 16 tokens), over a process pool with one process per visible core.
--impl reference times the oracle alone the same way (the CPU reference arm).
--workload kda_in_proj_mtp | kda_in_proj_1k | linear_tiny runs the dense
W4A16 linear instead (nvfp4_linear_forward on the fused KDA in_proj shape,
N=12576 K=4096, at T=2 and T=1024), with the same keys.
Multi-GPU: replicas only (one independent layer per rank, no collective in
the data path); value is the tokens of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s; decode weight GB/s & prefill TFLOP/s as % of GB300 roofline"
WORKLOAD = "decode_mtp"
FLUSH_BYTES = 256 << 20
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "decode_stream_kernel_decode_mtp.json")


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="time only --workload (the default line also carries decode_c16, prefill_1k, prefill_16k)")
    ap.add_argument("--w4a4", action="store_true",
                    help="the W4A4 comparison variant (activations quantised to NVFP4 with input scales)")
    ap.add_argument("--router", action="store_true",
                    help="compute the router logits in the library (nvfp4_moe_forward_routed) inside each step")
    return ap.parse_args()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _workload_desc(cfg):
    shared = " + 1 shared expert" if cfg.shared else ""
    return (f"{cfg.name}: E{cfg.num_experts} H{cfg.hidden} I{cfg.inter} top{cfg.top_k}{shared} T{cfg.tokens}, "
            f"NVFP4 (E2M1 + E4M3/16 + FP32/tensor) experts, BF16 activations")


# ---------------------------------------------------------------------------
# CPU oracle timing (the baseline and the reference arm): the float64 oracle,
# unchanged, over a spawn process pool, one task per touched expert, one BLAS
# thread per process, as many processes as cores visible to this process
# ---------------------------------------------------------------------------

def _time_oracle_steps(inp, steps, warm, pool):
    """Wall time of each of `steps` full layer steps of the oracle (after
    `warm` untimed ones) on the pool."""
    from oracle.pool import moe_forward_pool
    cfg = inp.config
    times = []
    for s in range(warm + steps):
        t0 = time.perf_counter()
        moe_forward_pool(inp.logits, inp.x_bits, inp.weights, cfg.top_k, num_shared=cfg.shared, pool=pool)
        if s >= warm:
            times.append(time.perf_counter() - t0)
    return times


def _oracle_sample(inp):
    """A bounded sample of the workload for the CPU legs: at most 16 tokens."""
    from synth import make_inputs
    ns = min(inp.config.tokens, 16)
    return (make_inputs(inp.config.with_tokens(ns)) if ns < inp.config.tokens else inp), ns


def cpu_baseline(inp, reps=3):
    """The oracle on the host's cores, timed on a bounded sample of the step."""
    from oracle.pool import make_pool
    sub, ns = _oracle_sample(inp)
    pool, n = make_pool()
    try:
        times = _time_oracle_steps(sub, reps, 1, pool)
    finally:
        pool.close()
        pool.join()
    cfg = inp.config
    return {"value": ns / statistics.mean(times), "unit": "tokens/s", "cores": n, "kind": "oracle",
            "sample": f"{ns} token(s) of the step ({ns * (cfg.top_k + cfg.shared)} routed rows), the whole "
                      f"float64 layer (route, expert FFNs, combine), {reps} timed repetitions after one warm-up; "
                      f"a spawn pool of {n} processes (one per core in os.sched_getaffinity), one task per "
                      f"touched expert, 1 BLAS thread each"}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from synth import make_inputs
    from oracle.pool import make_pool
    inp = make_inputs(args.workload)
    sub, ns = _oracle_sample(inp)
    pool, n = make_pool()
    try:
        times = _time_oracle_steps(sub, args.steps, args.warmup, pool)
    finally:
        pool.close()
        pool.join()
    sec = sum(times)
    value = args.steps * ns / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded PCG64, shapes of the pages' workloads)",
        "config": {"workload": _workload_desc(inp.config)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": n, "kind": "oracle",
                         "sample": f"each step the whole float64 layer on {ns} token(s) of the workload "
                                   f"(route, expert FFNs, combine), a spawn pool of {n} processes, one task "
                                   f"per touched expert, 1 BLAS thread each"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.fh = None

    def start(self):
        try:
            self.fh = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
                                          "--format=csv,noheader,nounits", "-lms", "20", "-i", str(self.idx)],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.seek(0)
        rows = [r.split(",") for r in self.fh.read().strip().splitlines() if r.count(",") == len(self.FIELDS) - 1]
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].strip().replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def replica_throughput(ms, ms_e2e, tokens_per_rank, ws, device):
    """Replicas only: every rank runs its own copy of the layer on its own
    tokens.  The step time is the slowest rank's (MAX over ranks), and the
    whole job's throughput is all ranks' tokens over that time.  Returns
    (ms, ms_e2e, tokens/s, e2e tokens/s)."""
    import torch
    if ws > 1:
        t = torch.tensor([ms, ms_e2e], dtype=torch.float64, device=device)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms, ms_e2e = float(t[0]), float(t[1])
    return ms, ms_e2e, ws * tokens_per_rank / (ms / 1e3), ws * tokens_per_rank / (ms_e2e / 1e3)


def code_fingerprint(text):
    """sha256 of a CUDA/C++ source with its comments and whitespace removed:
    it changes when the code does, not when a comment does."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return hashlib.sha256(re.sub(r"\s+", "", text).encode()).hexdigest()


def _traffic_for(kernel_src):
    """DRAM traffic per launch from the committed ncu summary, if the kernel's
    code is unchanged since it was captured; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            rec = json.load(f)
        with open(kernel_src, encoding="utf-8") as f:
            fp = code_fingerprint(f.read())
        if rec.get("code_sha256") == fp:
            return rec.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


def _peak(key, fallback):
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)[key]), "measured"
    except Exception:
        return fallback, "fallback"


def measure_layer(name, steps, warmup, dev, flush, barrier, ws=1, router=False, w4a4=False):
    """One workload's timed steps on this GPU.  Returns a dict: step time,
    tokens/s, end-to-end tokens/s through the C ABI with host buffers, the
    dominant kernel's roofline, and per-stage times (prefill)."""
    import torch
    import nvfp4_weight_only_w4a16_gb300 as pkg
    from synth import make_inputs, make_router_weight, make_input_scales
    inp = make_inputs(name)
    cfg = inp.config
    T, k, H, E, I, S = cfg.tokens, cfg.top_k, cfg.hidden, cfg.num_experts, cfg.inter, cfg.shared
    decode = T <= 16
    layer = pkg.MoELayer(E, H, I, T, k, device=dev.index, num_shared_experts=S)
    n_ours = 1 if decode else 6     # kernels of ours per forward (decode / prefill path)
    pkg.upload_layer(layer, inp.weights, dev)
    if w4a4:
        layer.nvfp4_moe_set_act_quant(torch.from_numpy(make_input_scales(cfg)).to(dev))
    logits = torch.from_numpy(inp.logits).to(dev)
    x = torch.from_numpy(inp.x_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    if router:
        # the logits come from the router linear on the GPU inside every step
        layer.nvfp4_moe_set_router(torch.from_numpy(make_router_weight(cfg).view(np.int16)).to(dev).view(torch.bfloat16))
        layer.nvfp4_moe_forward_routed(x, k, out)
        torch.cuda.synchronize()
        logits = layer.nvfp4_moe_debug_logits(T)
        fwd = lambda: layer.nvfp4_moe_forward_routed(x, k, out)
        n_ours += 1 if decode else 2
    else:
        fwd = lambda: layer.nvfp4_moe_forward(logits, x, k, out)
    ids, _, _, _ = layer.nvfp4_moe_debug_route(logits, T, k)
    distinct = int(torch.unique(ids).numel())

    for _ in range(warmup):
        fwd()
    torch.cuda.synchronize()
    st, _ = layer.nvfp4_moe_get_status()
    if st != 0:
        raise RuntimeError(f"{name}: device status {pkg.STATUS[st]} after warm-up")

    # one forward captured into a CUDA graph (launch-overhead free replay)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fwd()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()

    # --- timed region: graph replays, L2 flushed before each ---
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier()
    for s, e in evs:
        flush.zero_()
        s.record(stream)
        graph.replay()
        e.record(stream)
    barrier()
    step_ms = [s.elapsed_time(e) for s, e in evs]

    # --- per-kernel durations (direct calls, events inside the library on its stream) ---
    layer.nvfp4_moe_set_profiling(True)
    barrier()
    for _ in range(steps):
        flush.zero_()
        fwd()
    barrier()
    stage_ms, nfwd = layer.nvfp4_moe_get_stage_times()
    layer.nvfp4_moe_set_profiling(False)
    stage_ms = [v / max(nfwd, 1) for v in stage_ms]

    # --- end to end through the C ABI with host buffers ---
    # the inputs start in pinned host memory and the result ends there, every step.  On the
    # W4A16 decode path the library reads and writes those buffers in place
    # (nvfp4_moe_forward_host: no copy engine); every path is also timed with explicit
    # cudaMemcpyAsync copies around the device forward
    h_logits = torch.from_numpy(inp.logits).pin_memory()
    h_x = torch.from_numpy(inp.x_bits.view(np.int16)).pin_memory()
    h_out = torch.empty((T, H), dtype=torch.int16).pin_memory()
    d_x16 = x.view(torch.int16)
    in_place = decode and not (router or w4a4)

    def e2e_copies():
        if not router:
            logits.copy_(h_logits, non_blocking=True)
        d_x16.copy_(h_x, non_blocking=True)
        fwd()
        h_out.copy_(out.view(torch.int16), non_blocking=True)

    def e2e_host():
        layer.nvfp4_moe_forward_host(h_logits, h_x.view(torch.bfloat16), k, h_out.view(torch.bfloat16))

    def time_e2e(step):
        evs_ = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for _ in range(warmup):
            step()
        barrier()
        for s, e in evs_:
            flush.zero_()
            s.record(stream)
            step()
            e.record(stream)
        barrier()
        return [s.elapsed_time(e) for s, e in evs_]

    e2e_ms_copies = time_e2e(e2e_copies)
    e2e_ms = time_e2e(e2e_host) if in_place else e2e_ms_copies
    st, _ = layer.nvfp4_moe_get_status()
    if st != 0:
        raise RuntimeError(f"{name}: device status {pkg.STATUS[st]} after the timed region")
    layer.close()

    ms, ms_e2e, value, value_e2e = replica_throughput(statistics.mean(step_ms), statistics.mean(e2e_ms), T, ws, dev)
    _, ms_e2e_copies, _, value_e2e_copies = replica_throughput(statistics.mean(step_ms), statistics.mean(e2e_ms_copies),
                                                               T, ws, dev)
    layer_bytes = distinct * cfg.expert_bytes + T * H * 2 * 2 + T * E * 4
    layer_flops = 2.0 * T * (k + S) * 3 * H * I
    if decode:
        # decode: one kernel streams every touched expert's weights once (the W4A4 variant
        # runs on the earlier decode kernel)
        kernel = "decode_fused_kernel" if w4a4 else "decode_stream_kernel"
        kern_ms = stage_ms[1]
        algo = layer_bytes
        achieved = algo / (kern_ms / 1e3) / 1e9
        bound, unit = "hbm", "GB/s"
        peak, peak_src = _peak("hbm_gbs", 6800.0)
        traffic = _traffic_for(os.path.join(ROOT, "nvfp4_weight_only_w4a16_gb300", "csrc", "decode_stream.cu")) \
            if name == WORKLOAD and not (router or w4a4) else None
        stages = {kernel + " (route + gate/up + down + combine)": kern_ms}
    else:
        # prefill: the gate/up GEMM's dense flops on the tensor cores
        kernel = "prefill_gemm_kernel<gate/up>"
        kern_ms = stage_ms[1]
        algo = 2.0 * T * (k + S) * (2 * I) * H
        achieved = algo / (kern_ms / 1e3) / 1e12
        bound, unit = "tensor", "TFLOP/s"
        peak, peak_src = _peak("bf16_tflops", 1900.0)
        traffic = None
        stages = {"route_permute" + (" (+ router linear)" if router else ""): stage_ms[0],
                  "gate_up": stage_ms[1], "down": stage_ms[2], "combine": stage_ms[3]}
    return {
        "inp": inp, "ms": ms, "ms_e2e": ms_e2e, "value": value, "value_e2e": value_e2e,
        "distinct": distinct, "layer_bytes": layer_bytes, "layer_flops": layer_flops,
        "n_ours": n_ours, "stages": stages,
        "roofline": {"bound": bound, "kernel": kernel, "achieved": achieved, "peak": peak,
                     "peak_source": peak_src, "unit": unit, "frac": achieved / peak,
                     "algorithmic_per_launch": algo, "kernel_ms": kern_ms, "traffic": traffic},
        "e2e": {"value": value_e2e, "unit": "tokens/s",
                "h2d_bytes_per_step": (0 if router else T * E * 4) + T * H * 2,
                "d2h_bytes_per_step": T * H * 2,
                "transfer": ("in place: nvfp4_moe_forward_host reads the pinned inputs and writes the pinned "
                             "result over the CPU-GPU link" if in_place else
                             "cudaMemcpyAsync of the pinned inputs, nvfp4_moe_forward, cudaMemcpyAsync of the result"),
                "with_copy_engine": {"value": value_e2e_copies, "ms_per_step": ms_e2e_copies}},
    }


SECONDARY = ("decode_c16", "prefill_1k", "prefill_16k")


def run_ours(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import nvfp4_weight_only_w4a16_gb300 as pkg
    pkg.build()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.1)
    m = measure_layer(args.workload, args.steps, args.warmup, dev, flush, barrier, ws, args.router, args.w4a4)
    secondary = {}
    if args.workload == WORKLOAD and not (args.router or args.w4a4 or args.no_secondary):
        for name in SECONDARY:
            r = measure_layer(name, min(args.steps, 30), max(3, min(args.warmup, 5)), dev, flush, barrier, ws)
            secondary[name] = {
                "workload": _workload_desc(r["inp"].config), "distinct_experts": r["distinct"],
                "ms_per_step": r["ms"], "tokens_per_s": r["value"], "e2e_tokens_per_s": r["value_e2e"],
                "layer_weight_gbs": r["layer_bytes"] / (r["ms"] / 1e3) / 1e9,
                "layer_tflops": r["layer_flops"] / (r["ms"] / 1e3) / 1e12,
                "stage_ms": r["stages"], "roofline": r["roofline"], "gpu_launches_per_step": r["n_ours"],
            }
    clocks = sampler.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(m["inp"])

    if rank == 0:
        cfg = m["inp"].config
        line = {
            "metric": METRIC, "value": m["value"], "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": m["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "w4a16: e2m1*e4m3 weights -> fp16/bf16 mma, fp32 accumulate",
            "data": "synthetic (seeded PCG64, shapes of the pages' workloads)",
            "config": {"workload": _workload_desc(cfg) + (" + BF16 router linear" if args.router else "") +
                                   (" [W4A4 comparison variant: NVFP4 activations]" if args.w4a4 else ""),
                       "distinct_experts": m["distinct"],
                       "layer_weight_bytes_per_step": m["layer_bytes"],
                       "layer_weight_gbs": m["layer_bytes"] / (m["ms"] / 1e3) / 1e9,
                       "layer_tflops": m["layer_flops"] / (m["ms"] / 1e3) / 1e12,
                       "l2": "flushed before every step (256 MiB write, outside the step events)",
                       "launch": "CUDA graph replay of one " + (
                           "nvfp4_moe_forward_routed (router linear on the GPU)" if args.router else "nvfp4_moe_forward"),
                       "parallelism": f"replicas x{ws}",
                       "stage_ms": m["stages"],
                       "secondary": secondary},
            "roofline": m["roofline"],
            "e2e": m["e2e"],
            "gpu_launches": m["n_ours"] * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


# ---------------------------------------------------------------------------
# Dense W4A16 linear workloads (--workload kda_in_proj_mtp | kda_in_proj_1k | linear_tiny)
# ---------------------------------------------------------------------------

LINEAR_METRIC = "W4A16 NVFP4 dense linear tokens/s; decode weight GB/s & prefill TFLOP/s as % of GB300 roofline"

_LINEAR_ORACLE_CHILD = r"""
import sys, time, json, numpy as np
sys.path.insert(0, sys.argv[1])
import oracle
d = np.load(sys.argv[2])
reps = int(sys.argv[3])
times = []
for _ in range(reps):
    t0 = time.perf_counter(); oracle.linear_forward(d["x_bits"], d["w_q"], d["w_s"], float(d["g"])); times.append(time.perf_counter() - t0)
print(json.dumps({"times": times}))
"""


def _linear_desc(cfg):
    return (f"{cfg.name}: dense linear N{cfg.out_features} K{cfg.in_features} T{cfg.tokens}, NVFP4 "
            f"(E2M1 + E4M3/16 + FP32/tensor) weights, BF16 activations")


def _time_linear_oracle(inp, ns, reps):
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    np.savez(path, x_bits=inp.x_bits[:ns], w_q=inp.w_q, w_s=inp.w_s, g=np.float32(inp.gscale))
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[v] = "1"
    try:
        r = subprocess.run([sys.executable, "-c", _LINEAR_ORACLE_CHILD, ROOT, path, str(reps)],
                           capture_output=True, text=True, env=env)
    finally:
        os.unlink(path)
    if r.returncode != 0:
        raise RuntimeError("oracle timing failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])["times"]


def run_linear_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from synth import make_linear_inputs
    inp = make_linear_inputs(args.workload)
    cfg = inp.config
    times = _time_linear_oracle(inp, 1, args.warmup + args.steps)[args.warmup:]
    sec = sum(times)
    value = args.steps / sec   # one token per step
    line = {
        "impl": "reference", "metric": LINEAR_METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded PCG64, the pages' fused KDA in_proj shape)",
        "config": {"workload": _linear_desc(cfg)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "one token per step (dequantise W, one float64 GEMV), 1 thread"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_linear(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import nvfp4_weight_only_w4a16_gb300 as pkg
    from synth import make_linear_inputs
    pkg.build()
    inp = make_linear_inputs(args.workload)
    cfg = inp.config
    T, N, K = cfg.tokens, cfg.out_features, cfg.in_features
    lin = pkg.Linear(N, K, T, device=dev.index)
    lin.nvfp4_linear_pack(torch.from_numpy(inp.w_q).to(dev), torch.from_numpy(inp.w_s).to(dev),
                          torch.tensor([float(inp.gscale)], dtype=torch.float32, device=dev))
    decode = T <= 16
    n_ours = 1 if decode else 2     # the GEMV kernel / the tables kernel + the GEMM
    x = torch.from_numpy(inp.x_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        lin.nvfp4_linear_forward(x, out)
    torch.cuda.synchronize()
    st, _ = lin.nvfp4_moe_get_status()
    if st != 0:
        raise RuntimeError(f"device status {pkg.STATUS[st]} after warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        lin.nvfp4_linear_forward(x, out)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.1)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for s, e in evs:
        flush.zero_()
        s.record(stream)
        graph.replay()
        e.record(stream)
    barrier()
    step_ms = [s.elapsed_time(e) for s, e in evs]

    lin.nvfp4_moe_set_profiling(True)
    barrier()
    for _ in range(args.steps):
        flush.zero_()
        lin.nvfp4_linear_forward(x, out)
    barrier()
    stage_ms, nfwd = lin.nvfp4_moe_get_stage_times()
    lin.nvfp4_moe_set_profiling(False)

    h_x = torch.from_numpy(inp.x_bits.view(np.int16)).pin_memory()
    h_out = torch.empty((T, N), dtype=torch.int16).pin_memory()
    d_x16 = x.view(torch.int16)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for s, e in e2e_ev:
        flush.zero_()
        s.record(stream)
        d_x16.copy_(h_x, non_blocking=True)
        lin.nvfp4_linear_forward(x, out)
        h_out.copy_(out.view(torch.int16), non_blocking=True)
        e.record(stream)
    barrier()
    e2e_ms = [s.elapsed_time(e) for s, e in e2e_ev]
    clocks = sampler.stop()
    st, _ = lin.nvfp4_moe_get_status()
    if st != 0:
        raise RuntimeError(f"device status {pkg.STATUS[st]} after the timed region")

    ms, ms_e2e, value, value_e2e = replica_throughput(statistics.mean(step_ms), statistics.mean(e2e_ms), T, ws, dev)
    kern_ms = stage_ms[2] / max(nfwd, 1)   # the GEMV / GEMM launch (tables kernel excluded)
    wbytes = cfg.weight_bytes
    if decode:
        kernel, bound, unit, peak_key = "decode_stream_kernel (linear)", "hbm", "GB/s", "hbm_gbs"
        algo = wbytes + T * K * 2 + T * N * 2
        achieved = algo / (kern_ms / 1e3) / 1e9
    else:
        kernel, bound, unit, peak_key = "prefill_gemm_kernel<down> (linear)", "tensor", "TFLOP/s", "bf16_tflops"
        algo = 2.0 * T * N * K
        achieved = algo / (kern_ms / 1e3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)[peak_key])
        peak_src = "measured"
    except Exception:
        peak, peak_src = (6800.0 if bound == "hbm" else 1900.0), "fallback"

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        times = _time_linear_oracle(inp, 1, 2)
        cpu = {"value": 1 / statistics.mean(times), "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": "1 token of the step (dequantise W, one float64 GEMV), twice, 1 thread"}
    if rank == 0:
        line = {
            "metric": LINEAR_METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "w4a16: e2m1*e4m3 weights -> fp16/bf16 mma, fp32 accumulate",
            "data": "synthetic (seeded PCG64, the pages' fused KDA in_proj shape)",
            "config": {"workload": _linear_desc(cfg), "weight_bytes": wbytes,
                       "weight_gbs": wbytes / (ms / 1e3) / 1e9, "tflops": 2.0 * T * N * K / (ms / 1e3) / 1e12,
                       "kernel_ms": kern_ms,
                       "l2": "flushed before every step (256 MiB write, outside the step events)",
                       "launch": "CUDA graph replay of one nvfp4_linear_forward",
                       "parallelism": f"replicas x{ws}"},
            "roofline": {"bound": bound, "kernel": kernel, "achieved": achieved, "peak": peak,
                         "peak_source": peak_src, "unit": unit, "frac": achieved / peak,
                         "algorithmic_per_launch": algo, "traffic": None},
            "e2e": {"value": value_e2e, "unit": "tokens/s", "h2d_bytes_per_step": T * K * 2,
                    "d2h_bytes_per_step": T * N * 2},
            "gpu_launches": n_ours * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    lin.close()
    if ws > 1:
        torch.distributed.destroy_process_group()


def main():
    args = _args()
    from synth import LINEAR_CONFIGS
    linear = args.workload in LINEAR_CONFIGS
    if args.impl == "reference":
        (run_linear_reference if linear else run_reference)(args)
    else:
        (run_linear if linear else run_ours)(args)


if __name__ == "__main__":
    main()
