"""Benchmark of the W4A8 grouped-expert MoE prefill layer on GB300.

One step = one MoE FFN prefill layer through the C ABI (fge_moe_layer_forward: top-k gate,
permute with the per-(token, 128) e4m3 quantization folded into its row copy, gate_up
grouped GEMM with fused SwiGLU requant, down grouped GEMM, combine).  The headline workload
is the largest single-GPU one, the large skewed layer: T=16384 tokens, H=4096, 128 experts,
I=1536, top-8, Zipf(1.1)-biased routing (the hottest expert gets > 10x the mean rows, some
get none), int4 expert banks with 128-group fp32 scales, bf16 activations ~N(0,1) with 1%
of channels x20.

Beside the headline the line reports every other workload: the tiny and mid layers, the
dense per-tensor W8A8 projection at M = 16, 256, 2048, 8192 (N=6656, K=2560) and the stacked
prefill at depth 4, 8 and 12 (T=2048): each with tokens/s, TFLOPS and the fraction of its
roofline, max(flops / fp8 peak, bytes / HBM bandwidth) / time.  The HBM-bound kernels of
the headline layer (top-k, quantization, permute, combine) get their achieved GB/s.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead on a bounded
sample of the same workload.  Under torchrun (N > 1) every rank runs its own replica of the
workload (weak scaling, no collective on the data path); the step time is the max over
ranks.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "large"
METRIC = "MoE prefill tokens/s; grouped-GEMM TFLOPS as % of GB300 FP8 peak, 1 GPU"
L2_FLUSH_BYTES = 256 << 20

# DRAM bytes (read + write) of one gate_up grouped-GEMM launch, from an ncu capture, keyed
# by the workload and the hash of the kernel code it was taken on (_kernel_key: sources with
# comments removed).  A kernel changed since its capture reports traffic = null.
# large: 1410997504 read + 211325696 written (profiles/moe_layer_large_launch_list.md).
KNOWN_GATE_UP_TRAFFIC = {
    ("large", "code:89989aa6314a006d:c4c688e683c7b15a"): 1622.32e6,
}


def _strip_comments(src):
    """C++ source without // and /* */ comments and with blank runs collapsed, so that an
    edit to a comment does not change the key below (string literals in these files hold no
    comment markers)."""
    import re
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return re.sub(r"\s+", " ", src).strip()


def _kernel_key():
    """Hash of the grouped GEMM's code (its source and device header, comments removed): the
    DRAM traffic recorded from an ncu capture applies only while this key is unchanged."""
    import hashlib
    parts = []
    for f in ("gemm.cu", "fge_device.cuh"):
        with open(os.path.join(ROOT, "fp8_grouped_expert_gb300", "csrc", f), encoding="utf-8") as fh:
            parts.append(hashlib.sha256(_strip_comments(fh.read()).encode()).hexdigest()[:16])
    return "code:" + ":".join(parts)


def job_step_ms(local_ms, device=None):
    """Step time of the whole job: the max over ranks (the slowest replica sets the pace).
    Uses the default torch.distributed group when one is initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(local_ms)
    t = torch.tensor([float(local_ms)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_rank, world, step_ms):
    """Whole-job throughput: every rank processes its own tokens_per_rank per step."""
    return world * tokens_per_rank / (step_ms / 1e3)


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            mp = json.load(f)
        return float(mp["hbm_gbs"]), float(mp["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": smax or None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------- CPU oracle
# The timed oracle is the single-threaded C++ one (oracle/oracle_ref.cpp): one host core.
ORACLE_CORES = 1


def oracle_tokens_per_s(inp, sample_tokens, seconds, seed=0):
    """Time the single-threaded C++ CPU oracle on repeated samples of `sample_tokens` tokens
    (each a whole layer call: gate, quant, permute, both GEMMs, SwiGLU, combine) for
    ~`seconds`."""
    from oracle import native
    native.build()
    rng = np.random.default_rng(seed)
    done, t0 = 0, time.perf_counter()
    while True:
        rows = np.sort(rng.choice(inp.T, size=sample_tokens, replace=False))
        native.moe_layer_forward(inp.logits[rows], inp.x[rows], inp.k, inp.w_gu, inp.s_gu,
                                 inp.w_dn, inp.s_dn, inp.I, out_dtype=inp.out)
        done += sample_tokens
        el = time.perf_counter() - t0
        if el >= seconds:
            return done / el, done, el


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return 0
    from workloads import moe_inputs
    inp = moe_inputs(args.workload, seed=0)
    sample = 64 if inp.T <= 4096 else 16
    for _ in range(args.warmup):
        oracle_tokens_per_s(inp, sample, 0.0)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle_tokens_per_s(inp, sample, 0.0, seed=i + 1)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = sample / (ms / 1e3)
    cores = ORACLE_CORES
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": _config(inp, note="each step: the single-threaded float64 C++ CPU oracle on "
                                    "%d sampled tokens" % sample),
        "cpu_baseline": dict({"value": value, "unit": "tokens/s", "cores": cores,
                              "kind": "oracle",
                              "sample": "%d random tokens of the T=%d layer per step"
                                        % (sample, inp.T)}, **cpu_info()),
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def _config(inp, note=None):
    routing = (", Zipf(1.1)-skewed routing, 1% outlier channels x20" if inp.name == "large"
               else "")
    c = {"workload": "%s MoE layer prefill: T=%d tokens, H=%d, E=%d experts, I=%d, top-%d%s, "
                     "int4 experts, e4m3 activations"
                     % (inp.name, inp.T, inp.H, inp.E, inp.I, inp.k, routing),
         "T": inp.T, "H": inp.H, "E": inp.E, "I": inp.I, "k": inp.k,
         "global_batch": inp.T, "seq_len": inp.T, "parallelism": "replicas",
         "l2": "flushed (256 MB write) before every timed step; resident int4 banks + "
               "scales %.0f MB" % ((inp.w_gu.nbytes + inp.w_dn.nbytes + inp.s_gu.nbytes
                                   + inp.s_dn.nbytes) / 1e6)}
    if note:
        c["note"] = note
    return c


# ------------------------------------------------------------------------------ GPU arm
def run_gpu(args):
    import torch
    import fp8_grouped_expert_gb300 as fge
    from fp8_grouped_expert_gb300 import build as fge_build
    from workloads import moe_inputs

    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(fge.LIB_PATH):
        fge_build.build()
    if world > 1:
        dist.barrier()
    fge.lib()

    inp = moe_inputs(args.workload, seed=rank)
    x_host = torch.from_numpy(inp.x_bits.view(np.int16)).view(torch.bfloat16)
    lg_host = torch.from_numpy(inp.logits)
    x = x_host.to(dev)
    logits = lg_host.to(dev)
    fmt = fge.W4_SUBNORMAL
    canon = [torch.from_numpy(a).to(dev) for a in (inp.w_gu, inp.s_gu, inp.w_dn, inp.s_dn)]
    w_gu, s_gu = fge.w4_prepack(canon[0], canon[1], True, fmt)
    w_dn, s_dn = fge.w4_prepack(canon[2], canon[3], False, fmt)
    ws = fge.new_workspace(fge.workspace_bytes(fge.OP_MOE_LAYER, inp.T, inp.H, inp.I, inp.E,
                                               inp.k), dev)
    out = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        fge.moe_layer_forward(logits, x, inp.k, inp.I, w_gu, s_gu, w_dn, s_dn, fmt=fmt,
                              workspace=ws, out=out)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    # the layer call is stream-ordered with no host sync and shape-only branches, so it can
    # be captured once as a CUDA graph and replayed: the 8 kernels launch without host gaps
    run_step = step
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
        run_step = graph.replay
        for _ in range(max(args.warmup, 3)):
            run_step()
        torch.cuda.synchronize()
    fge.clear_device_status(ws)

    # ---- timed region: K steps, L2 flushed before each, device time by CUDA events
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            run_step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)
    status = fge.read_device_status(ws)
    if status != 0:
        raise RuntimeError("device status %d after the timed steps" % status)
    launches_per_step = 8   # topk, permute count/scan/rank, quantizing row copy, gate_up, down, combine
    ms = job_step_ms(ms, dev)
    value = job_value(inp.T, world, ms)

    # ---- per-stage breakdown and the dominant kernel (gate_up grouped GEMM) timed alone
    stages = stage_times(fge, torch, inp, x, logits, w_gu, s_gu, w_dn, s_dn, fmt, flush, dev,
                         args.steps)

    # ---- the combine folded into the down GEMM's epilogue (bit-identical output), timed
    #      the same way as a step, beside the plain layer
    fused_ms = timed_calls(torch, lambda: fge.moe_layer_forward(
        logits, x, inp.k, inp.I, w_gu, s_gu, w_dn, s_dn, fmt=fmt, workspace=ws, out=out,
        fused_combine=True), flush, stream, 3, max(3, args.steps))

    # ---- FP4 activations (E2M1 + a power-of-two scale per 32): the dispatch-buffer half of
    #      the E2M1 row, timed beside the e4m3 G128 quantization (not part of the step)
    mx_ms = mx_quant_time(fge, torch, x, flush, dev, args.steps)

    # ---- the per-token int4 dispatch that the grouped GEMM replaces (context, untimed)
    base_ms = None
    if not args.no_baseline:
        # launched the same way as the timed steps (a replayed CUDA graph unless --no-graph)
        dout = torch.empty((inp.T, inp.H), dtype=torch.bfloat16, device=dev)
        dws = fge.new_workspace(fge.workspace_bytes(fge.OP_DISPATCH_BASELINE, inp.T, inp.H,
                                                    inp.I, inp.E, inp.k), dev)

        def dispatch():
            fge.moe_layer_per_token_dispatch(logits, x, inp.k, inp.I, *canon, workspace=dws,
                                             out=dout)

        dispatch()
        torch.cuda.synchronize()
        run_dispatch = dispatch
        if not args.no_graph:
            dgraph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(dgraph):
                dispatch()
            run_dispatch = dgraph.replay
            run_dispatch()
            torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(2):
            run_dispatch()
        b1.record(stream)
        torch.cuda.synchronize()
        base_ms = b0.elapsed_time(b1) / 2

    # ---- end to end through the public API with host buffers: every step copies its
    #      inputs up from pinned memory and its output down; HostLayerPipeline overlaps
    #      those copies with the neighbouring steps' layers on two copy streams
    x_pin = x_host.pin_memory()
    lg_pin = lg_host.pin_memory()
    out_pin = torch.empty((inp.T, inp.H), dtype=torch.bfloat16).pin_memory()
    pipe = fge.HostLayerPipeline(inp.T, inp.H, inp.E, inp.k, inp.I, w_gu, s_gu, w_dn, s_dn,
                                 fmt=fmt, device=dev)
    for _ in range(2):
        pipe.submit(x_pin, lg_pin, out_pin)
    pipe.finish()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.up)
    for _ in range(args.steps):
        pipe.submit(x_pin, lg_pin, out_pin)
    e1.record(pipe.down)
    pipe.finish()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    h2d = x_pin.numel() * 2 + lg_pin.numel() * 4
    d2h = out_pin.numel() * 2

    hbm, bf16, peak_kind = _peaks()
    fp8_peak = 2.0 * bf16  # fp8 dense = 2x bf16 dense (nominal ratio 4.5 / 2.25 PFLOP/s)
    e2m1_gemm = e2m1_gemm_time(fge, torch, inp, x, logits, w_gu, s_gu, flush, dev,
                               max(3, args.steps), fp8_peak)
    r = inp.T * inp.k
    gu_flops = 2.0 * r * (2 * inp.I) * inp.H
    gu_ms = stages["gate_up_gemm"]
    achieved = gu_flops / (gu_ms / 1e3) / 1e12
    ids_dev, _ = fge.moe_topk_gate(logits, inp.k)
    counts = torch.bincount(ids_dev.flatten().long(), minlength=inp.E).cpu().numpy()
    layer_flops, layer_bytes = layer_work(inp, counts)
    layer_frac, layer_bound = roofline_frac(layer_flops, layer_bytes, ms, fp8_peak, hbm)

    # the HBM-bound stages of this layer against the measured copy bandwidth
    sb = stage_bytes(inp)
    wb = stage_write_bytes(inp)
    write_gbs = write_ceiling_gbs(torch, dev)
    memory_kernels = {name: {"ms": stages[name], "bytes": nbytes, "bytes_written": wb[name],
                             "hbm_gbs": nbytes / (stages[name] / 1e3) / 1e9,
                             "hbm_frac": nbytes / (stages[name] / 1e3) / 1e9 / hbm,
                             "floor_ms": memory_floor_ms(nbytes, wb[name], hbm, write_gbs),
                             "frac_of_floor": memory_floor_ms(nbytes, wb[name], hbm, write_gbs)
                                              / stages[name]}
                      for name, nbytes in sb.items()}
    memory_kernels["ceilings"] = {
        "copy_gbs": hbm, "write_gbs": write_gbs,
        "what": "hbm_frac: bytes / time against the measured copy bandwidth; frac_of_floor: "
                "max(bytes / copy bandwidth, bytes written / plain-write bandwidth) / time, "
                "the plain-write bandwidth measured here by a 1 GiB memset"}

    # every other workload, each on its own line of the object (rank 0 only)
    configs = None
    if rank == 0 and not args.no_extras:
        reps = max(5, min(args.steps, 20))
        configs = {}
        for name in ("tiny", "mid", "large"):
            if name != args.workload:
                configs[name] = layer_config(fge, torch, name, dev, flush, reps, fp8_peak, hbm)
        configs["dense_w8a8"] = dense_sweep(fge, torch, dev, flush, reps, fp8_peak, hbm)
        configs["stacked_prefill"] = stacked_depths(fge, torch, dev, flush, max(5, reps // 2),
                                                    fp8_peak, hbm)

    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        sample = 64 if inp.T <= 4096 else 16
        rate, done, el = oracle_tokens_per_s(inp, sample, args.cpu_seconds)
        cpu = dict({"value": rate, "unit": "tokens/s", "cores": ORACLE_CORES, "kind": "oracle",
                    "sample": "%d tokens (random %d-token samples of the T=%d layer, each a "
                              "whole layer call of the single-threaded float64 C++ oracle) "
                              "in %.1f s" % (done, sample, inp.T, el)}, **cpu_info())
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 x int4 -> f32 accumulate", "data": "synthetic",
        "config": dict(_config(inp), launch="direct stream launches" if args.no_graph
                       else "CUDA graph of the layer call, replayed per step"),
        "layer_tflops": layer_flops / (ms / 1e3) / 1e12,
        "layer_roofline": {"bound": layer_bound, "frac": layer_frac, "flops": layer_flops,
                           "bytes": layer_bytes,
                           "what": "max(flops / fp8 peak, irreducible bytes / HBM) / layer "
                                   "time; bytes = activations in + logits + output + the "
                                   "banks and scales of the experts that got rows"},
        "stages_ms": stages,
        "roofline": {"bound": "tensor", "kernel": "grouped_gemm gate_up (fused SwiGLU requant)",
                     "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                     "frac": achieved / fp8_peak,
                     "traffic": KNOWN_GATE_UP_TRAFFIC.get((inp.name, _kernel_key())),
                     "peak_source": "%s bf16 burst %.1f TF x 2 (fp8/bf16 nominal ratio)"
                                    % (peak_kind, bf16),
                     "algorithmic_flops_per_launch": gu_flops},
        "memory_kernels": memory_kernels,
        "configs": configs,
        "cpu_baseline": cpu,
        "e2e": {"value": world * inp.T / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": "pinned host -> device and back every step, overlapped with the "
                          "neighbouring steps' layers (HostLayerPipeline, two copy streams)"},
        "gpu_launches": launches_per_step * args.steps,
        "e2m1_gemm": e2m1_gemm,
        "e2m1_activations": {
            "quant_ms": mx_ms,
            "bytes_read": 2 * inp.T * inp.H,
            "bytes_written": inp.T * inp.H // 2 + inp.T * inp.H // 32,
            "hbm_gbs": (2 * inp.T * inp.H + inp.T * inp.H // 2 + inp.T * inp.H // 32)
                       / (mx_ms / 1e3) / 1e9,
            "hbm_frac": (2 * inp.T * inp.H + inp.T * inp.H // 2 + inp.T * inp.H // 32)
                        / (mx_ms / 1e3) / 1e9 / hbm,
            "e4m3_g128_quant_ms": stages["quant_g128"],
            "e4m3_g128_bytes_written": inp.T * inp.H + inp.T * inp.H // 128 * 4,
            "what": "fge_mx_quant_e2m1 on the layer's activations: E2M1 codes + E8M0 scale "
                    "per 32 values (dispatch bytes), against the e4m3 G128 quantization"},
        "fused_combine": {
            "ms_per_step": fused_ms, "plain_ms_per_step": ms,
            "what": "fge_moe_layer_forward_fused_combine: the k-th slot row of each (token, "
                    "128-column chunk) to leave the down GEMM sums the chunk in slot order "
                    "inside the epilogue (no combine kernel; bit-identical output)"},
        "per_token_dispatch_baseline": None if base_ms is None else {
            "ms_per_step": base_ms, "grouped_speedup": base_ms / ms,
            "what": "same layer, one CTA per routed token: int4 weights dequantized in "
                    "registers, fp32 activations, no grouped GEMM"},
        "clocks": clocks.summary(),
    }
    print(json.dumps(line))
    return 0


def mx_quant_time(fge, torch, x, flush, dev, steps):
    """FP4 (E2M1, MXFP4) quantization of the layer's activations through its C-ABI call,
    timed like a stage (L2 flushed before each call; first call dropped)."""
    stream = torch.cuda.current_stream(dev)
    times = []
    for i in range(steps + 1):
        flush.fill_(5)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fge.mx_quant_e2m1(x)
        b.record(stream)
        times.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in times[1:]) / steps


def e2m1_gemm_time(fge, torch, inp, x, logits, w_gu, s_gu, flush, dev, steps, fp8_peak):
    """The gate_up GEMM shape of the layer (R = T*k routed rows, N = 2I, K = H, plain bf16
    store) with MXFP4 activations (fge_grouped_gemm_mxf4_w4: E2M1 codes, a power-of-two scale
    per 32 values applied in the block-scaled MMA) beside the same GEMM with e4m3 G128
    activations (fge_grouped_gemm_w4a8), each through its C-ABI call, L2 flushed before each
    call.  The routed activations are prepared outside the timing."""
    stream = torch.cuda.current_stream(dev)
    ids, _ = fge.moe_topk_gate(logits, inp.k)
    xq, xs = fge.fp8_quant_act(x, "g128")
    p = fge.moe_permute(ids, inp.E, xq, xs)
    codes_t, scales_t = fge.mx_quant_e2m1(x)
    rt = p["row_token"].long()
    codes = codes_t.index_select(0, rt).contiguous()
    scales = scales_t.index_select(0, rt).contiguous()
    r = inp.T * inp.k
    n = 2 * inp.I
    ws = fge.new_workspace(fge.workspace_bytes(fge.OP_GROUPED_GEMM), dev)
    y = torch.empty((r, n), dtype=torch.bfloat16, device=dev)
    calls = {
        "e4m3_g128": lambda: fge.grouped_gemm_w4a8(p["aq"], p["as_"], p["offsets"], w_gu, s_gu,
                                                   out_dtype=torch.bfloat16, workspace=ws,
                                                   out=y),
        "mxfp4": lambda: fge.grouped_gemm_mxf4_w4(codes, scales, p["offsets"], w_gu, s_gu,
                                                  out_dtype=torch.bfloat16, workspace=ws, out=y),
    }
    res = {}
    flops = 2.0 * r * n * inp.H
    for name, fn in calls.items():
        fn()
        torch.cuda.synchronize()
        times = []
        for i in range(steps):
            flush.fill_(9)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            times.append((a, b))
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in times) / steps
        res[name] = {"ms": ms, "tflops": flops / (ms / 1e3) / 1e12,
                     "frac_of_fp8_peak": flops / (ms / 1e3) / 1e12 / fp8_peak}
    if fge.read_device_status(ws) != 0:
        raise RuntimeError("device status %d in the E2M1 GEMM timing" % fge.read_device_status(ws))
    res["activation_bytes"] = {"e4m3_g128": r * inp.H + r * (inp.H // 128) * 4,
                               "mxfp4": r * inp.H // 2 + r * (inp.H // 32)}
    res["shape"] = {"R": r, "N": n, "K": inp.H, "E": inp.E}
    return res


def stage_times(fge, torch, inp, x, logits, w_gu, s_gu, w_dn, s_dn, fmt, flush, dev, steps):
    """Each stage of the layer through its own C-ABI call, timed with CUDA events on the
    launching stream, L2 flushed before each stage.  'permute_quant' is the layer's own
    routing stage (histogram, scan, rank and the row copy that quantizes); 'quant_g128' and
    'permute' are the same work as two separate calls."""
    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    acc = {}

    def timed(name, fn):
        flush.fill_(7)
        a, b = ev(), ev()
        a.record(stream)
        res = fn()
        b.record(stream)
        acc.setdefault(name, []).append((a, b))
        return res

    # the GEMMs write into buffers allocated here, so that each GEMM stage times the kernel
    # alone (no zero fill of its output inside the timed region)
    r = inp.T * inp.k
    ws = fge.new_workspace(fge.workspace_bytes(fge.OP_GROUPED_GEMM), dev)
    hq = torch.empty((r, inp.I), dtype=torch.uint8, device=dev)
    hs = torch.empty((r, inp.I // 128), dtype=torch.float32, device=dev)
    y = torch.empty((r, inp.H), dtype=torch.bfloat16, device=dev)
    cws = ws if (inp.H % 2048 == 0 and inp.k <= 8) else None
    for _ in range(steps + 1):
        ids, gates = timed("topk_gate", lambda: fge.moe_topk_gate(logits, inp.k))
        xq, xs = timed("quant_g128", lambda: fge.fp8_quant_act(x, "g128"))
        timed("permute", lambda: fge.moe_permute(ids, inp.E, xq, xs))
        p = timed("permute_quant", lambda: fge.moe_permute_quant(ids, inp.E, x))
        timed("gate_up_gemm", lambda: fge.grouped_gemm_w4a8(
            p["aq"], p["as_"], p["offsets"], w_gu, s_gu, fmt=fmt, epilogue="swiglu",
            workspace=ws, out=hq, scales=hs))
        timed("down_gemm", lambda: fge.grouped_gemm_w4a8(
            hq, hs, p["offsets"], w_dn, s_dn, fmt=fmt, out_dtype=torch.bfloat16, workspace=ws,
            out=y))
        # the layer's own combine (slot rows staged by bulk copies) where it applies
        timed("combine", lambda: fge.moe_combine(y, p["token_row"], gates, workspace=cws))
    torch.cuda.synchronize()
    # the first pass includes allocator warm-up; drop it
    return {k: sum(a.elapsed_time(b) for a, b in v[1:]) / (len(v) - 1) for k, v in acc.items()}


def stage_bytes(inp):
    """Algorithmic HBM bytes of the memory-bound stages (each tensor read or written once):
    what each stage must move, not what it happens to move."""
    t, h, e, k = inp.T, inp.H, inp.E, inp.k
    r = t * k
    g = h // 128
    return {
        # logits in; ids and gates out
        "topk_gate": t * e * 4 + r * 8,
        # bf16 in; codes and one scale per 128 out
        "quant_g128": t * h * 2 + t * h + t * g * 4,
        # ids read (histogram and rank), codes and scales read once, written k times; the
        # row and token index maps written
        "permute": 2 * r * 4 + t * h + t * g * 4 + r * h + r * g * 4 + 2 * r * 4,
        # the layer's routing stage: bf16 rows read once, codes and scales written k times
        "permute_quant": 2 * r * 4 + t * h * 2 + r * h + r * g * 4 + 2 * r * 4,
        # expert outputs (bf16) read once with their gates and row map; bf16 out
        "combine": r * h * 2 + r * 8 + t * h * 2,
    }


def stage_write_bytes(inp):
    """The written part of stage_bytes: HBM writes are slower than reads on this part (a
    plain write stream, cudaMemset, reaches well under the copy bandwidth), so a stage that
    mostly writes has a lower ceiling than the copy figure suggests."""
    t, h, e, k = inp.T, inp.H, inp.E, inp.k
    r = t * k
    g = h // 128
    return {
        "topk_gate": r * 8,
        "quant_g128": t * h + t * g * 4,
        "permute": r * h + r * g * 4 + 2 * r * 4,
        "permute_quant": r * h + r * g * 4 + 2 * r * 4,
        "combine": t * h * 2,
    }


def memory_floor_ms(total_bytes, written_bytes, copy_gbs, write_gbs):
    """Shortest time the bytes allow: the copy bandwidth bounds all traffic, the plain-write
    bandwidth bounds the writes."""
    return max(total_bytes / copy_gbs, written_bytes / write_gbs) / 1e6


def write_ceiling_gbs(torch, dev, nbytes=1 << 30, reps=5):
    """Plain write bandwidth: a memset of a buffer far larger than L2, median of reps."""
    buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    buf.zero_()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        buf.zero_()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = sorted(a.elapsed_time(b) for a, b in ts)[reps // 2]
    del buf
    return nbytes / (ms / 1e3) / 1e9


def layer_work(inp, counts):
    """(flops, irreducible HBM bytes) of one MoE layer call: the two grouped GEMMs' flops,
    and the bytes no implementation can avoid -- activations in, logits in, output out,
    and the int4 banks and scales of every expert that received a row."""
    r = inp.T * inp.k
    flops = 2.0 * r * (2 * inp.I) * inp.H + 2.0 * r * inp.H * inp.I
    active = int((np.asarray(counts) > 0).sum())
    bank = (2 * inp.I * inp.H // 2 + inp.H * inp.I // 2            # int4 bytes
            + (2 * inp.I * (inp.H // 128) + inp.H * (inp.I // 128)) * 4)  # scales
    nbytes = inp.T * inp.H * 2 * 2 + inp.T * inp.E * 4 + active * bank
    return flops, nbytes


def roofline_frac(flops, nbytes, ms, fp8_peak_tf, hbm_gbs):
    """Fraction of the roofline: the slower of flops at the fp8 peak and bytes at the HBM
    bandwidth, over the measured time."""
    t_floor = max(flops / (fp8_peak_tf * 1e12), nbytes / (hbm_gbs * 1e9))
    return t_floor / (ms / 1e3), ("tensor" if flops / (fp8_peak_tf * 1e12)
                                  >= nbytes / (hbm_gbs * 1e9) else "hbm")


def timed_calls(torch, fn, flush, stream, warm, reps, graph=True):
    """Median device time (ms) of fn() over reps calls, L2 flushed before each; fn is
    captured once as a CUDA graph and replayed unless graph=False."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    run = fn
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        run = g.replay
        run()
        torch.cuda.synchronize()
    evs = []
    for i in range(reps):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    ts = sorted(a.elapsed_time(b) for a, b in evs)
    return ts[len(ts) // 2]


def layer_config(fge, torch, name, dev, flush, reps, fp8_peak, hbm):
    """One MoE layer workload timed like the headline (graph replay, L2 flushed)."""
    from workloads import moe_inputs
    inp = moe_inputs(name, seed=0)
    x = torch.from_numpy(inp.x_bits.view(np.int16)).view(torch.bfloat16).to(dev)
    logits = torch.from_numpy(inp.logits).to(dev)
    fmt = fge.W4_SUBNORMAL
    w_gu, s_gu = fge.w4_prepack(torch.from_numpy(inp.w_gu).to(dev),
                                torch.from_numpy(inp.s_gu).to(dev), True, fmt)
    w_dn, s_dn = fge.w4_prepack(torch.from_numpy(inp.w_dn).to(dev),
                                torch.from_numpy(inp.s_dn).to(dev), False, fmt)
    od = torch.float32 if inp.out == "f32" else torch.bfloat16
    ws = fge.new_workspace(fge.workspace_bytes(fge.OP_MOE_LAYER, inp.T, inp.H, inp.I, inp.E,
                                               inp.k), dev)
    out = torch.empty((inp.T, inp.H), dtype=od, device=dev)
    ms = timed_calls(torch, lambda: fge.moe_layer_forward(logits, x, inp.k, inp.I, w_gu, s_gu,
                                                         w_dn, s_dn, fmt=fmt, out_dtype=od,
                                                         workspace=ws, out=out),
                     flush, torch.cuda.current_stream(dev), 3, reps)
    ids, _ = fge.moe_topk_gate(logits, inp.k)
    counts = torch.bincount(ids.flatten().long(), minlength=inp.E).cpu().numpy()
    flops, nbytes = layer_work(inp, counts)
    frac, bound = roofline_frac(flops, nbytes, ms, fp8_peak, hbm)
    return {"workload": "%s MoE layer: T=%d, H=%d, E=%d, I=%d, top-%d" % (
                name, inp.T, inp.H, inp.E, inp.I, inp.k),
            "ms": ms, "tokens_per_s": inp.T / (ms / 1e3), "tflops": flops / (ms / 1e3) / 1e12,
            "roofline": {"bound": bound, "frac": frac, "flops": flops, "bytes": nbytes}}


def dense_sweep(fge, torch, dev, flush, reps, fp8_peak, hbm, copies=16):
    """Dense per-tensor W8A8 projection (N=6656, K=2560): quantization + GEMM through
    fge_linear_w8a8 at each M, with the weights coming from HBM.

    M = 2048, 8192: one call per timed replay, L2 flushed before each.  M = 16, 256 (a few
    microseconds a call, below what one event pair resolves well): a CUDA graph of `copies`
    calls, each on its own copy of the weights (16 x 17 MB, more than L2 holds, so every
    call reads its weights from HBM, as consecutive projections of a model do), timed as
    one replay and divided by the call count -- the weight rotation the dense-projection
    page uses past its GPU's L2."""
    gen = torch.Generator(device=dev).manual_seed(1)
    n, k = 6656, 2560
    stream = torch.cuda.current_stream(dev)
    banks = []
    for _ in range(copies):
        w = (torch.randn((n, k), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
        banks.append(fge.fp8_quant_act(w, "tensor"))
        del w
    res = {}
    for m in (16, 256, 2048, 8192):
        x = torch.randn((m, k), generator=gen, device=dev).to(torch.bfloat16)
        ws = fge.new_workspace(fge.workspace_bytes(fge.OP_LINEAR_W8A8, m, k, n), dev)
        y = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        if m <= 256:
            def calls():
                for wq, sw in banks:
                    fge.linear_w8a8(x, wq, sw, workspace=ws, out=y)
            for _ in range(3):
                calls()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                calls()
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                g.replay()
                b.record(stream)
                ts.append((a, b))
            torch.cuda.synchronize()
            ms = sorted(a.elapsed_time(b) for a, b in ts)[len(ts) // 2] / copies
            method = "%d calls per graph replay, each on its own weight copy (%d MB > L2)" % (
                copies, copies * n * k // (1 << 20))
        else:
            wq, sw = banks[0]
            ms = timed_calls(torch, lambda: fge.linear_w8a8(x, wq, sw, workspace=ws, out=y),
                             flush, stream, 3, reps)
            method = "one call per replay, L2 flushed before each"
        flops = 2.0 * m * n * k
        nbytes = n * k + 2 * m * k + 2 * m * n
        frac, bound = roofline_frac(flops, nbytes, ms, fp8_peak, hbm)
        res["M=%d" % m] = {"ms": ms, "tokens_per_s": m / (ms / 1e3),
                           "tflops": flops / (ms / 1e3) / 1e12,
                           "hbm_gbs": nbytes / (ms / 1e3) / 1e9, "timing": method,
                           "roofline": {"bound": bound, "frac": frac, "flops": flops,
                                        "bytes": nbytes}}
    return res


def stacked_layers_on_device(torch, dev, L, H=2048, E=64, I=768, q=2048, kv=512, seed=0):
    """Weights of an L-layer stack drawn on the device from a seeded generator, the stacked
    workload's recipe: bf16 q/k/v/o projections ~N(0, 0.02), fp32 router ~N(0, 0.02), and int4
    expert banks from N(0, 0.02) draws with s = absmax/7 per (row, 128) and q = clamp(round(w /
    s), -8, 7) packed two per byte (even element in the low nibble)."""
    gen = torch.Generator(device=dev).manual_seed(seed)

    def int4_bank(e, n, kk):
        w = torch.randn((e, n, kk // 128, 128), generator=gen, device=dev) * 0.02
        s = (w.abs().amax(dim=3) / 7.0).float()
        s = torch.where(s == 0, torch.ones_like(s), s)
        qv = torch.clamp(torch.round(w / s[..., None]), -8, 7).to(torch.int32).reshape(e, n, kk)
        lo = qv[..., 0::2] & 0xF
        hi = qv[..., 1::2] & 0xF
        return (lo | (hi << 4)).to(torch.uint8).contiguous(), s.contiguous()

    layers = []
    for _ in range(L):
        d = {}
        for name, rows in (("q", q), ("k", kv), ("v", kv), ("o", H)):
            d["w" + name] = (torch.randn((rows, H), generator=gen, device=dev) * 0.02
                             ).to(torch.bfloat16)
        d["w_router"] = torch.randn((E, H), generator=gen, device=dev) * 0.02
        d["w_gu"], d["s_gu"] = int4_bank(E, 2 * I, H)
        d["w_dn"], d["s_dn"] = int4_bank(E, H, I)
        layers.append(d)
    return layers


def stacked_depths(fge, torch, dev, flush, reps, fp8_peak, hbm):
    """The stacked prefill (T=2048, H=2048, 16 query / 4 kv heads, MoE 64 x 768 top-8) timed
    over 4, 8 and 12 layers, each depth captured as one CUDA graph."""
    T, H, E, I, k = 2048, 2048, 64, 768, 8
    layers = stacked_layers_on_device(torch, dev, 12)
    model = fge.StackedPrefill(layers, T, H, E, I, k, 16, 4, dev)
    del layers
    gen = torch.Generator(device=dev).manual_seed(2)
    h0 = torch.randn((T, H), generator=gen, device=dev)
    h = h0.clone()
    per_layer_flops = (2.0 * T * H * (2048 + 512 + 512) + 2.0 * T * 2048 * H    # q, k, v, o
                       + 2.0 * T * E * H                                        # router
                       + 2.0 * T * k * (2 * I * H + H * I))                     # experts
    per_layer_bytes = ((2048 + 512 + 512 + 2048) * H                            # e4m3 weights
                       + E * (2 * I * H // 2 + H * I // 2
                              + (2 * I * (H // 128) + H * (I // 128)) * 4)      # int4 banks
                       + E * H * 4)                                             # router
    res = {}
    for L in (4, 8, 12):
        def run():
            h.copy_(h0)
            model.forward(h, layers=range(L))
        ms = timed_calls(torch, run, flush, torch.cuda.current_stream(dev), 2, reps)
        flops = L * per_layer_flops
        nbytes = L * per_layer_bytes + T * H * 4 * 2
        frac, bound = roofline_frac(flops, nbytes, ms, fp8_peak, hbm)
        res["L=%d" % L] = {"ms": ms, "tokens_per_s": T / (ms / 1e3),
                           "tflops": flops / (ms / 1e3) / 1e12,
                           "roofline": {"bound": bound, "frac": frac, "flops": flops,
                                        "bytes": nbytes}}
    return res


def cpu_info():
    """The host CPU's model name and the number of cores the OS offers."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith(("model name", "cpu part")):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"cpu_model": model, "machine": platform.machine(), "nproc": os.cpu_count()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, choices=["mid", "large", "tiny"],
                    help="MoE layer workload of the headline (default: large)")
    ap.add_argument("--no-extras", action="store_true",
                    help="headline only: skip the other workloads' lines")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the timed layer calls directly instead of replaying a CUDA graph")
    ap.add_argument("--no-baseline", action="store_true",
                    help="skip the per-token int4 dispatch comparison")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
