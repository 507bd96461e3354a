#!/usr/bin/env python3
"""Benchmark of the W4A8 block-64 prefill linear on GB300 (one JSON line on rank 0).

A step is one pass of the whole hot path over one batch: for every linear of the
workload, the fused call w4a8_prefill_linear (activation pre-pass + tensor-core
contraction + epilogue), inputs resident in HBM.  L2 is flushed (256 MiB written, then read back)
before every timed step, outside the timed events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c1] [--impl ours|reference]

Multi-GPU runs are replicas: each rank runs the whole workload on its own GPU with no
data exchange (weak scaling); value = units of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "W4A8 block64 prefill linear: effective TOPS & tok/s at M=512; % of INT8 peak"
DECODE_METRIC = "W4A8 block64 decode linear: tokens/s at M=1 (weights streamed at 4.5 bits each); % of HBM"
L2_FLUSH_BYTES = 256 << 20
WIDE_M = 4096   # from this many tokens on the contraction runs 256-token tiles from weight records
# The other INT8 denominator: the integer tensor path sm_103a still has, the legacy warp-level
# mma.sync.m16n8k32.s8.s8.s32, measured on a GB300 of this kind by a standalone probe (608 CTAs
# x 8 warps, 8 independent accumulators per warp, SM clock 2070 MHz).  tcgen05 has no integer
# kind on sm_103a, so this is the only "INT8 tensor peak" the part offers.
MMA_SYNC_S8_TOPS = 158.2
MMA_SYNC_S8_SOURCE = "measured: mma.sync.m16n8k32.s8 probe on GB300 (608 CTAs x 8 warps, 8 accumulators per warp)"


def prepass_bytes(M: int, K: int) -> int:
    """Algorithmic bytes of one activation pre-pass: x read (4 B per element); the int8 codes
    (1 B), the int32 block row sums (4 B per 64 elements) and the row's scale written --
    M*K*(4 + 1 + 4/64) + 8*M."""
    return M * K * 4 + M * K + M * (K // 64) * 4 + 8 * M


def record_prepass_bytes(M: int, K: int) -> int:
    """Bytes the fused call's pre-pass actually moves in its tensor-core record format: x read,
    two e4m3 nibble planes (2 B per element), one 16-byte zero-point operand entry per 64
    elements and the scale written."""
    return M * K * 4 + M * K * 2 + M * (K // 64) * 16 + 4 * M


def fused_step_bytes(M: int, K: int, N: int, bias: bool):
    """Bytes of one fused prefill call (w4a8_prefill_linear) two ways.
    algorithmic: x read, the packed u4 weights and their fp16 scales and zeros read, bias read,
    y written, each once.
    as designed: what the call moves through its tensor-core records, each written once and read
    back once (re-reads served by L2 not counted): the pre-pass reads x and writes the token
    records (two e4m3 planes, 16-byte zero-point entries, s_a); its weight job reads the packed
    weights, scales and zeros and writes the weight records (1 B per weight, 16-byte zero-point
    entries per 64, rows padded to 128) and the fp32 scales; the contraction reads all of those
    records and the bias and writes y."""
    nb = K // 64
    n_pad = (N + 127) // 128 * 128
    packed = N * K // 2 + 2 * 2 * N * nb
    algorithmic = 4 * M * K + packed + (4 * N if bias else 0) + 4 * M * N
    tok_rec = M * K * 2 + M * nb * 16 + 4 * M
    w_rec = n_pad * K + n_pad * nb * 16 + n_pad * nb * 4
    designed = (4 * M * K + tok_rec) + (packed + w_rec) + (tok_rec + w_rec + (4 * N if bias else 0) + 4 * M * N)
    return algorithmic, designed


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default="c1", choices=["c0", "c1", "c2", "c3", "c4", "d1", "d3", "d4"])
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle sample")
    p.add_argument("--shape", default=None,
                   help="M,K,N: one linear of this shape instead of the workload (profiling aid)")
    p.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi clocks")
    p.add_argument("--profile", action="store_true",
                   help="only the warm-up and timed fused steps (for ncu captures); prints a short line")
    p.add_argument("--no-targets", action="store_true",
                   help="skip the 7B-class kernel measurements of the targets object")
    return p.parse_args(argv)


# ------------------------------------------------------------------ distributed (replicas)
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value: float, world: int, device) -> float:
    """Max over ranks (the timed region's slowest rank)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.proc = None
        self.lines = []
        self.enabled = enabled
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = str(device_index)
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "50", "-i", ident]

    def __enter__(self):
        if not self.enabled:
            return self
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Median SM clock and the throttle reasons seen in [t0, t1] (wall clock); when the
        window holds fewer than 3 samples, every sample taken after the sampler started."""
        lines = [ln for t, ln in self.lines if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
        if len(lines) < 3:
            lines = [ln for _, ln in self.lines]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ ncu traffic record
def sources_sha256(paths):
    """sha256 over the listed source files' bytes, concatenated in order (the kernel's .cu
    file and every in-tree header it includes)."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the workload's dominant kernel from the
    committed ncu capture, or None when there is none or any source file of that kernel (its
    .cu file or an in-tree header it includes) changed since it was taken."""
    rec = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(rec):
        return None
    with open(rec) as f:
        e = json.load(f).get(workload)
    if not e or not e.get("sources"):
        return None
    if not all(os.path.isfile(os.path.join(ROOT, p)) for p in e["sources"]):
        return None
    if sources_sha256(e["sources"]) != e.get("sha256"):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ peaks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ workload
def workload_config(key, title, specs, world):
    """The `config` object of a bench line (the same for both arms)."""
    return {"workload": f"{key}: {title}",
            "linears": [{"name": s.name, "M": s.M, "K": s.K, "N": s.N, "bias": s.bias} for s in specs],
            "tokens_per_step": specs[0].M, "ops_per_step": sum(s.ops for s in specs),
            "l2": "flushed before every timed step (256 MiB written, then read back; outside the timed events)",
            "parallelism": f"replicas x{world}"}


def load_workload(key, device, shape=None):
    from w4a8_block_quantized_gb300 import binding, synth
    if shape:
        M, K, N = (int(v) for v in shape.split(","))
        title, specs = f"custom M{M} K{K} N{N}", (synth.LinearSpec("custom", M, K, N),)
    else:
        title, specs = synth.workload(key)
    lin = []
    for spec in specs:
        d = synth.make_linear(spec)
        t = {k: (torch.from_numpy(v).to(device) if isinstance(v, np.ndarray) else v) for k, v in d.items()}
        t["ws"] = binding.workspace(binding.prefill_workspace_bytes(spec.M, spec.N, spec.K), device)
        t["y"] = torch.empty((spec.M, spec.N), dtype=torch.float32, device=device)
        t["spec"] = spec
        t["host"] = d
        lin.append(t)
    return title, specs, lin


def run_bench(args):
    from w4a8_block_quantized_gb300 import binding
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    binding.load()
    title, specs, lin = load_workload(args.workload, device, args.shape)
    M = specs[0].M
    ops_per_step = sum(s.ops for s in specs)
    stream = torch.cuda.current_stream(device)
    flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    flush_sink = torch.zeros((), dtype=torch.float32, device=device)

    class _Flush:
        @staticmethod
        def zero_():
            # write a buffer twice the size of L2, then read it back: the read evicts the
            # written lines, so their write-back to HBM happens here and not inside the
            # next timed kernel
            flush_buf.zero_()
            torch.sum(flush_buf.view(torch.float32), dim=0, out=flush_sink)

    flush = _Flush()

    decode = M <= 8
    # a decode step runs its linears as one batch call: every few-token kernel after the first
    # streams its weights while the previous one is still running
    batch = binding.Batch([dict(x=t["x"], wq=t["wq"], s_w=t["s_w"], z_w=t["z_w"], bias=t["bias"], y=t["y"],
                                ws=t["ws"]) for t in lin], stream) if decode else None

    def step_on(s):
        if batch is not None:
            batch.run(s)
            return
        for t in lin:
            binding.prefill_linear(t["x"], t["wq"], t["s_w"], t["z_w"], t["bias"], y=t["y"], ws=t["ws"],
                                   stream=s)

    def step():
        step_on(stream)

    # the kernels one step launches, counted from a command tape of one step (its kernel nodes)
    side = torch.cuda.Stream(device=device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step_on(side)                    # one ordinary step before recording
        with binding.Tape(side) as tape:
            step_on(side)
    side.synchronize()
    kernels_per_step = tape.kernels()
    tape.free()

    # The clock sampler starts before the warm-up so that nvidia-smi's own start-up (which
    # can stall a fresh box for seconds) never falls inside the timed region.
    clk = ClockSampler(local, enabled=not args.no_clocks).__enter__()
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(device)
    if binding.sync_status(stream) != 0:
        raise RuntimeError("device status reported a timeout during warm-up")

    # ---------------- timed region: K fused steps, L2 flushed before each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    dist_barrier(world)
    torch.cuda.synchronize(device)
    t_start = time.time()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    t_end = time.time()
    dist_barrier(world)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_s = reduce_max(sum(step_ms) / 1e3, world, device)
    if binding.sync_status(stream) != 0:
        raise RuntimeError("device status reported a timeout in the timed region")
    ms_per_step = total_s * 1e3 / args.steps
    value_tops = whole_job_rate(ops_per_step * args.steps, world, total_s) / 1e12
    tok_s = whole_job_rate(M * args.steps, world, total_s)
    if args.profile:
        clk.__exit__(None, None, None)
        if rank == 0:
            print(json.dumps({"profile": title, "ms_per_step": ms_per_step, "tops": value_tops,
                              "status": binding.sync_status(stream),
                              "step_ms": [round(v, 4) for v in step_ms[:20]]}), flush=True)
        return

    # ---------------- kernel-level timing (same stream, CUDA events), each after an L2
    # flush: the pre-pass alone, then the contraction alone -- through the split calls
    # (prepared operands, tensor-core GEMM) or, for the few-token form, quant_pack +
    # w4a8_linear (the weight-streaming kernel).
    from w4a8_block_quantized_gb300 import synth
    assert decode == (M <= synth.DECODE_MAX_M)
    # few tokens of moderate depth: the fused call is one launch (the kernel quantizes)
    one_launch = decode and all(binding.prefill_workspace_bytes(s.M, s.N, s.K) == 0 for s in specs)
    gemm_ms, prep_ms = [], []
    prepared = []
    for t in lin:
        s = t["spec"]
        if one_launch:
            prepared.append(None)
        elif decode:
            prepared.append(binding.quant_pack(t["x"], stream=stream) +
                            (binding.workspace(0, device),))
        else:
            act = binding.prepare_activations(t["x"], stream=stream)
            pw = binding.prepare_weights(t["wq"], t["s_w"], t["z_w"], stream=stream)
            prepared.append((act, pw))
    # a decode step that is one few-token launch over all its linears: that launch is the
    # kernel timed, on the step's own batch call
    step_launch = one_launch and batch is not None and kernels_per_step == 1 and len(lin) > 1
    n_launch = 1 if step_launch else len(lin)
    kreps = max(20, min(args.steps, 200))
    for _ in range(kreps):
        if step_launch:
            e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            flush.zero_()
            e1.record(stream)
            batch.run(stream)
            e2.record(stream)
            e2.synchronize()
            gemm_ms.append(e1.elapsed_time(e2))
            prep_ms.append(0.0)
            continue
        g_ms = p_ms = 0.0
        for t, pre in zip(lin, prepared):
            s = t["spec"]
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            flush.zero_()
            e0.record(stream)
            if one_launch:
                e1.record(stream)
                binding.prefill_linear(t["x"], t["wq"], t["s_w"], t["z_w"], t["bias"], y=t["y"], ws=t["ws"],
                                       stream=stream)
            elif decode:
                a_q, s_a, rs, ws0 = pre
                binding.quant_pack(t["x"], a_q=a_q, a_scale=s_a, rowsum=rs, stream=stream)
                e1.record(stream)
                binding.linear(a_q, s_a, rs, t["wq"], t["s_w"], t["z_w"], t["bias"], y=t["y"], ws=ws0,
                               stream=stream)
            else:
                act, pw = pre
                binding.prepare_activations(t["x"], act=act, stream=stream)
                e1.record(stream)
                binding.linear_prepared(act, pw, s.M, s.N, s.K, bias=t["bias"], y=t["y"], stream=stream)
            e2.record(stream)
            e2.synchronize()
            p_ms += e0.elapsed_time(e1)
            g_ms += e1.elapsed_time(e2)
        gemm_ms.append(g_ms)
        prep_ms.append(p_ms)
    gemm_avg = statistics.fmean(gemm_ms) / n_launch   # per launch
    prep_avg = statistics.fmean(prep_ms) / len(lin)

    hbm_gbs, bf16_tf, peak_src = measured_peaks()
    # Contraction peak in effective int8-equivalent ops: fp8 = 2x bf16 (nominal ratio),
    # and each int8 x u4 MAC costs two e4m3 MACs (the two nibble planes).
    tensor_peak = bf16_tf * 2.0 / 2.0
    gemm_ops = ops_per_step / n_launch
    gemm_tops = gemm_ops / (gemm_avg * 1e-3) / 1e12
    if decode:
        # x read; a_q, s_a and the int32 row sums written (API layout)
        prep_bytes = sum(prepass_bytes(s.M, s.K) for s in specs) / len(lin)
        # packed weights + s_w + z_w, the activations (x when the kernel quantizes, else the
        # codes, row sums and scales), bias and y
        gemv_bytes = sum(synth.weight_bytes(s) + (4 * s.M * s.K if one_launch else
                                                  s.M * s.K + s.M * (s.K // 64) * 4 + s.M * 4) +
                         (4 * s.N if s.bias else 0) + 4 * s.M * s.N for s in specs) / n_launch
        gemv_gbs = gemv_bytes / (gemm_avg * 1e-3) / 1e9
    else:
        # the algorithmic bytes of the step (int8 codes, int32 row sums); the record format's own
        # bytes (two e4m3 planes, 16-byte zero-point entries) ride along as a second reading
        prep_bytes = sum(prepass_bytes(s.M, s.K) for s in specs) / len(lin)
        prep_fmt_bytes = sum(record_prepass_bytes(s.M, s.K) for s in specs) / len(lin)
    # (reported only where the pre-pass is a launch of its own; a quantizing few-token launch has none)
    prep_gbs = prep_bytes / (prep_avg * 1e-3) / 1e9 if prep_avg > 0 else 0.0
    gemm_hbm_bytes = sum(s.M * s.K + s.M * (s.K // 64) * 4 + s.N * s.K // 2 + 2 * s.N * (s.K // 64) * 2 +
                         (4 * s.N if s.bias else 0) + 4 * s.M * s.N for s in specs) / len(lin)

    # ---------------- end to end through the C ABI with host buffers: the host-buffer call
    # (x in, y out in page-locked host memory; its chunked copies overlap the computation),
    # and for comparison the plain sequence copy in -> fused call -> copy out
    x_host = [torch.from_numpy(t["host"]["x"]).pin_memory() for t in lin]
    y_host = [torch.empty(t["y"].shape, dtype=torch.float32).pin_memory() for t in lin]
    ws_host = [binding.workspace(binding.prefill_host_workspace_bytes(s.M, s.N, s.K), device) for s in specs]
    e2e_steps = max(5, min(args.steps, 200))

    def host_call():
        for t, xh, yh, wh in zip(lin, x_host, y_host, ws_host):
            binding.prefill_linear_host(xh, t["wq"], t["s_w"], t["z_w"], t["bias"], y=yh, ws=wh, stream=stream)

    def copies_then_call():
        for t, xh, yh in zip(lin, x_host, y_host):
            t["x"].copy_(xh, non_blocking=True)
            binding.prefill_linear(t["x"], t["wq"], t["s_w"], t["z_w"], t["bias"], y=t["y"], ws=t["ws"],
                                   stream=stream)
            yh.copy_(t["y"], non_blocking=True)

    def e2e_time(body):
        ms = []
        for i in range(e2e_steps + 3):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            body()
            b.record(stream)
            b.synchronize()
            if i >= 3:
                ms.append(a.elapsed_time(b))
        return reduce_max(sum(ms) / 1e3, world, device)

    e2e_s = e2e_time(host_call)
    e2e_serial_s = e2e_time(copies_then_call)

    # the end-to-end bound: the copy engines' own rates, measured here on the largest linear's
    # buffers.  Within a call the copies in and out overlap (and hide the linear), calls run
    # in order, so a step takes at least sum over linears of max(x / h2d rate, y / d2h rate).
    def copy_rate(dst, src, reps=5):
        for _ in range(2):
            dst.copy_(src, non_blocking=True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record(stream)
        b.synchronize()
        return reps * src.numel() * src.element_size() / (a.elapsed_time(b) * 1e-3)

    big = max(range(len(lin)), key=lambda i: specs[i].M * (specs[i].K + specs[i].N))
    h2d_rate = copy_rate(lin[big]["x"], x_host[big])
    d2h_rate = copy_rate(y_host[big], lin[big]["y"])
    copy_bound_s = sum(max(s.M * s.K * 4 / h2d_rate, s.M * s.N * 4 / d2h_rate) for s in specs)
    e2e_bound = {"copy_bound_ms": round(copy_bound_s * 1e3, 4),
                 "frac": round(copy_bound_s * e2e_steps / e2e_s, 4),
                 "h2d_GBs": round(h2d_rate / 1e9, 1), "d2h_GBs": round(d2h_rate / 1e9, 1),
                 "rule": "sum over linears of max(x bytes / h2d rate, y bytes / d2h rate), "
                         "rates of one copy engine per direction measured in this run"}
    h2d = sum(s.M * s.K * 4 for s in specs)
    d2h = sum(s.M * s.N * 4 for s in specs)

    layer = None
    if args.workload in ("c3", "d3") and not args.shape:
        layer = layer_step(lin, specs, stream, flush, max(20, min(args.steps, 200)), decode)

    targets = None
    if not decode and not args.shape and not args.no_targets:
        targets = measure_targets(device, stream, flush, clk, tensor_peak, hbm_gbs, peak_src)
    clk.__exit__(None, None, None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(lin, specs, args.cpu_seconds)

    clocks = clk.summary(t_start, t_end)
    if decode:
        roofline = {"bound": "hbm",
                    "kernel": "gemv_kernel (packed u4 weights streamed, dp4a blocks + f32 epilogue)" +
                              (f"; one launch runs all {len(lin)} linears of the step" if step_launch else
                               "; one launch per linear"),
                    "achieved": round(gemv_gbs, 1), "peak": hbm_gbs, "unit": "GB/s",
                    "frac": round(gemv_gbs / hbm_gbs, 4),
                    "traffic": None if args.shape else recorded_traffic(args.workload), "peak_source": peak_src,
                    "bytes_per_launch": int(gemv_bytes), "gemv_us_per_launch": round(gemm_avg * 1e3, 3)}
    else:
        roofline = {"bound": "tensor",
                    "kernel": ("gemm_kernel (weight records; tcgen05 kind::f8f6f4 + kind::f16 zero-point MMA; "
                               "128-token tiles)" if M < WIDE_M else
                               "gemm_wide_kernel (weight records; tcgen05 kind::f8f6f4 + kind::f16 zero-point MMA; "
                               "256-token tiles)"),
                    "achieved": round(gemm_tops, 2), "peak": round(tensor_peak, 1), "unit": "TOPS",
                    "frac": round(gemm_tops / tensor_peak, 4),
                    "traffic": None if args.shape else recorded_traffic(args.workload),
                    "peak_source": f"{peak_src} bf16 burst x2 (fp8 nominal ratio) /2 (two e4m3 MACs per int8 MAC)",
                    "int8_mma_sync": {"peak": MMA_SYNC_S8_TOPS, "frac": round(gemm_tops / MMA_SYNC_S8_TOPS, 4),
                                      "unit": "TOPS", "source": MMA_SYNC_S8_SOURCE},
                    "gemm_us_per_launch": round(gemm_avg * 1e3, 3),
                    # small M is also read against HBM: the bytes a launch must move (codes, row
                    # sums, packed weights, scales and zeros, bias, y) over the same time
                    "hbm_view": {"bytes_per_launch": int(gemm_hbm_bytes),
                                 "achieved": round(gemm_hbm_bytes / (gemm_avg * 1e-3) / 1e9, 1),
                                 "peak": hbm_gbs, "unit": "GB/s",
                                 "frac": round(gemm_hbm_bytes / (gemm_avg * 1e-3) / 1e9 / hbm_gbs, 4)}}
    e2e_tops = whole_job_rate(ops_per_step * e2e_steps, world, e2e_s) / 1e12
    if decode:
        # a decode step is one token (per sequence of the batch) through every linear:
        # the headline is tokens per second, the TOPS ride along
        metric, unit, value, e2e_value = DECODE_METRIC, "tok/s", round(tok_s, 1), \
            round(whole_job_rate(M * e2e_steps, world, e2e_s), 1)
        if cpu is not None:
            cpu = dict(cpu, value=round(cpu["value"] * 1e12 / (ops_per_step / M), 3), unit="tok/s",
                       tops=cpu["value"])
    else:
        metric, unit, value, e2e_value = METRIC, "TOPS", round(value_tops, 3), round(e2e_tops, 3)
    out = {
        "metric": metric,
        "value": value,
        "unit": unit,
        "tok_s": round(tok_s, 1),
        "tops": round(value_tops, 4),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "ms_median": round(statistics.median(step_ms), 5),
        "ms_min": round(min(step_ms), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("int8 x u4 dp4a -> exact int32 blocks, f32 epilogue" if decode else
                  "e4m3xe4m3->f32 (exact int8 x u4 blocks), f32 epilogue"),
        "data": "synthetic (seeded Philox; no model weights)",
        "config": workload_config(args.workload, title, specs, world),
        "roofline": roofline,
        "prepass": ({"fused": "the few-token kernel quantizes the rows itself (no pre-pass launch)"}
                    if one_launch else
                    dict({"bound": "hbm", "achieved": round(prep_gbs, 1), "peak": hbm_gbs, "unit": "GB/s",
                          "frac": round(prep_gbs / hbm_gbs, 4), "us_per_launch": round(prep_avg * 1e3, 3),
                          "bytes_per_launch": int(prep_bytes),
                          "bytes_rule": "M*K*(4 + 1 + 4/64) + 8*M: x read; int8 codes, int32 block row sums, "
                                        "scale written",
                          "peak_source": peak_src},
                         **({} if decode else {"format_bytes": {
                             "bytes_per_launch": int(prep_fmt_bytes),
                             "achieved": round(prep_fmt_bytes / (prep_avg * 1e-3) / 1e9, 1),
                             "frac": round(prep_fmt_bytes / (prep_avg * 1e-3) / 1e9 / hbm_gbs, 4),
                             "rule": "bytes of the tensor-core record format: x read; two e4m3 nibble planes, "
                                     "16-byte zero-point entries per 64 elements, scale written"}}))),
        "e2e": {"value": e2e_value, "unit": unit,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_s * 1e3 / e2e_steps, 4),
                "call": "w4a8_prefill_linear_host: page-locked host x and y; a call of 16 MiB or more "
                        "overlaps its row chunks' copies with the linear, a smaller one reads x and writes y "
                        "in place over the host link (the few-token form copies x)",
                "bound": e2e_bound,
                "copies_then_call": {"value": round(e2e_value * e2e_s / e2e_serial_s, 3 if not decode else 1),
                                     "ms_per_step": round(e2e_serial_s * 1e3 / e2e_steps, 4)}},
        "gpu_launches": args.steps * kernels_per_step,
        "gpu_launches_per_step": kernels_per_step,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if not decode:
        # the whole fused step's data movement over the step time: the bytes the method needs,
        # and the bytes this design moves through its records (the weight expansion included)
        alg, des = (sum(v) for v in zip(*(fused_step_bytes(s.M, s.K, s.N, s.bias) for s in specs)))
        step_s = ms_per_step * 1e-3
        out["step_bytes"] = {"algorithmic": alg, "as_designed": des, "ratio": round(des / alg, 3),
                             "algorithmic_GBs": round(alg / step_s / 1e9, 1),
                             "as_designed_GBs": round(des / step_s / 1e9, 1), "peak": hbm_gbs,
                             "rule": "algorithmic: x, packed u4 weights, fp16 scales and zeros, bias read, y "
                                     "written, once each; as designed: plus the token and weight records "
                                     "written by the pre-pass and read by the contraction (weight rows padded "
                                     "to 128; L2 re-reads not counted)"}
    if layer is not None:
        out["layer"] = layer
    if targets is not None:
        out["targets"] = targets
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------ 7B-class kernel targets
def measure_targets(device, stream, flush, clk, tensor_peak, hbm_gbs, peak_src, reps=20):
    """The two kernel targets on the 7B-class workload (M 8192: K 4096 -> N 14336, then
    K 14336 -> N 4096), timed alone with CUDA events on the launching stream, L2 flushed
    before every launch (outside the events):
      - the contraction (gemm_wide_kernel, through w4a8_linear_prepared) against the INT8
        peaks: >= 50 % targeted;
      - the activation pre-pass against HBM on the algorithmic bytes M*K*(4 + 1 + 4/64) + 8*M,
        both as the fused call runs it (tensor-core records, w4a8_prepare_activations) and in
        the API layout (int8 a_q, s_a, int32 row sums: w4a8_quant_pack): >= 70 % targeted."""
    from w4a8_block_quantized_gb300 import binding, synth
    title, specs = synth.workload("c4")
    t0 = time.time()
    rows = {"gemm": [], "prep": [], "quant_pack": []}
    for spec in specs:
        d = synth.make_linear(spec)
        x = torch.from_numpy(d["x"]).to(device)
        wq, sw, zw = (torch.from_numpy(d[k]).to(device) for k in ("wq", "s_w", "z_w"))
        act = binding.prepare_activations(x, stream=stream)
        pw = binding.prepare_weights(wq, sw, zw, stream=stream)
        a_q, s_a, rs = binding.quant_pack(x, stream=stream)
        y = torch.empty((spec.M, spec.N), dtype=torch.float32, device=device)
        calls = {"gemm": lambda: binding.linear_prepared(act, pw, spec.M, spec.N, spec.K, y=y, stream=stream),
                 "prep": lambda: binding.prepare_activations(x, act=act, stream=stream),
                 "quant_pack": lambda: binding.quant_pack(x, a_q=a_q, a_scale=s_a, rowsum=rs, stream=stream)}
        for name, fn in calls.items():
            ms = []
            for i in range(reps + 3):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                b.synchronize()
                if i >= 3:
                    ms.append(a.elapsed_time(b))
            rows[name].append(statistics.fmean(ms) * 1e3)   # us per launch
        del x, wq, sw, zw, act, pw, a_q, s_a, rs, y
        torch.cuda.empty_cache()
    t1 = time.time()
    if binding.sync_status(stream) != 0:
        raise RuntimeError("device status reported a timeout in the targets leg")
    ops = sum(s.ops for s in specs)
    g_us = sum(rows["gemm"])
    g_tops = ops / (g_us * 1e-6) / 1e12
    pbytes = sum(prepass_bytes(s.M, s.K) for s in specs)
    fbytes = sum(record_prepass_bytes(s.M, s.K) for s in specs)

    def hbm(bytes_, us):
        gbs = bytes_ / (us * 1e-6) / 1e9
        return round(gbs, 1), round(gbs / hbm_gbs, 4)

    p_gbs, p_frac = hbm(pbytes, sum(rows["prep"]))
    q_gbs, q_frac = hbm(pbytes, sum(rows["quant_pack"]))
    f_gbs, f_frac = hbm(fbytes, sum(rows["prep"]))
    return {
        "workload": f"c4: {title}",
        "timing": f"each kernel alone, {reps} launches per linear after 3 warm-up launches, L2 flushed before "
                  "every launch (outside the events); figures over the two linears",
        "gemm": {"kernel": "gemm_wide_kernel (tcgen05 kind::f8f6f4 + kind::f16 zero-point MMA, 256-token tiles)",
                 "us_per_launch": [round(v, 2) for v in rows["gemm"]], "achieved": round(g_tops, 1),
                 "unit": "TOPS", "target_frac": 0.5,
                 "fp8_derived": {"peak": round(tensor_peak, 1), "frac": round(g_tops / tensor_peak, 4),
                                 "met": g_tops / tensor_peak >= 0.5,
                                 "source": f"{peak_src} bf16 burst x2 (fp8 nominal ratio) /2 (two e4m3 MACs "
                                           "per int8 MAC)"},
                 "int8_mma_sync": {"peak": MMA_SYNC_S8_TOPS, "frac": round(g_tops / MMA_SYNC_S8_TOPS, 4),
                                   "met": g_tops / MMA_SYNC_S8_TOPS >= 0.5, "source": MMA_SYNC_S8_SOURCE}},
        "prepass": {"kernel": "quant_kernel, tensor-core record output (the fused call's pre-pass)",
                    "us_per_launch": [round(v, 2) for v in rows["prep"]], "achieved": p_gbs, "unit": "GB/s",
                    "peak": hbm_gbs, "frac": p_frac, "target_frac": 0.7, "met": p_frac >= 0.7,
                    "bytes": int(pbytes), "bytes_rule": "M*K*(4 + 1 + 4/64) + 8*M",
                    "format_bytes": {"bytes": int(fbytes), "achieved": f_gbs, "frac": f_frac}},
        "quant_pack": {"kernel": "quant_kernel, API layout (int8 a_q, fp32 s_a, int32 row sums)",
                       "us_per_launch": [round(v, 2) for v in rows["quant_pack"]], "achieved": q_gbs,
                       "unit": "GB/s", "peak": hbm_gbs, "frac": q_frac, "target_frac": 0.7, "met": q_frac >= 0.7,
                       "bytes": int(pbytes), "bytes_rule": "M*K*(4 + 1 + 4/64) + 8*M"},
        "clocks": clk.summary(t0, t1),
    }


# ------------------------------------------------------------------ decoder layer as a layer
# Inputs a real decoder layer shares: q, k, v read one activation, gate and up another.  A
# layer stores each such group's weights with their rows concatenated (one linear of
# N = sum of the group's N), so the shared input is quantized once and contracted in one call.
LAYER_GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


def layer_step(lin, specs, stream, flush, reps, decode):
    """The 7-linear set run the way a decoder layer runs it: q/k/v and gate/up as
    row-concatenated groups on their shared inputs (4 linears).  Prefill: weights prepared
    once at load time, per step one pre-pass and one contraction per group; decode: the four
    groups in one batch call (one few-token launch where they fit one).  Timed per step (L2 flushed before each,
    outside the events) as eager calls and replayed from a command tape."""
    from w4a8_block_quantized_gb300 import binding
    by = {t["spec"].name: t for t in lin}
    M = specs[0].M
    dev = lin[0]["x"].device
    calls = []
    group_entries = []
    for grp in LAYER_GROUPS:
        ts = [by[nm] for nm in grp]
        K = ts[0]["spec"].K
        N = sum(t["spec"].N for t in ts)
        x = ts[0]["x"]
        wq = torch.cat([t["wq"] for t in ts]).contiguous()
        s_w = torch.cat([t["s_w"] for t in ts]).contiguous()
        z_w = torch.cat([t["z_w"] for t in ts]).contiguous()
        bias = None
        if any(t["bias"] is not None for t in ts):
            bias = torch.cat([t["bias"] if t["bias"] is not None else torch.zeros(t["spec"].N, device=dev)
                              for t in ts]).contiguous()
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        if decode:
            ws = binding.workspace(binding.prefill_workspace_bytes(M, N, K), dev)
            group_entries.append(dict(x=x, wq=wq, s_w=s_w, z_w=z_w, bias=bias, y=y, ws=ws))
        else:
            act = binding.workspace(binding.prepared_activations_bytes(M, K), dev)
            pw = binding.prepare_weights(wq, s_w, z_w, stream=stream)
            calls.append(lambda s, x=x, act=act: binding.prepare_activations(x, act=act, stream=s))
            calls.append(lambda s, act=act, pw=pw, N=N, K=K, bias=bias, y=y: binding.linear_prepared(
                act, pw, M, N, K, bias=bias, y=y, stream=s))
    if decode:
        # the four groups as one batch call (one few-token launch per group, weights streamed early)
        layer_batch = binding.Batch(group_entries, stream)
        calls.append(lambda s: layer_batch.run(s))
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for c in calls:
            c(side)                      # one ordinary call of each before recording
        with binding.Tape(side) as tape:
            for c in calls:
                c(side)
    side.synchronize()
    launches = tape.kernels()

    def timed(run):
        ms = []
        for i in range(reps + 3):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(side)
            run()
            b.record(side)
            b.synchronize()
            if i >= 3:
                ms.append(a.elapsed_time(b))
        return statistics.fmean(ms)

    with torch.cuda.stream(side):
        side.wait_stream(torch.cuda.current_stream())
        t_eager = timed(lambda: [c(side) for c in calls])
        t_tape = timed(lambda: tape.replay(side))
    if binding.sync_status(side) != 0:
        raise RuntimeError("device status reported a timeout in the layer step")
    tape.free()
    ops = sum(s.ops for s in specs)
    return {"mode": ("q/k/v and gate/up as row-concatenated groups on shared inputs (4 linears); " +
                     ("one batch call (the four groups in one few-token launch where they fit one, "
                      "else a launch each)" if decode else
                      "weights prepared at load, per group one pre-pass + one contraction")),
            "launches_per_step": launches,
            "ms_per_step_eager": round(t_eager, 5), "ms_per_step_tape": round(t_tape, 5),
            "tok_s_tape": round(M / (t_tape * 1e-3), 1), "tops_tape": round(ops / (t_tape * 1e-3) / 1e12, 3),
            "l2": "flushed before every step (outside the events)"}


# ------------------------------------------------------------------ CPU oracle legs
def oracle_rows_for(spec, seconds, x, host):
    """Rows of the workload the oracle processes in about `seconds` (calibrated on 4 rows)."""
    import oracle
    rows = np.arange(min(4, spec.M), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.prefill_linear(x, host["wq"], host["s_w"], host["z_w"], host["bias"], rows=rows)
    dt = max(time.perf_counter() - t0, 1e-4) / len(rows)
    return int(max(4, min(spec.M, seconds / dt)))


def cpu_baseline(lin, specs, seconds):
    import oracle
    oracle.build()
    total_ops, total_s, parts = 0, 0.0, []
    for t, s in zip(lin, specs):
        h = t["host"]
        n = oracle_rows_for(s, seconds / len(specs), h["x"], h)
        rows = np.linspace(0, s.M - 1, n).astype(np.int64)
        t0 = time.perf_counter()
        oracle.prefill_linear(h["x"], h["wq"], h["s_w"], h["z_w"], h["bias"], rows=rows)
        dt = time.perf_counter() - t0
        # a workload the oracle finishes well inside the target is repeated up to the target
        reps = int(max(0, min(1000, seconds / len(specs) / max(dt, 1e-6) - 1)))
        t0 = time.perf_counter()
        for _ in range(reps):
            oracle.prefill_linear(h["x"], h["wq"], h["s_w"], h["z_w"], h["bias"], rows=rows)
        dt += time.perf_counter() - t0
        total_ops += 2 * n * s.N * s.K * (reps + 1)
        total_s += dt
        parts.append(f"{s.name}: {n}/{s.M} rows x {reps + 1}")
    out = {"value": round(total_ops / total_s / 1e12, 6), "unit": "TOPS", "cores": oracle.num_threads(),
           "kind": "oracle", "sample": "evenly spaced rows of the workload, all outputs: " + "; ".join(parts),
           "seconds": round(total_s, 2), "cpu": cpu_model(), "nproc": os.cpu_count()}
    # the same oracle compiled without OpenMP, on one core, for a quarter of the time
    oracle.build(tag="oracle_1core", openmp=False)
    s, h = specs[0], lin[0]["host"]
    rows1 = np.arange(min(4, s.M), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.prefill_linear(h["x"], h["wq"], h["s_w"], h["z_w"], h["bias"], rows=rows1, tag="oracle_1core")
    dt1 = max(time.perf_counter() - t0, 1e-4) / len(rows1)
    n1 = int(max(4, min(s.M, seconds / 4 / dt1)))
    rows1 = np.linspace(0, s.M - 1, n1).astype(np.int64)
    reps1 = max(1, min(1000, int(seconds / 4 / (dt1 * n1))))
    t0 = time.perf_counter()
    for _ in range(reps1):
        oracle.prefill_linear(h["x"], h["wq"], h["s_w"], h["z_w"], h["bias"], rows=rows1, tag="oracle_1core")
    dt1 = time.perf_counter() - t0
    out["one_core"] = {"value": round(2 * n1 * s.N * s.K * reps1 / dt1 / 1e12, 6), "unit": "TOPS",
                       "sample": f"{s.name}: {n1}/{s.M} rows x {reps1}", "seconds": round(dt1, 2)}
    return out


def cpu_model() -> str:
    """The host CPU's model name (lscpu), else the machine type."""
    import platform
    try:
        text = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in text.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from w4a8_block_quantized_gb300 import synth
    oracle.build()
    title, specs = synth.workload(args.workload)
    hosts = [synth.make_linear(s) for s in specs]
    per_step = max(0.5, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    rows = [np.linspace(0, s.M - 1, oracle_rows_for(s, per_step / len(specs), h["x"], h)).astype(np.int64)
            for s, h in zip(specs, hosts)]

    def step():
        for s, h, r in zip(specs, hosts, rows):
            oracle.prefill_linear(h["x"], h["wq"], h["s_w"], h["z_w"], h["bias"], rows=r)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    ops = args.steps * sum(2 * len(r) * s.N * s.K for s, r in zip(specs, rows))
    value = ops / dt / 1e12
    toks = args.steps * sum(len(r) for r in rows) / len(rows) / dt
    sample = "; ".join(f"{s.name}: {len(r)}/{s.M} evenly spaced rows" for s, r in zip(specs, rows))
    metric, unit = METRIC, "TOPS"
    if specs[0].M <= synth.DECODE_MAX_M:
        metric, unit, value = DECODE_METRIC, "tok/s", toks
    out = {
        "metric": metric, "value": round(value, 6), "unit": unit, "tok_s": round(toks, 2), "impl": "reference",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32/int64 blocks, f64 output", "data": "synthetic (seeded Philox)",
        "config": workload_config(args.workload, title, specs, args.gpus),
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_bench(args)


if __name__ == "__main__":
    main()
