#!/usr/bin/env python
"""Benchmark of the GB300 Llama decoder block (C ABI, sm_103a kernels).

Workload (one step = one llama_block_forward): the Llama-3-8B-shaped block
prefill, B=1, S=8192, d_model=4096, 32 query / 8 KV heads of width 128,
d_ff=14336, rope_theta=5e5, bf16 with fp32 accumulation, causal, start_pos=0,
synthetic seeded inputs (x ~ N(0,1), weights ~ N(0,0.02), gains 1+N(0,0.1)).

Prints one JSON line (rank 0).  value = whole-job tokens/s with inputs resident
in HBM; e2e = the same through llama_block_forward_host with pinned host
buffers (copies inside the timed region); roofline = the gate/up + SwiGLU GEMM
(largest share of the step) timed with CUDA events inside the timed region;
cpu_baseline = the fp64 oracle on the host cores on a bounded sample of the
same workload.  `--impl reference` times that oracle as the reference arm.

Multi-GPU (torchrun): replicas only -- every rank runs its own block on its own
sequence; no collective on the data path; barrier + max-over-ranks timing.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decoder-block tokens/s (prefill) & decode µs/step; % of bf16 TC / HBM roofline"
WORKLOAD = "llama3_8b_block_prefill_b1s8192"
SHAPE = dict(d_model=4096, n_heads=32, n_kv_heads=8, d_ff=14336, norm_eps=1e-5, rope_theta=5e5, dtype="bf16",
             B=1, S=8192, start_pos=0, max_seq_len=8192)
SMOLLM2_SHAPE = dict(d_model=576, n_heads=9, n_kv_heads=3, d_ff=1536, norm_eps=1e-5, rope_theta=1e5, B=8, S=1024)
DECODE = dict(SHAPE, B=64, S=1, start_pos=4095, max_seq_len=4096)


def block_flops(s):
    d, H, G, F = s["d_model"], s["n_heads"], s["n_kv_heads"], s["d_ff"]
    D = d // H
    T = s["B"] * s["S"]
    linear = 2.0 * T * (d * (H + 2 * G) * D + H * D * d + d * 2 * F + F * d)
    pairs = s["B"] * sum(s["start_pos"] + i + 1 for i in range(s["S"]))  # causal (query, key) pairs
    attn = 4.0 * D * H * pairs
    return linear, attn


def gate_up_flops(s):
    return 2.0 * s["B"] * s["S"] * s["d_model"] * 2 * s["d_ff"]


def decode_attention_bytes(s):
    D = s["d_model"] // s["n_heads"]
    kv = 2.0 * s["B"] * s["n_kv_heads"] * (s["start_pos"] + 1) * D * 2
    qo = 2.0 * s["B"] * s["n_heads"] * D * 2
    return kv + qo


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return m, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def choose_bf16_peak(peaks, timed_s, clocks):
    """The measured bf16 peak a tensor-bound kernel is held to: the burst
    figure when the timed region was short (under 1 s) and ran at full clock
    (median SM clock within 5 % of its maximum), else the sustained figure,
    which was measured over seconds under the power cap."""
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    full_clock = sm is not None and smax and sm >= 0.95 * smax
    if timed_s < 1.0 and full_clock:
        return burst, "bf16_tflops (burst)", f"timed region {timed_s:.2f} s at median SM {sm:.0f} of {smax:.0f} MHz"
    why = f"timed region {timed_s:.2f} s" + (f", median SM {sm:.0f} of {smax:.0f} MHz" if sm and smax else "")
    return sustained, "bf16_tflops_sustained", why


def kernel_traffic(name):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        table = json.load(f)
    ent = table.get(name)
    if not ent or "sources" not in ent:
        return None
    h = hashlib.sha256()
    for rel in ent["sources"]:  # the kernel's source files, hashed in the listed order
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        with open(src, "rb") as f:
            h.update(f.read())
    return ent["dram_bytes_per_launch"] if h.hexdigest() == ent["sources_sha256"] else None


# ----------------------------------------------------------- clock sampler ---

class NvmlClockSampler:
    """SM clock and clock-event reasons of one GPU, read (never set) through
    NVML every 10 ms on a host thread, with host timestamps, so that the
    samples falling inside a timed region can be picked out even when the
    region lasts only tens of milliseconds."""
    NVML_CLOCK_SM = 1
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, uuid: str, period_s: float = 0.01):
        import ctypes
        import threading
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.handle)) != 0:
            raise OSError(f"no NVML device {uuid}")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.sm_max = float(mx.value) if self.lib.nvmlDeviceGetMaxClockInfo(
            self.handle, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0 else None
        self.period = period_s
        self.samples = []  # (host time, SM MHz, reason bits)
        self.stop_evt = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_evt.is_set():
            t = time.perf_counter()
            if self.lib.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, ct.byref(clk)) == 0:
                bits = rs.value if self.reasons_fn(self.handle, ct.byref(rs)) == 0 else 0
                self.samples.append((t, float(clk.value), bits))
            self.stop_evt.wait(self.period)

    def start(self):
        self.thread.start()
        t_end = time.perf_counter() + 1.0
        while not self.samples and time.perf_counter() < t_end:  # running before the timed region
            time.sleep(0.005)

    def stop(self):
        self.stop_evt.set()
        self.thread.join(timeout=2)

    def window(self, t0, t1):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        if not inside and self.samples:  # a region shorter than one period: the nearest sample
            inside = [min(self.samples, key=lambda x: abs(x[0] - 0.5 * (t0 + t1)))]
        sm = [x[1] for x in inside]
        reasons = sorted({n for x in inside for b, n in self.REASON_BITS.items() if x[2] & b})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.sm_max, "reasons": reasons,
                "samples": len(sm), "sampler": f"NVML every {int(self.period * 1e3)} ms, inside the timed region",
                "window_s": t1 - t0}


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names[1:], parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ cpu oracle ---

def oracle_sample(tokens: int, seed_tag: str = "bench"):
    """Inputs of a bounded sample of the workload: same weights, first `tokens` positions."""
    import synth
    s = dict(SHAPE, S=tokens, max_seq_len=tokens)
    w = synth.block_weights(SHAPE)
    wf = {k: synth.as_f64(v) for k, v in w.items()}
    x = synth.as_f64(synth.block_activations(s, tag=seed_tag, B=1, S=tokens))
    kc, vc = synth.kv_cache(s, max_batch=1, max_seq_len=tokens)
    return s, wf, x, synth.as_f64(kc), synth.as_f64(vc)


def time_oracle(tokens: int, reps: int = 1):
    import oracle
    s, wf, x, kc, vc = oracle_sample(tokens)
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.block_forward(s, wf, x, 0, kc, vc)
        times.append(time.perf_counter() - t0)
    return times


def cpu_info():
    return {"cores": os.cpu_count()}


# ------------------------------------------------------------------ main ---

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, tokens_per_rank_step, steps, max_ms):
    """Whole-job tokens/s of `world` replicas that each ran `steps` steps of `tokens_per_rank_step`
    tokens, timed by the slowest rank (max_ms over the timed region)."""
    return world * tokens_per_rank_step * steps / (max_ms / 1e3)


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    tokens = args.ref_tokens
    times = time_oracle(tokens, reps=args.warmup + args.steps)
    timed = times[args.warmup:]
    total = sum(timed)
    value = tokens * len(timed) / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(timed),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": SHAPE["B"], "S": SHAPE["S"], "sample_tokens_per_step": tokens,
                   "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"first {tokens} positions of the B=1 S=8192 prefill per step, same block weights"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=2048, help="oracle sample size for cpu_baseline")
    ap.add_argument("--ref-tokens", type=int, default=512, help="oracle sample per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary block shapes (SmolLM2-shaped block, 8B prefill B=4 S=2048)")
    ap.add_argument("--no-stack", action="store_true", help="skip the 32-layer stack measurement")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode step (B=64 at start_pos 4095); for profiler captures")
    ap.add_argument("--smollm2-only", action="store_true",
                    help="time only the SmolLM2-shaped block (B=8, S=1024, d_model 576); for profiler captures")
    ap.add_argument("--standalone-only", action="store_true",
                    help="time only the standalone RMSNorm and RoPE + KV-write launches; for profiler captures")
    ap.add_argument("--seq", type=int, default=8192,
                    help="prefill length S (default 8192; smaller values are for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    global SHAPE, WORKLOAD
    if args.seq != SHAPE["S"]:
        SHAPE = dict(SHAPE, S=args.seq, max_seq_len=args.seq)
        WORKLOAD = f"llama3_8b_block_prefill_b1s{args.seq}"

    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import numpy as np
    import torch

    import decoder_block_gb300 as lb
    import synth

    lb.load()  # raises when the library has not been built: there is no fallback
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    if args.standalone_only:
        ops = bench_standalone_ops(lb, torch, dev, stream, args, measured_peaks()[0])
        if rank == 0:
            print(json.dumps({"metric": "standalone RMSNorm and RoPE + KV write, % of HBM", "value":
                              ops["rmsnorm_8192x4096"]["hbm_frac"], "unit": "fraction of measured HBM GB/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                              "dtype": "bf16", "data": "synthetic", "config": {"workload": "standalone_ops_8192x4096"},
                              "standalone_ops": ops}), flush=True)
        return 0
    if args.smollm2_only:
        sm = bench_block_shape(lb, torch, dev, stream, SMOLLM2_SHAPE, args)
        if rank == 0:
            print(json.dumps({"metric": "SmolLM2-shaped block tokens/s", "value": sm["tokens_per_s"], "unit": "tokens/s",
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                              "dtype": "bf16", "data": "synthetic",
                              "config": {"workload": "smollm2_135m_block_b8s1024"}, "smollm2": sm}), flush=True)
        return 0
    # ---- inputs (seeded synthetic, the same recipe as the parity tests) ----
    w_np = synth.block_weights(SHAPE)
    w = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(dev) for k, v in w_np.items()}
    B, S, d = SHAPE["B"], SHAPE["S"], SHAPE["d_model"]
    G, D = SHAPE["n_kv_heads"], d // SHAPE["n_heads"]
    if args.decode_only:
        decode = bench_decode(lb, torch, w, dev, stream, args, measured_peaks()[0])
        if rank == 0:
            print(json.dumps({"metric": "decode block step µs (B=64 at start_pos 4095)", "value": decode["us_per_step"],
                              "unit": "us/step", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "higher_is_better": False, "dtype": "bf16", "data": "synthetic",
                              "config": {"workload": decode["workload"]}, "decode": decode}), flush=True)
        return 0
    x_np = synth.block_activations(SHAPE)
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(dev)
    y = torch.empty_like(x)
    kc = torch.zeros((B, G, SHAPE["max_seq_len"], D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    cfg = lb.make_config(d, SHAPE["n_heads"], G, SHAPE["d_ff"], SHAPE["max_seq_len"], SHAPE["norm_eps"],
                         SHAPE["rope_theta"], lb.LLAMA_BF16)
    st, blk = lb.llama_block_create(cfg, lb.make_weights(w), B * S)
    lb.check(st, "llama_block_create")
    kv = lb.make_kv_cache(kc, vc, B, SHAPE["max_seq_len"])

    def step():
        lb.check(lb.llama_block_forward(blk, x, y, B, S, 0, kv, stream), "llama_block_forward")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    lb.check(lb.llama_block_device_status(blk), "device status")

    # ---- timed region: K forwards, inputs resident in HBM ----
    gpu_index = local
    try:
        gpu_index = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    try:
        clocks = NvmlClockSampler(gpu_index)
    except (OSError, AttributeError):
        clocks = ClockSampler(gpu_index)  # nvidia-smi every 50 ms
    clocks.start()
    lb.check(lb.llama_block_profile_enable(blk, args.steps), "profile enable")
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = lb.llama_kernel_launch_count()
    t_region0 = time.perf_counter()
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    launches_timed = lb.llama_kernel_launch_count() - launches0
    torch.cuda.synchronize()
    t_region1 = time.perf_counter()
    barrier(world)
    elapsed_ms = ev0.elapsed_time(ev1)
    st, launches, total_ms = lb.llama_block_profile_read(blk)
    lb.check(st, "profile read")
    lb.llama_block_profile_disable(blk)
    if isinstance(clocks, NvmlClockSampler):
        clocks.stop()
        clock_info = clocks.window(t_region0, t_region1)
    else:
        clock_info = clocks.stop()
    lb.check(lb.llama_block_device_status(blk), "device status")
    max_ms = max_over_ranks(elapsed_ms, world)
    ms_per_step = max_ms / args.steps
    value = replica_throughput(world, B * S, args.steps, max_ms)

    # ---- end to end: host buffers through llama_block_forward_host ----
    # Every step copies its input from pinned host memory and reads its result back inside
    # the timed region.  Measured two ways: one stream (copies serialised with the compute),
    # and two independent sequences in flight on two streams and two block handles -- how a
    # serving engine pipelines requests -- so one stream's copies overlap the other's compute.
    xh = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    e2e_steps = max(4, min(args.steps, 40)) // 2 * 2
    for _ in range(2):
        lb.check(lb.llama_block_forward_host(blk, xh, yh, B, S, 0, kv, stream), "forward_host")
    torch.cuda.synchronize()
    barrier(world)
    ev0.record(stream)
    for _ in range(e2e_steps):
        lb.check(lb.llama_block_forward_host(blk, xh, yh, B, S, 0, kv, stream), "forward_host")
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_1s_ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    # second handle, cache, host buffers and stream
    st2, blk2 = lb.llama_block_create(cfg, lb.make_weights(w), B * S)
    lb.check(st2, "llama_block_create (second stream)")
    kc2, vc2 = torch.zeros_like(kc), torch.zeros_like(vc)
    kv2 = lb.make_kv_cache(kc2, vc2, B, SHAPE["max_seq_len"])
    xh2 = xh.clone().pin_memory()
    yh2 = torch.empty_like(xh).pin_memory()
    s2 = torch.cuda.Stream(device=dev)
    lanes = [(blk, kv, xh, yh, stream), (blk2, kv2, xh2, yh2, s2)]
    for hb, hkv, hx, hy, hs in lanes:
        lb.check(lb.llama_block_forward_host(hb, hx, hy, B, S, 0, hkv, hs), "forward_host")
    torch.cuda.synchronize()
    barrier(world)
    ev0.record(stream)
    s2.wait_event(ev0)
    for i in range(e2e_steps):
        hb, hkv, hx, hy, hs = lanes[i % 2]
        lb.check(lb.llama_block_forward_host(hb, hx, hy, B, S, 0, hkv, hs), "forward_host")
    ev_s2 = torch.cuda.Event()
    ev_s2.record(s2)
    stream.wait_event(ev_s2)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1), world)
    lb.check(lb.llama_block_device_status(blk2), "device status (second stream)")
    lb.llama_block_destroy(blk2)
    del kc2, vc2
    e2e_value = replica_throughput(world, B * S, e2e_steps, e2e_ms)
    e2e_1s_value = replica_throughput(world, B * S, e2e_steps, e2e_1s_ms)
    io_bytes = B * S * d * 2

    # ---- roofline of the dominant kernel (gate/up + SwiGLU GEMM) ----
    peaks, peak_kind = measured_peaks()
    gu = 6
    gu_ms = total_ms[gu] / max(launches[gu], 1)
    gu_tflops = gate_up_flops(SHAPE) / (gu_ms / 1e3) / 1e12
    peak, peak_name, peak_why = choose_bf16_peak(peaks, max_ms / 1e3, clock_info)
    burst = float(peaks["bf16_tflops"])
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    traffic = kernel_traffic("gate_up_swiglu")
    # steps fused into another step's kernel launch nothing and read 0 launches
    step_ms = {lb.llama_profile_step_name(i): total_ms[i] / launches[i] for i in range(len(launches)) if launches[i]}
    lin, att = block_flops(SHAPE)
    block_tflops = (lin + att) / (ms_per_step / 1e3) / 1e12

    # ---- secondary: decode step (B=64 at start_pos 4095 over a filled cache) ----
    decode = None
    if not args.no_decode:
        decode = bench_decode(lb, torch, w, dev, stream, args, peaks)

    lb.llama_block_destroy(blk)
    del kc, vc

    secondary = {}
    if not args.no_secondary:
        secondary["smollm2_135m_block_b8s1024"] = bench_block_shape(lb, torch, dev, stream, SMOLLM2_SHAPE, args)
        secondary["llama3_8b_block_prefill_b4s2048"] = bench_block_shape(
            lb, torch, dev, stream, dict(SHAPE, B=4, S=2048), args, weights=w)
        secondary["llama4_scout_shaped_moe_block"] = bench_moe(lb, torch, dev, stream, args)
        secondary["standalone_ops"] = bench_standalone_ops(lb, torch, dev, stream, args, peaks)
    stack = None
    if not args.no_stack:
        del w
        torch.cuda.empty_cache()
        stack = bench_stack(lb, torch, dev, stream, args)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "S": S, "d_model": d, "n_heads": SHAPE["n_heads"],
                   "n_kv_heads": G, "d_ff": SHAPE["d_ff"], "start_pos": 0, "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (436 MB of weights read per step, plus activations and KV)",
                   "block_tflops": block_tflops, "block_frac_of_bf16_peak": block_tflops / peak,
                   "block_frac_of_bf16_burst": block_tflops / burst,
                   "block_frac_of_bf16_sustained": block_tflops / sustained},
        "roofline": {"kernel": "gate_up_swiglu (tcgen05 GEMM, SiLU*up epilogue)", "bound": "tensor",
                     "achieved": gu_tflops, "peak": peak, "unit": "TFLOP/s", "frac": gu_tflops / peak,
                     "traffic": traffic, "peak_source": f"{peak_kind} {peak_name}: {peak_why}",
                     "frac_of_burst": gu_tflops / burst, "frac_of_sustained": gu_tflops / sustained},
        "step_ms": step_ms,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": io_bytes,
                "d2h_bytes_per_step": io_bytes, "steps": e2e_steps,
                "how": "llama_block_forward_host with pinned host buffers; two sequences in flight on two streams "
                       "(two block handles), copies inside the timed region",
                "single_stream_value": e2e_1s_value},
        "gpu_launches": launches_timed,
        "clocks": clock_info,
    }
    if decode is not None:
        line["decode"] = decode
    if secondary:
        line["secondary"] = secondary
    if stack is not None:
        line["stack"] = stack
    if rank == 0 and not args.no_cpu_baseline:
        times = time_oracle(args.cpu_tokens)
        line["cpu_baseline"] = {"value": args.cpu_tokens / times[0], "unit": "tokens/s", "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"fp64 numpy oracle, first {args.cpu_tokens} positions of the B=1 S=8192 "
                                          f"prefill with the same block weights ({times[0]:.1f} s)"}
    if decode is not None:  # kept short and last, so that a truncated tail of the line still holds it
        line["decode_summary"] = {k: decode[k] for k in ("us_per_step", "step_hbm_frac", "attention_us",
                                                         "attention_hbm_frac")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _rand_weights(torch, dev, s, seed):
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    d, H, G, F = s["d_model"], s["n_heads"], s["n_kv_heads"], s["d_ff"]
    D = d // H

    def rn(*shape, std=0.02, mean=0.0):
        return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std + mean).to(torch.bfloat16)

    return {"attn_norm": rn(d, std=0.1, mean=1.0), "wq": rn(H * D, d), "wk": rn(G * D, d), "wv": rn(G * D, d),
            "wo": rn(d, H * D), "ffn_norm": rn(d, std=0.1, mean=1.0), "w_gate": rn(F, d), "w_up": rn(F, d),
            "w_down": rn(d, F)}


def bench_block_shape(lb, torch, dev, stream, s, args, weights=None):
    """tokens/s of one block forward at another shape (device-generated inputs)."""
    B, S, d, G = s["B"], s["S"], s["d_model"], s["n_kv_heads"]
    D = d // s["n_heads"]
    w = weights if weights is not None else _rand_weights(torch, dev, s, 2)
    cfg = lb.make_config(d, s["n_heads"], G, s["d_ff"], S, s["norm_eps"], s["rope_theta"], lb.LLAMA_BF16)
    st, blk = lb.llama_block_create(cfg, lb.make_weights(w), B * S)
    lb.check(st, "llama_block_create (secondary)")
    x = torch.randn((B, S, d), device=dev, dtype=torch.float32).to(torch.bfloat16)
    y = torch.empty_like(x)
    kc = torch.zeros((B, G, S, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    kv = lb.make_kv_cache(kc, vc, B, S)
    for _ in range(args.warmup):
        lb.check(lb.llama_block_forward(blk, x, y, B, S, 0, kv, stream))
    steps = max(10, min(args.steps, 100))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    n0 = lb.llama_kernel_launch_count()
    e0.record(stream)
    for _ in range(steps):
        lb.check(lb.llama_block_forward(blk, x, y, B, S, 0, kv, stream))
    e1.record(stream)
    per_forward = (lb.llama_kernel_launch_count() - n0) // steps
    torch.cuda.synchronize()
    ms_plain = e0.elapsed_time(e1) / steps
    # the same step captured once in a CUDA graph and replayed (no per-kernel launch gaps)
    gstream = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gstream):
        lb.check(lb.llama_block_forward(blk, x, y, B, S, 0, kv, gstream))
        gstream.synchronize()
        with torch.cuda.graph(graph, stream=gstream):
            lb.check(lb.llama_block_forward(blk, x, y, B, S, 0, kv, gstream))
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_graph = e0.elapsed_time(e1) / steps
    lb.check(lb.llama_block_device_status(blk))
    lb.llama_block_destroy(blk)
    ms = min(ms_plain, ms_graph)
    lin, att = block_flops(dict(s, start_pos=0))
    return {"B": B, "S": S, "d_model": d, "ms_per_step": ms, "ms_per_step_plain_launches": ms_plain,
            "ms_per_step_cuda_graph": ms_graph, "tokens_per_s": B * S / (ms / 1e3),
            "tflops": (lin + att) / (ms / 1e3) / 1e12, "steps": steps, "kernels_per_step": per_forward,
            "gpu_launches": per_forward * steps}


def bench_moe(lb, torch, dev, stream, args, B=1, S=8192):
    """A Llama-4-Scout-shaped mixture-of-experts block prefill: d 5120, 40 query / 8 KV heads of width 128,
    16 experts of width 8192, top-1 routing, one shared expert of width 8192 (device-generated weights)."""
    d, H, G, D, E, k, F, Fs = 5120, 40, 8, 128, 16, 1, 8192, 8192
    g = torch.Generator(device=dev)
    g.manual_seed(5)

    def rn(*shape, std=0.02, mean=0.0):
        return (torch.randn(shape, generator=g, device=dev, dtype=torch.float32) * std + mean).to(torch.bfloat16)

    w = {"attn_norm": rn(d, std=0.1, mean=1.0), "wq": rn(H * D, d), "wk": rn(G * D, d), "wv": rn(G * D, d),
         "wo": rn(d, H * D), "ffn_norm": rn(d, std=0.1, mean=1.0), "w_gate": rn(E, F, d), "w_up": rn(E, F, d),
         "w_down": rn(E, d, F), "router": rn(E, d), "shared_gate": rn(Fs, d), "shared_up": rn(Fs, d),
         "shared_down": rn(d, Fs)}
    cfg = lb.make_config(d, H, G, F, S, 1e-5, 5e5, lb.LLAMA_BF16, n_experts=E, top_k=k, d_ff_shared=Fs)
    st, blk = lb.llama_block_create(cfg, lb.make_weights(w), B * S)
    lb.check(st, "llama_block_create (moe)")
    del w
    torch.cuda.empty_cache()
    x = torch.randn((B, S, d), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    y = torch.empty_like(x)
    kc = torch.zeros((B, G, S, D), dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    kv = lb.make_kv_cache(kc, vc, B, S)
    for _ in range(args.warmup):
        lb.check(lb.llama_block_forward(blk, x, y, B, S, 0, kv, stream))
    steps = max(10, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    n0 = lb.llama_kernel_launch_count()
    e0.record(stream)
    for _ in range(steps):
        lb.check(lb.llama_block_forward(blk, x, y, B, S, 0, kv, stream))
    e1.record(stream)
    per_forward = (lb.llama_kernel_launch_count() - n0) // steps
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # per-step breakdown (events around each step's kernels, plain launches)
    lb.check(lb.llama_block_profile_enable(blk, 3))
    for _ in range(3):
        lb.check(lb.llama_block_forward(blk, x, y, B, S, 0, kv, stream))
    torch.cuda.synchronize()
    _, launches, total_ms = lb.llama_block_profile_read(blk)
    lb.llama_block_profile_disable(blk)
    names = {5: "routing_dispatch", 6: "experts_gate_up_and_shared_gate_up", 7: "experts_down_shared_down_combine"}
    step_ms = {names.get(i, lb.llama_profile_step_name(i)): total_ms[i] / max(launches[i], 1)
               for i in range(len(launches)) if launches[i] > 0}
    ids = torch.empty((B * S, k), dtype=torch.int32, device=dev)
    wts = torch.empty((B * S, k), dtype=torch.float32, device=dev)
    lb.check(lb.llama_block_moe_routing(blk, ids, wts, stream))
    torch.cuda.synchronize()
    load = torch.bincount(ids.flatten().long(), minlength=E).cpu().tolist()
    status = lb.llama_block_device_status(blk)
    lb.llama_block_destroy(blk)
    T = B * S
    lin = 2.0 * T * (d * (H + 2 * G) * D + H * D * d + d * 64 + k * 3 * d * F + 3 * d * Fs)
    att = 4.0 * D * H * (S * (S + 1) / 2) * B
    return {"workload": "llama4_scout_shaped_moe_block_prefill_b1s8192_e16_top1_shared",
            "ms_per_step": ms, "tokens_per_s": T / (ms / 1e3), "tflops": (lin + att) / (ms / 1e3) / 1e12,
            "rows_per_expert": load, "steps": steps, "kernels_per_step": per_forward, "step_ms": step_ms,
            "gpu_launches": per_forward * steps, "device_status": status}


def bench_standalone_ops(lb, torch, dev, stream, args, peaks):
    """The per-step entry points whose own HBM roofline the scope table lists:
    RMSNorm over 8192 x 4096 bf16 (read x, write the normalised rows: 134.2 MB)
    and RoPE + KV-cache write at the prefill workload (read qkv, write rotated q,
    rotated k and v into the cache: 201.3 MB).  Each launch is timed alone with
    CUDA events on the launching stream, after a read of a buffer larger than L2,
    so that the operands come from HBM and L2 holds no dirty lines (after a
    write flush the launch would also pay for writing back up to 129 MB of the
    flush buffer, as much as its own traffic).  The event durations measured here
    fall on steps of about 2 us (2.048 us), a tenth of these launches; a launch
    starts at a random phase of that step, so the mean over the launches is
    reported (the median is kept beside it: it moves in whole steps)."""
    T, d, H, G, D = 8192, SHAPE["d_model"], SHAPE["n_heads"], SHAPE["n_kv_heads"], SHAPE["d_model"] // SHAPE["n_heads"]
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    hbm = float(peaks["hbm_gbs"])
    n = max(min(args.steps, 50), 10)

    def timed(fn):
        for _ in range(3):
            fn()
        times = []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(n):
            flush_sum = flush.sum()  # reads 512 MB: evicts the operands, leaves L2 clean
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3)
        times.sort()
        return sum(times) / len(times), times[len(times) // 2]

    x = torch.randn((T, d), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    gain = (1 + 0.1 * torch.randn((d,), generator=g, device=dev, dtype=torch.float32)).to(torch.bfloat16)
    out = torch.empty_like(x)
    n0 = lb.llama_kernel_launch_count()
    us_norm, med_norm = timed(lambda: lb.check(lb.llama_op_rmsnorm(lb.LLAMA_BF16, x, gain, out, T, d, 1e-5, stream)))
    launches = lb.llama_kernel_launch_count() - n0
    norm_bytes = 2.0 * T * d * 2 + d * 2
    del x, out
    qkv = torch.randn((T, (H + 2 * G) * D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    q_out = torch.empty((T, H * D), device=dev, dtype=torch.bfloat16)
    kc = torch.zeros((1, G, T, D), device=dev, dtype=torch.bfloat16)
    vc = torch.zeros((1, G, T, D), device=dev, dtype=torch.bfloat16)
    kv = lb.make_kv_cache(kc, vc, 1, T)
    table = torch.empty((T, D // 2, 2), device=dev, dtype=torch.float32)
    lb.check(lb.llama_op_rope_table(table, T, D, SHAPE["rope_theta"], None, stream))
    n0 = lb.llama_kernel_launch_count()
    us_rope, med_rope = timed(lambda: lb.check(lb.llama_op_rope_kv_write(lb.LLAMA_BF16, qkv, q_out, kv, table, T, 1, T, 0, H, G,
                                                               D, 0, stream)))
    launches += lb.llama_kernel_launch_count() - n0
    rope_bytes = T * (H + 2 * G) * D * 2.0 + T * H * D * 2.0 + 2.0 * T * G * D * 2
    torch.cuda.synchronize()
    return {"rmsnorm_8192x4096": {"us": us_norm, "us_median": med_norm, "gbs": norm_bytes / us_norm / 1e3,
                                  "hbm_frac": norm_bytes / us_norm / 1e3 / hbm, "algorithmic_bytes": norm_bytes},
            "rope_kv_write_b1s8192": {"us": us_rope, "us_median": med_rope, "gbs": rope_bytes / us_rope / 1e3,
                                      "hbm_frac": rope_bytes / us_rope / 1e3 / hbm, "algorithmic_bytes": rope_bytes},
            "hbm_peak_gbs": hbm, "gpu_launches": launches,
            "timing": f"mean of {n} single launches (event durations come in steps of about 2 us), L2 flushed "
                      "before each by reading a 512 MB buffer"}


def bench_stack(lb, torch, dev, stream, args, n_layers=32, vocab=128256, S=8192):
    """32-layer Llama-3-8B-shaped stack prefill, B=1, S=8192, untied LM head (device-generated weights)."""
    s = SHAPE
    d, G = s["d_model"], s["n_kv_heads"]
    D = d // s["n_heads"]
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    layers = [_rand_weights(torch, dev, s, 100 + l) for l in range(n_layers)]
    embed = (torch.randn((vocab, d), generator=g, device=dev, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    head = (torch.randn((vocab, d), generator=g, device=dev, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    fnorm = (1.0 + 0.1 * torch.randn((d,), generator=g, device=dev, dtype=torch.float32)).to(torch.bfloat16)
    cfg = lb.make_config(d, s["n_heads"], G, s["d_ff"], S, s["norm_eps"], s["rope_theta"], lb.LLAMA_BF16)
    st, stk = lb.llama_stack_create(cfg, n_layers, vocab, embed, [lb.make_weights(w) for w in layers], fnorm, head, S)
    lb.check(st, "llama_stack_create")
    del layers, embed, head
    torch.cuda.empty_cache()
    caches = [(torch.zeros((1, G, S, D), dtype=torch.bfloat16, device=dev),
               torch.zeros((1, G, S, D), dtype=torch.bfloat16, device=dev)) for _ in range(n_layers)]
    kvs = [lb.make_kv_cache(k, v, 1, S) for k, v in caches]
    tokens = torch.randint(0, vocab, (1, S), generator=g, device=dev, dtype=torch.int32)
    logits = torch.empty((1, S, vocab), dtype=torch.float32, device=dev)
    for _ in range(3):
        lb.check(lb.llama_stack_forward(stk, tokens, 1, S, 0, kvs, logits, stream))
    steps = 5
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    n0 = lb.llama_kernel_launch_count()
    e0.record(stream)
    for _ in range(steps):
        lb.check(lb.llama_stack_forward(stk, tokens, 1, S, 0, kvs, logits, stream))
    e1.record(stream)
    n_launched = lb.llama_kernel_launch_count() - n0
    torch.cuda.synchronize()
    status = lb.llama_stack_device_status(stk)
    ok = bool(torch.isfinite(logits).all().item())
    ms = e0.elapsed_time(e1) / steps
    lin, att = block_flops(dict(s, S=S))
    total = n_layers * (lin + att) + 2.0 * S * d * vocab
    del caches, kvs, logits
    torch.cuda.empty_cache()
    gen = bench_generate(lb, torch, dev, stream, stk, n_layers, vocab, g)
    lb.llama_stack_destroy(stk)
    return {"workload": "llama3_8b_stack_32l_prefill_b1s8192_vocab128256", "ms_per_step": ms,
            "tokens_per_s": S / (ms / 1e3), "tflops": total / (ms / 1e3) / 1e12, "steps": steps,
            "logits_finite": ok, "device_status": status,
            "gpu_launches": n_launched, "generate": gen}


def bench_generate(lb, torch, dev, stream, stk, n_layers, vocab, g, B=64, start_pos=4064, n_new=32, L=4096):
    """Greedy decoding through the 32-layer stack: B sequences, a one-token prompt at start_pos over caches
    pre-filled with N(0,1) values, n_new tokens chosen on the device (no host round trip per token)."""
    s = SHAPE
    G, D = s["n_kv_heads"], s["d_model"] // s["n_heads"]
    caches = [(torch.randn((B, G, L, D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16),
               torch.randn((B, G, L, D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16))
              for _ in range(n_layers)]
    kvs = [lb.make_kv_cache(k, v, B, L) for k, v in caches]
    prompt = torch.randint(0, vocab, (B, 1), generator=g, device=dev, dtype=torch.int32)
    out = torch.empty((B, n_new), dtype=torch.int32, device=dev)
    logits = torch.empty((B, vocab), dtype=torch.float32, device=dev)
    lb.check(lb.llama_stack_generate(stk, prompt, B, 1, start_pos, n_new, kvs, out, logits, stream))
    torch.cuda.synchronize()
    steps = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = lb.llama_kernel_launch_count()
    e0.record(stream)
    for _ in range(steps):
        lb.check(lb.llama_stack_generate(stk, prompt, B, 1, start_pos, n_new, kvs, out, logits, stream))
    e1.record(stream)
    n_launched = lb.llama_kernel_launch_count() - n0
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    ids = out.cpu()
    return {"workload": f"llama3_8b_stack_32l_greedy_b{B}_pos{start_pos}_new{n_new}_vocab{vocab}",
            "ms_per_call": ms, "ms_per_token_step": ms / n_new, "tokens_per_s": B * n_new / (ms / 1e3),
            "ids_in_range": bool(((ids >= 0) & (ids < vocab)).all().item()), "steps": steps,
            "device_status": lb.llama_stack_device_status(stk), "gpu_launches": n_launched}


def bench_decode(lb, torch, w, dev, stream, args, peaks):
    s = DECODE
    B, d, G = s["B"], s["d_model"], s["n_kv_heads"]
    D = d // s["n_heads"]
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    kc = torch.randn((B, G, s["max_seq_len"], D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    vc = torch.randn((B, G, s["max_seq_len"], D), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    x = torch.randn((B, 1, d), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    y = torch.empty_like(x)
    cfg = lb.make_config(d, s["n_heads"], G, s["d_ff"], s["max_seq_len"], s["norm_eps"], s["rope_theta"],
                         lb.LLAMA_BF16)
    st, blk = lb.llama_block_create(cfg, lb.make_weights(w), B)
    lb.check(st, "llama_block_create (decode)")
    kv = lb.make_kv_cache(kc, vc, B, s["max_seq_len"])
    sp = s["start_pos"]
    for _ in range(args.warmup):
        lb.check(lb.llama_block_forward(blk, x, y, B, 1, sp, kv, stream))
    torch.cuda.synchronize()
    steps = max(min(args.steps, 200), 20)
    # per-step breakdown (events around each kernel), plain launches
    lb.check(lb.llama_block_profile_enable(blk, steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = lb.llama_kernel_launch_count()
    e0.record(stream)
    for _ in range(steps):
        lb.check(lb.llama_block_forward(blk, x, y, B, 1, sp, kv, stream))
    e1.record(stream)
    per_forward = (lb.llama_kernel_launch_count() - n0) // steps
    torch.cuda.synchronize()
    st, launches, total_ms = lb.llama_block_profile_read(blk)
    lb.llama_block_profile_disable(blk)
    us_plain = 1e3 * e0.elapsed_time(e1) / steps
    # the decode step as a CUDA graph (launch-bound inner loop): one captured forward, replayed
    gstream = torch.cuda.Stream(device=dev)

    def graph_us():
        graph = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.stream(gstream):
            lb.check(lb.llama_block_forward(blk, x, y, B, 1, sp, kv, gstream))  # warm the capture stream
            gstream.synchronize()
            with torch.cuda.graph(graph, stream=gstream):
                lb.check(lb.llama_block_forward(blk, x, y, B, 1, sp, kv, gstream))
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return 1e3 * e0.elapsed_time(e1) / steps

    us_kernels = graph_us()
    lb.check(lb.llama_block_device_status(blk))
    # the same step as one cooperative kernel (fused decode mode)
    fused = {"available": False}
    if lb.llama_block_set_decode_mode(blk, lb.LLAMA_DECODE_FUSED) == lb.LLAMA_OK:
        for _ in range(args.warmup):
            lb.check(lb.llama_block_forward(blk, x, y, B, 1, sp, kv, stream))
        torch.cuda.synchronize()
        n0 = lb.llama_kernel_launch_count()
        e0.record(stream)
        for _ in range(steps):
            lb.check(lb.llama_block_forward(blk, x, y, B, 1, sp, kv, stream))
        e1.record(stream)
        fused_per_forward = (lb.llama_kernel_launch_count() - n0) // steps
        torch.cuda.synchronize()
        fused = {"available": True, "us_per_step_plain_launches": 1e3 * e0.elapsed_time(e1) / steps,
                 "kernels_per_step": fused_per_forward}
        try:
            fused["us_per_step"] = graph_us()
        except Exception as ex:  # capture of a cooperative launch refused: plain launches only
            torch.cuda.synchronize()
            fused["graph_error"] = str(ex)[:200]
            fused["us_per_step"] = fused["us_per_step_plain_launches"]
        lb.check(lb.llama_block_device_status(blk))
        lb.check(lb.llama_block_set_decode_mode(blk, lb.LLAMA_DECODE_KERNELS))
    lb.llama_block_destroy(blk)
    us = us_kernels
    att_ms = total_ms[3] / max(launches[3], 1)
    gbs = decode_attention_bytes(s) / (att_ms / 1e3) / 1e9
    hbm = float(peaks["hbm_gbs"])
    weights_bytes = 2.0 * (d * (s["n_heads"] + 2 * G) * D + s["n_heads"] * D * d + 3 * d * s["d_ff"])
    step_bytes = weights_bytes + decode_attention_bytes(s)
    return {"workload": "llama3_8b_block_decode_b64_pos4095", "us_per_step": us, "us_per_step_plain_launches": us_plain,
            "timing": "CUDA graph of one llama_block_forward, replayed; step_us from per-kernel events in plain launches",
            "step_hbm_gbs": step_bytes / (us / 1e6) / 1e9, "step_hbm_frac": step_bytes / (us / 1e6) / 1e9 / hbm,
            "attention_us": 1e3 * att_ms, "attention_gbs": gbs, "attention_hbm_frac": gbs / hbm,
            "hbm_peak_gbs": hbm, "kernels_per_step": per_forward, "gpu_launches": per_forward * steps,
            "fused_kernel": dict(fused, **({"step_hbm_frac": step_bytes / (fused["us_per_step"] / 1e6) / 1e9 / hbm}
                                           if fused.get("us_per_step") else {})),
            "step_us": {lb.llama_profile_step_name(i): 1e3 * total_ms[i] / launches[i]
                        for i in range(len(launches)) if launches[i]}}


if __name__ == "__main__":
    sys.exit(main())
