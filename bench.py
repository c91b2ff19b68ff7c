"""Benchmark of the Hadamard-route prompt path on GB300.

One step = one pass of the pp512 GEMM chain on the rotated 4-bit route: for
each projection of a dense transformer layer (attention 5120 -> 5120, FFN
gate/up 5120 -> 2 x 17408, FFN down 17408 -> 5120) rotate+quantize the 512
tokens' bf16 activations to 4-bit codes, then run the block-scaled W4A4 GEMM
against rotated Q4_0 weights.  Metric: prompt tokens per second.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
        (N > 1: launched by torch.distributed.run, one replica per GPU)

Prints one JSON line (rank 0).  Inputs are synthetic (seeded), resident in HBM
when the timed region starts; two weight/activation sets alternate between
steps so each step's 165 MB of weights and 28 MB of activations exceed the
129 MB L2 and no step reuses the previous step's data from L2.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from hadamard_rotated_bit_gb300 import workloads as wl  # noqa: E402

METRIC = "prompt tokens/s (pp512 GEMM chain) + int-MMA TOPS and act-quant GB/s vs GB300 peak"
UNIT = "tokens/s"
CHAIN = [wl.ATTN, wl.FFN_GATE_UP, wl.FFN_DOWN]
M_TOKENS = 512
WORKLOAD = ("pp512 GEMM chain, rotated 4-bit route: 512 tokens through attention "
            "5120->5120, FFN gate/up 5120->34816, FFN down 17408->5120 "
            "(quantize activations + W4A4 GEMM per projection)")
# operand forms of the chain: "tc" = weights repacked once into tensor-core bytes,
# activations quantized straight into that form; "q4_0" = Q4_0 weights and
# nibble-packed activations consumed directly; "widen" = the Q4_0 weight planes
# widened into tensor-core bytes in shared memory by the GEMM, activations in
# tensor-core form
FORMS = ("tc", "q4_0", "widen")
# the tc GEMMs' workspace argument: None lets the binding split the last wave's
# pieces along K where the schedule gains; --no-split passes False (the
# schedule without the split, for comparison)
TC_WS = None
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
_CSRC = os.path.join(ROOT, "hadamard_rotated_bit_gb300", "csrc")
PROFILE_SUMMARY = {"tc": os.path.join(ROOT, "profiles", "gemm_tc_w4a4_pp512_ffn_gate_up.md"),
                   "q4_0": os.path.join(ROOT, "profiles", "gemm_w4a4_pp512_ffn_gate_up.md"),
                   "widen": os.path.join(ROOT, "profiles",
                                         "gemm_tc_widen_w4a4_pp512_ffn_gate_up.md")}
# the sources a GEMM kernel is compiled from (the profile's traffic is only
# reported while they are unchanged)
GEMM_SOURCES = {"tc": [os.path.join(_CSRC, f) for f in ("h32_gemm_tc.cu", "h32_common.cuh",
                                                        "h32_epilogue.cuh", "h32_tcform.cuh")],
                "q4_0": [os.path.join(_CSRC, f) for f in ("h32_gemm.cu", "h32_common.cuh",
                                                          "h32_epilogue.cuh")]}
GEMM_SOURCES["widen"] = GEMM_SOURCES["tc"]
PEAKS_SUMMARY = os.path.join(ROOT, "profiles", "peaks_gb300.md")
PEAKS_SOURCE = os.path.join(ROOT, "hadamard_rotated_bit_gb300", "peaks", "h32_peaks.cu")
FP32_LANES_PER_SM = 128   # fp32 lanes per SM per clock (the unit count)
# per-SM rates measured on GB300 by the probes of hadamard_rotated_bit_gb300/peaks
# (`bench.py --peaks`), as committed in profiles/peaks_gb300.md; used when that file
# cannot be read
FALLBACK_RATES = {"fp32_mix_lane_ops_per_clock_per_sm": 168.5,
                  "tcgen05_f8f6f4_macs_per_clock_per_sm": 7826.0,
                  "mma_sync_s8_macs_per_clock_per_sm": 252.0}
ISOLATED_REPS = 25        # launches a kernel is timed alone (median), L2 flushed before each


# --------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# --------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """The slowest rank's time: every replica's work counts only when all finished."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# peaks and profile bookkeeping
# --------------------------------------------------------------------------
def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


def load_rates():
    """The per-SM rates the rooflines divide by: fp32 lane operations per clock of
    the epilogue's mul.f32x2 + fma.f32x2 mix, and the MACs per clock of the FP8
    tensor cores (tcgen05) and of the legacy int8 path (mma.sync s8), read from the
    committed probe summary."""
    rates = dict(FALLBACK_RATES)
    try:
        text = open(PEAKS_SUMMARY).read()
    except OSError:
        return rates, "fallback constants in bench.py"
    for k in rates:
        m = re.search(rf"{k}:\s*([0-9.]+)", text)
        if m:
            rates[k] = float(m.group(1))
    return rates, "profiles/peaks_gb300.md (measured with bench.py --peaks)"


def source_sha(paths) -> str:
    """Hash of the code of the given sources, comments and blank lines left out
    (a comment edit does not make a profile's counters stale)."""
    h = hashlib.sha256()
    for path in paths:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(form):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources (else None)."""
    try:
        text = open(PROFILE_SUMMARY[form]).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)\s*\(source sha256/16:\s*([0-9a-f]+)\)",
                  text)
    if not m or m.group(2) != source_sha(GEMM_SOURCES[form]):
        return None
    return float(m.group(1))


# --------------------------------------------------------------------------
# clocks sampled during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="h32clk", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


# --------------------------------------------------------------------------
# the chain on the device
# --------------------------------------------------------------------------
class Chain:
    """Resident inputs, outputs and intermediate buffers of the pp512 chain."""

    def __init__(self, torch, h32, device, sets=2, seed=0, form="tc"):
        self.torch, self.h32, self.device, self.form = torch, h32, device, form
        self.sets = []
        base = []
        for p in CHAIN:
            cid = wl.CFG_ATTN if p is wl.ATTN else wl.CFG_FFN
            w = torch.from_numpy(p.weights(seed, cid)).to(device)
            wq, wd = h32.h32_rotate_quantize_weights_q4_0(w)
            del w
            if form == "tc":   # the offline repack, once per weight matrix
                wq, wd = h32.h32_prepack_weights_q4_0_tc(wq, wd)
            xb = p.activations(M_TOKENS, seed, cid)
            x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(device)
            base.append((wq, wd, x))
        for s in range(sets):
            projs = []
            for (wq, wd, x) in base:
                K = x.shape[1]
                d = {"wq": wq if s == 0 else wq.clone(), "wd": wd if s == 0 else wd.clone(),
                     "x": x if s == 0 else x.clone(),
                     "y": torch.empty((M_TOKENS, wq.shape[0]), dtype=torch.float32, device=device)}
                if form in ("tc", "widen"):
                    d["xq"] = torch.empty((M_TOKENS, K), dtype=torch.uint8, device=device)
                    d["xd"] = torch.zeros((K // 32, M_TOKENS), dtype=torch.float32, device=device)
                else:
                    d["xq"] = torch.empty((M_TOKENS, K // 2), dtype=torch.uint8, device=device)
                    d["xd"] = torch.empty((M_TOKENS, K // 32), dtype=torch.float32, device=device)
                projs.append(d)
            self.sets.append(projs)
        torch.cuda.synchronize()

    def kernel_fn(self, s, k, stream):
        """Kernel k of the chain (2 i = projection i's quantizer, 2 i + 1 its GEMM)
        on input set s, as a callable."""
        h = self.h32
        p = self.sets[s % len(self.sets)][k // 2]
        tc = self.form == "tc"
        if k % 2 == 0:
            if self.form == "widen":
                return lambda: h.h32_quantize_act_q4_tc_e5m2(p["x"], xw=p["xq"], xdt=p["xd"],
                                                             stream=stream)
            if tc:
                return lambda: h.h32_quantize_act_q4_tc(p["x"], xw=p["xq"], xdt=p["xd"],
                                                        stream=stream)
            return lambda: h.h32_quantize_act_q4(p["x"], xq=p["xq"], xd=p["xd"], stream=stream)
        if self.form == "widen":
            return lambda: h.q4_0_x_q4_gemm_tc_widen(p["wq"], p["wd"], p["xq"], p["xd"],
                                                     M=M_TOKENS, y=p["y"], stream=stream)
        if tc:
            return lambda: h.q4_0_x_q4_gemm_tc(p["wq"], p["wd"], p["xq"], p["xd"], M=M_TOKENS,
                                               y=p["y"], stream=stream, workspace=TC_WS)
        return lambda: h.q4_0_x_q4_gemm(p["wq"], p["wd"], p["xq"], p["xd"], y=p["y"],
                                        stream=stream)

    def step(self, s, stream, events=None):
        """Enqueue one chain pass on `stream`; optionally bracket each kernel with events."""
        h = self.h32
        tc = self.form == "tc"
        for i, p in enumerate(self.sets[s % len(self.sets)]):
            if events is not None:
                events[2 * i][0].record(stream)
            if self.form == "widen":
                h.h32_quantize_act_q4_tc_e5m2(p["x"], xw=p["xq"], xdt=p["xd"], stream=stream)
            elif tc:
                h.h32_quantize_act_q4_tc(p["x"], xw=p["xq"], xdt=p["xd"], stream=stream)
            else:
                h.h32_quantize_act_q4(p["x"], xq=p["xq"], xd=p["xd"], stream=stream)
            if events is not None:
                events[2 * i][1].record(stream)
                events[2 * i + 1][0].record(stream)
            if self.form == "widen":
                h.q4_0_x_q4_gemm_tc_widen(p["wq"], p["wd"], p["xq"], p["xd"], M=M_TOKENS,
                                          y=p["y"], stream=stream)
            elif tc:
                h.q4_0_x_q4_gemm_tc(p["wq"], p["wd"], p["xq"], p["xd"], M=M_TOKENS, y=p["y"],
                                    stream=stream, workspace=TC_WS)
            else:
                h.q4_0_x_q4_gemm(p["wq"], p["wd"], p["xq"], p["xd"], y=p["y"], stream=stream)
            if events is not None:
                events[2 * i + 1][1].record(stream)


def kernel_names(form):
    qs = {"tc": "_tc", "q4_0": "", "widen": "_tc_e5m2"}[form]
    gs = {"tc": "_tc", "q4_0": "", "widen": "_tc_widen"}[form]
    names = []
    for p in CHAIN:
        names += [f"h32_quantize_act_q4{qs}[{p.name}]", f"q4_0_x_q4_gemm{gs}[{p.name}]"]
    return names


def algorithmic(p, form="tc", M=M_TOKENS):
    """Per-launch algorithmic work of one projection.  Bytes are the scope table's:
    bf16 in, 4-bit codes (0.5 B) and fp32 scales out for the quantizer (2.625 B an
    element); Q4_0 weights (0.5 B a code, fp16 scales), 4-bit activations and the
    fp32 output for the GEMM.  The tc form stores a code in a byte: its actual
    bytes are the `*_traffic_bytes` (the widening form reads the Q4_0 weights
    themselves and tc-form activations)."""
    N, K = p.N, p.K
    nb = K // 32
    code = 1 if form == "tc" else 0.5          # bytes per stored 4-bit weight code
    wscale = 4 if form == "tc" else 2          # fp32 (tc) or fp16 (Q4_0) weight scales
    xcode = 0.5 if form == "q4_0" else 1       # bytes per stored 4-bit activation code
    return {
        "quant_bytes": int(M * K * 2 + M * K * 0.5 + M * nb * 4),
        "quant_traffic_bytes": int(M * K * 2 + M * K * xcode + M * nb * 4),
        "gemm_alu_ops": 2 * M * N * nb,                            # d_w*d_x and one fma per block
        "gemm_int_ops": 2 * M * N * K,                             # 2 MNK (multiply + add)
        "gemm_bytes": int(N * K * 0.5 + N * nb * 2 + M * K * 0.5 + M * nb * 4 + M * N * 4),
        "gemm_traffic_bytes": int(N * K * code + N * nb * wscale + M * K * xcode + M * nb * 4
                                  + M * N * 4),
    }


def isolated_median_ms(torch, fn, stream, flush, reps=ISOLATED_REPS):
    """Median device time of `fn` over `reps` launches, each after writing a buffer
    of twice the L2 size (so every launch reads its inputs from HBM)."""
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
    stream.synchronize()
    return float(np.median([a.elapsed_time(b) for a, b in evs]))


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(world, "nccl")
    import hadamard_rotated_bit_gb300 as h32
    from hadamard_rotated_bit_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    barrier(dist, device)
    h32.lib()

    chain = Chain(torch, h32, device, form=args.form)
    stream = torch.cuda.Stream(device)
    peaks, peak_src = load_peaks()

    # warm-up
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            chain.step(i, stream)
    stream.synchronize()
    if h32.h32_device_status(stream) != 0:
        raise RuntimeError("device status not OK after warm-up")

    # timed region: device-resident inputs, no events between the kernels (they
    # would keep each kernel from starting under its predecessor's tail)
    nk = 2 * len(CHAIN)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(dist, device)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(args.steps):
            chain.step(i, stream)
        t1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(dist, device)
    elapsed_ms = t0.elapsed_time(t1)
    elapsed_ms = max_over_ranks(dist, elapsed_ms, device)
    status = h32.h32_device_status(stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    tokens = M_TOKENS * args.steps * world
    value = tokens / (elapsed_ms / 1e3)
    ms_per_step = elapsed_ms / args.steps

    # per-kernel device time in the chain: events around every kernel of every step
    # of a second pass of the same chain (same buffers, stream and input sets)
    ev_steps = max(20, min(args.steps, 400))
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(nk)] for _ in range(ev_steps)]
    with torch.cuda.stream(stream):
        for i in range(ev_steps):
            chain.step(i, stream, evs[i])
    stream.synchronize()
    per_kernel = np.array([np.mean([evs[i][k][0].elapsed_time(evs[i][k][1])
                                    for i in range(ev_steps)]) for k in range(nk)])

    # each kernel alone: median of ISOLATED_REPS launches, L2 flushed before each
    props = torch.cuda.get_device_properties(device)
    flush = torch.empty(max(2 * int(getattr(props, "L2_cache_size", 0)), 256 << 20),
                        dtype=torch.uint8, device=device)
    isolated = np.array([isolated_median_ms(torch, chain.kernel_fn(0, k, stream), stream, flush)
                         for k in range(nk)])
    del flush
    if h32.h32_device_status(stream) != 0:
        raise RuntimeError("device status not OK after the per-kernel timing")

    # end to end through host buffers: H2D of the step's activations, the
    # chain, D2H of the step's outputs, all inside the timed region
    e2e = time_e2e(torch, h32, chain, stream, args, dist, device, world)

    # rooflines: the SM count from the device, the per-SM rates measured by the
    # committed probes, the maximum SM clock of the measured peaks
    sms = int(props.multi_processor_count)
    rates, rate_src = load_rates()
    clock_mhz = float(peaks.get("sm_max_mhz", 2070.0))
    ghz = clock_mhz / 1e3
    fp32_peak = sms * rates["fp32_mix_lane_ops_per_clock_per_sm"] * ghz / 1e3   # T lane-ops/s
    fp32_units = sms * FP32_LANES_PER_SM * ghz / 1e3
    fp8_peak = 2 * sms * rates["tcgen05_f8f6f4_macs_per_clock_per_sm"] * ghz / 1e3   # T ops/s
    int8_peak = 2 * sms * rates["mma_sync_s8_macs_per_clock_per_sm"] * ghz / 1e3

    names = kernel_names(args.form)
    dom = int(np.argmax(per_kernel))
    p = CHAIN[dom // 2]
    alg = algorithmic(p, args.form)
    if dom % 2 == 1:
        achieved = alg["gemm_alu_ops"] / (per_kernel[dom] / 1e3) / 1e12
        roofline = {"kernel": names[dom], "bound": "alu", "achieved": round(achieved, 3),
                    "peak": round(fp32_peak, 3), "unit": "T fp32 lane ops/s",
                    "frac": round(achieved / fp32_peak, 4),
                    "traffic": profiled_traffic(args.form),
                    "peak_source": f"{sms} SMs x {rates['fp32_mix_lane_ops_per_clock_per_sm']:.1f} "
                                   f"fp32 lane ops per clock (mul.f32x2 + fma.f32x2, measured, "
                                   f"{rate_src}) x {clock_mhz:.0f} MHz ({peak_src} max SM clock)",
                    "algorithmic_per_launch": alg["gemm_alu_ops"],
                    "ms_per_launch": round(per_kernel[dom], 5),
                    "frac_of_fp32_unit_count": round(achieved / fp32_units, 4),
                    "frac_of_fp8_tensor_measured": round(
                        alg["gemm_int_ops"] / (per_kernel[dom] / 1e3) / 1e12 / fp8_peak, 4)}
    else:
        achieved = alg["quant_bytes"] / (per_kernel[dom] / 1e3) / 1e9
        roofline = {"kernel": names[dom], "bound": "hbm", "achieved": round(achieved, 1),
                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None}

    # every kernel of the chain, in the chain and alone
    kernels = {}
    for i, p in enumerate(CHAIN):
        alg = algorithmic(p, args.form)
        tq, tg = per_kernel[2 * i], per_kernel[2 * i + 1]
        iq, ig = isolated[2 * i], isolated[2 * i + 1]
        kernels[p.name] = {
            "quant_ms_in_chain": round(tq, 5),
            "quant_ms_alone": round(iq, 5),
            "quant_GBps_alone": round(alg["quant_bytes"] / (iq / 1e3) / 1e9, 1),
            "quant_hbm_frac_alone": round(alg["quant_bytes"] / (iq / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
            "quant_algorithmic_bytes": alg["quant_bytes"],
            "quant_traffic_bytes": alg["quant_traffic_bytes"],
            "gemm_ms_in_chain": round(tg, 5),
            "gemm_ms_alone": round(ig, 5),
            "gemm_eff_TOPS": round(alg["gemm_int_ops"] / (tg / 1e3) / 1e12, 1),
            "gemm_frac_of_fp32_measured": round(alg["gemm_alu_ops"] / (tg / 1e3) / 1e12 / fp32_peak, 4),
            "gemm_frac_of_fp32_unit_count": round(alg["gemm_alu_ops"] / (tg / 1e3) / 1e12 / fp32_units, 4),
            "gemm_frac_of_fp8_tensor_measured": round(alg["gemm_int_ops"] / (tg / 1e3) / 1e12 / fp8_peak, 4),
            "gemm_x_int8_mma_sync_measured": round(alg["gemm_int_ops"] / (tg / 1e3) / 1e12 / int8_peak, 3),
        }

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int4 codes (exact products), fp32 epilogue", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": M_TOKENS,
                   "operand_form": args.form,
                   "last_wave_k_split": args.form == "tc" and not args.no_split,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2: two alternating input sets of 193 MB each"},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": nk * args.steps,
        "clocks": clocks,
        "kernels": kernels,
        "kernel_timing": (f"in_chain: mean over {ev_steps} chain steps with events around every "
                          f"kernel (after the timed region); alone: median of {ISOLATED_REPS} "
                          "launches, L2 flushed before each"),
        "peaks": {"fp32_T_lane_ops": round(fp32_peak, 2), "fp32_unit_count_T_lane_ops": round(fp32_units, 2),
                  "fp8_tensor_TOPS": round(fp8_peak, 1), "int8_mma_sync_TOPS": round(int8_peak, 1),
                  "hbm_GBps": peaks["hbm_gbs"], "sms": sms, "hbm_source": peak_src,
                  "rates_source": rate_src},
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_tokens)
    if dist is not None:
        dist.destroy_process_group()
    return line if rank == 0 else None


def time_e2e(torch, h32, chain, stream, args, dist, device, world):
    """The chain end to end from pinned host memory: every step copies its
    activations in and its outputs out inside the timed region.  Steps alternate
    between the two device buffer sets, and the copies run on their own streams
    (one per direction), so step s's copies overlap the compute of its
    neighbours; events order each set's copy-in, compute and copy-out."""
    nsets = len(chain.sets)
    host_x = [p["x"].cpu().pin_memory() for p in chain.sets[0]]
    host_y = [[torch.empty(p["y"].shape, dtype=torch.float32).pin_memory() for p in chain.sets[k]]
              for k in range(nsets)]
    h2d = sum(t.numel() * t.element_size() for t in host_x)
    d2h = sum(t.numel() * t.element_size() for t in host_y[0])
    steps = max(3, min(args.steps, 50))
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    in_done = [ev() for _ in range(nsets)]
    comp_done = [ev() for _ in range(nsets)]
    out_done = [ev() for _ in range(nsets)]
    started = [False] * nsets

    def one(s):
        k = s % nsets
        pset = chain.sets[k]
        with torch.cuda.stream(s_in):
            if started[k]:
                s_in.wait_event(comp_done[k])      # the set's previous compute has read x
            for p, hx in zip(pset, host_x):
                p["x"].copy_(hx, non_blocking=True)
            in_done[k].record(s_in)
        stream.wait_event(in_done[k])
        if started[k]:
            stream.wait_event(out_done[k])         # the set's previous y has been read out
        chain.step(s, stream)
        comp_done[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[k])
            for p, hy in zip(pset, host_y[k]):
                hy.copy_(p["y"], non_blocking=True)
            out_done[k].record(s_out)
        started[k] = True

    for s in range(3):
        one(s)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist, device)
    torch.cuda.synchronize()
    t0.record(stream)
    s_in.wait_event(t0)
    for s in range(steps):
        one(s)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = max_over_ranks(dist, t0.elapsed_time(t1), device)
    return {"value": round(M_TOKENS * steps * world / (ms / 1e3), 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "copies": "pinned host buffers; copy-in and copy-out on their own streams overlap "
                      "the neighbouring steps' compute (two device buffer sets)"}


# --------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline / reference arm)
# --------------------------------------------------------------------------
def oracle_prepare(sample_tokens: int):
    """The oracle's offline step (weights rotated + quantized) and the sampled
    activations; not timed."""
    import oracle
    oracle.build()
    prepared = []
    for p in CHAIN:
        cid = wl.CFG_ATTN if p is wl.ATTN else wl.CFG_FFN
        wq, wd = oracle.quantize_weights_q4_0(p.weights(0, cid))
        x = p.activations(M_TOKENS, 0, cid)[:sample_tokens]
        prepared.append((wq, wd, x, p.K))
    return prepared


def oracle_step(prepared, pool=None, threads=1) -> float:
    """One timed pass of the oracle over the sample: quantize + full GEMM per
    projection.  With `threads` > 1 each GEMM's output columns are split among
    the pool's threads (the C oracle releases the GIL; every output is computed
    by the same function in the same order)."""
    import oracle
    t = time.perf_counter()
    for wq, wd, x, K in prepared:
        xq, xd = oracle.quantize_act_q4(x)
        if threads <= 1:
            oracle.gemm(wq, wd, xq, xd, K)
        else:
            N = wq.shape[0]
            cuts = np.linspace(0, N, threads + 1).astype(int)
            list(pool.map(lambda ab: oracle.gemm(wq[ab[0]:ab[1]], wd[ab[0]:ab[1]], xq, xd, K),
                          [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]))
    return time.perf_counter() - t


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(sample_tokens: int):
    """Time the CPU oracle, as it stands, on a bounded sample of the same
    workload: `sample_tokens` of the 512 tokens through the whole chain
    (quantize + GEMM for all three projections), on one core and on every core
    this process may run on."""
    from concurrent.futures import ThreadPoolExecutor
    prepared = oracle_prepare(sample_tokens)
    cores = host_cores()
    dt1 = oracle_step(prepared)
    with ThreadPoolExecutor(cores) as pool:
        dtn = oracle_step(prepared, pool, cores)
    return {"value": round(sample_tokens / dtn, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "seconds": round(dtn, 2), "value_one_core": round(sample_tokens / dt1, 4),
            "seconds_one_core": round(dt1, 2),
            "sample": f"{sample_tokens} of the 512 tokens through the whole chain "
                      f"(3 quantizations + 3 full GEMMs), C oracle; `value` with each GEMM's "
                      f"output columns split over {cores} threads (all granted cores), "
                      f"`value_one_core` single-threaded"}


REF_BUDGET_S = 120.0   # the reference arm's whole --steps + --warmup run, about


def ref_tokens_for(steps: int, warmup: int, secs_per_token: float) -> int:
    """Tokens per reference step (1 to 16) that keep steps + warmup passes near
    REF_BUDGET_S seconds at the measured time of one token."""
    per_step = REF_BUDGET_S / (max(steps + warmup, 1) * max(secs_per_token, 1e-9))
    return int(max(1, min(16, per_step)))


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores (every granted core),
    each step a bounded sample of the pp512 chain: `--ref-tokens` tokens, or by
    default as many (1 to 16) as keep the whole --steps + --warmup run near
    REF_BUDGET_S seconds, from the time of one calibration step of one token."""
    from concurrent.futures import ThreadPoolExecutor
    rank, world, local = dist_env()
    if rank != 0:
        return None
    cores = host_cores()
    tokens = args.ref_tokens
    with ThreadPoolExecutor(cores) as pool:
        if tokens is None:
            tokens = ref_tokens_for(args.steps, args.warmup,
                                    oracle_step(oracle_prepare(1), pool, cores))
        prepared = oracle_prepare(tokens)
        for _ in range(args.warmup):
            oracle_step(prepared, pool, cores)
        secs = sum(oracle_step(prepared, pool, cores) for _ in range(args.steps))
    value = tokens * args.steps / secs
    sample = (f"{tokens} of the 512 tokens per step through the whole chain "
              f"(3 quantizations + 3 full GEMMs), C oracle, each GEMM's output columns split "
              f"over {cores} threads")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * secs / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int64 block sums, fp32 epilogue",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens_per_step": tokens,
                       "note": "each step is a bounded sample of the pp512 chain"},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_peaks(args):
    """Build and run the rate microbenchmarks (hadamard_rotated_bit_gb300/peaks):
    their JSON lines, as committed in profiles/peaks_gb300.md."""
    out_dir = os.path.join(ROOT, "hadamard_rotated_bit_gb300", "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "h32_peaks")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                    PEAKS_SOURCE], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    if r.returncode != 0:
        raise RuntimeError(f"peak probes failed: {r.stdout}{r.stderr}")
    return lines


def run_only_moe_gemm(args):
    """A small case for profilers: one expert GEMM of the MoE micro-batch
    (1024 tokens, 128 experts, top 8) alone, in the operand form `args.form`
    (tc or widen), `warmup + steps` launches timed with CUDA events."""
    import torch
    import hadamard_rotated_bit_gb300 as h32
    from hadamard_rotated_bit_gb300 import _build
    _build.build()
    dev = torch.device("cuda", 0)
    cfg = wl.MOE
    row_idx, off, _ = wl.moe_routing(cfg)
    x_gu, x_dn = wl.moe_inputs(cfg)
    w_gu, w_dn = wl.moe_weights(cfg)
    up = args.only_gemm == "moe_gate_up"
    x, w = (x_gu, w_gu) if up else (x_dn, w_dn)
    E, N, K = w.shape
    R = int(off[-1])
    wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch.from_numpy(w.reshape(E * N, K)).to(dev))
    xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    ridx = torch.from_numpy(row_idx).to(dev)
    offs = torch.from_numpy(off).to(dev)
    y = torch.empty((R, N), dtype=torch.float32, device=dev)
    if args.form == "widen":
        xw, xdt = (h32.h32_quantize_act_q4_tc_e5m2_gather(xt, ridx) if up
                   else h32.h32_quantize_act_q4_tc_e5m2(xt))

        def gemm():
            h32.q4_0_x_q4_gemm_tc_widen_experts(wq, wd, xw, xdt, offs, N, R=R, y=y)
    elif args.form == "tc":
        wq, wd = h32.h32_prepack_weights_q4_0_tc(wq, wd)
        xw, xdt = h32.h32_quantize_act_q4_tc_gather(xt, ridx) if up else h32.h32_quantize_act_q4_tc(xt)

        def gemm():
            h32.q4_0_x_q4_gemm_tc_experts(wq, wd, xw, xdt, offs, N, R=R, y=y)
    else:
        raise SystemExit("--only-gemm moe_*: --form tc or widen")
    for _ in range(args.warmup):
        gemm()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(args.steps):
        gemm()
    t1.record()
    torch.cuda.synchronize()
    if h32.h32_device_status() != 0:
        raise RuntimeError("device status not OK")
    ms = t0.elapsed_time(t1) / args.steps
    return {"only_gemm": args.only_gemm, "form": args.form, "ms_per_launch": round(ms, 5),
            "eff_TOPS": round(2 * R * N * K / (ms / 1e3) / 1e12, 1),
            "steps": args.steps, "warmup": args.warmup}


def run_only_gemm(args):
    """A small case for profilers: one projection's GEMM alone (resident
    inputs, `warmup + steps` launches), timed with CUDA events."""
    if args.only_gemm.startswith("moe_"):
        return run_only_moe_gemm(args)
    import torch
    import hadamard_rotated_bit_gb300 as h32
    from hadamard_rotated_bit_gb300 import _build
    _build.build()
    p = {q.name: q for q in CHAIN}[args.only_gemm]
    cid = wl.CFG_ATTN if p is wl.ATTN else wl.CFG_FFN
    dev = torch.device("cuda", 0)
    wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch.from_numpy(p.weights(0, cid)).to(dev))
    x = torch.from_numpy(p.activations(M_TOKENS, 0, cid).view(np.int16)).view(torch.bfloat16).to(dev)
    y = torch.empty((M_TOKENS, p.N), dtype=torch.float32, device=dev)
    if args.form == "tc":
        wq, wd = h32.h32_prepack_weights_q4_0_tc(wq, wd)
        xq, xd = h32.h32_quantize_act_q4_tc(x)

        def gemm():
            h32.q4_0_x_q4_gemm_tc(wq, wd, xq, xd, M=M_TOKENS, y=y, workspace=TC_WS)
    elif args.form == "widen":
        xq, xd = h32.h32_quantize_act_q4_tc_e5m2(x)

        def gemm():
            h32.q4_0_x_q4_gemm_tc_widen(wq, wd, xq, xd, M=M_TOKENS, y=y)
    else:
        xq, xd = h32.h32_quantize_act_q4(x)

        def gemm():
            h32.q4_0_x_q4_gemm(wq, wd, xq, xd, y=y)
    for _ in range(args.warmup):
        gemm()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(args.steps):
        gemm()
    t1.record()
    torch.cuda.synchronize()
    if h32.h32_device_status() != 0:
        raise RuntimeError("device status not OK")
    ms = t0.elapsed_time(t1) / args.steps
    alg = algorithmic(p, args.form)
    return {"only_gemm": p.name, "form": args.form, "k_split": args.form == "tc" and not args.no_split,
            "ms_per_launch": round(ms, 5),
            "eff_TOPS": round(alg["gemm_int_ops"] / (ms / 1e3) / 1e12, 1),
            "steps": args.steps, "warmup": args.warmup}


def run_only_quant(args):
    """The activation quantizer alone, streaming a 16384 x 17408 bf16 matrix
    (`warmup + steps` launches, CUDA events)."""
    import torch
    import hadamard_rotated_bit_gb300 as h32
    from hadamard_rotated_bit_gb300 import _build
    _build.build()
    dev = torch.device("cuda", 0)
    M, K = 16384, 17408
    g = torch.Generator(device=dev).manual_seed(0)
    x = torch.randn((M, K), device=dev, generator=g).to(torch.bfloat16)
    kind = args.only_quant
    if kind in ("q4", "q8"):
        out = torch.empty((M, K // 2 if kind == "q4" else K), dtype=torch.uint8, device=dev)
        sc = torch.empty((M, K // 32), dtype=torch.float32, device=dev)
        fn = h32.h32_quantize_act_q4 if kind == "q4" else h32.h32_quantize_act_q8

        def call():
            fn(x, xq=out, xd=sc)
    else:
        out = torch.empty((M, K * (1 if kind == "q4_tc" else 2)), dtype=torch.uint8, device=dev)
        sc = torch.zeros((K // 32, M), dtype=torch.float32, device=dev)
        fn = h32.h32_quantize_act_q4_tc if kind == "q4_tc" else h32.h32_quantize_act_q8_tc

        def call():
            fn(x, xw=out, xdt=sc)
    for _ in range(args.warmup):
        call()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record()
    for _ in range(args.steps):
        call()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    nbytes = M * K * 2 + out.numel() + sc.numel() * 4
    return {"only_quant": kind, "ms_per_launch": round(ms, 5),
            "GBps": round(nbytes / (ms / 1e3) / 1e9, 1), "bytes_per_launch": nbytes,
            "steps": args.steps, "warmup": args.warmup}


# --------------------------------------------------------------------------
# --suite: the other configurations of the path (one JSON line each)
# --------------------------------------------------------------------------
def _events_time(torch, fn, steps, warmup, stream):
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / steps  # ms per call


class Peaks:
    """The roofline denominators of one run: measured HBM copy rate, and the fp32,
    FP8-tensor and mma.sync rates of the committed probes times the SM count and
    the maximum SM clock."""

    def __init__(self, torch, dev):
        hbm, self.hbm_source = load_peaks()
        self.hbm_gbs = float(hbm["hbm_gbs"])
        rates, self.rate_source = load_rates()
        self.sms = int(torch.cuda.get_device_properties(dev).multi_processor_count)
        ghz = float(hbm.get("sm_max_mhz", 2070.0)) / 1e3
        self.fp32 = self.sms * rates["fp32_mix_lane_ops_per_clock_per_sm"] * ghz / 1e3   # T/s
        self.fp8 = 2 * self.sms * rates["tcgen05_f8f6f4_macs_per_clock_per_sm"] * ghz / 1e3

    def fields(self, ms, int_ops=0, alu_ops=0, nbytes=0):
        """Effective rates of `ms` of work and their fractions of the peaks."""
        s = ms / 1e3
        out = {}
        if int_ops:
            out["eff_TOPS"] = round(int_ops / s / 1e12, 1)
            out["frac_of_fp8_tensor"] = round(int_ops / s / 1e12 / self.fp8, 4)
        if alu_ops:
            out["epilogue_T_lane_ops"] = round(alu_ops / s / 1e12, 2)
            out["frac_of_fp32"] = round(alu_ops / s / 1e12 / self.fp32, 4)
        if nbytes:
            out["HBM_GBps"] = round(nbytes / s / 1e9, 1)
            out["frac_of_hbm"] = round(nbytes / s / 1e9 / self.hbm_gbs, 4)
        return out


def chain_work(projs, M, xbits=4):
    """Algorithmic work of one pass of quantize + GEMM over `projs` at M tokens:
    2MNK integer ops, 2MN(K/32) epilogue lane ops, and the scope table's bytes
    (bf16 in, codes + scales out, Q4_0 weights, activation codes, fp32 output)."""
    ints = alu = nbytes = 0
    for p in projs:
        N, K = p.N, p.K
        nb = K // 32
        ints += 2 * M * N * K
        alu += 2 * M * N * nb
        code = 0.5 if xbits == 4 else 1.0
        nbytes += (M * K * 2 + M * K * code + M * nb * 4                      # quantizer
                   + N * K * 0.5 + N * nb * 2 + M * K * code + M * nb * 4 + M * N * 4)   # GEMM
    return int(ints), int(alu), int(nbytes)


def suite_tiny(torch, h32, dev, stream, steps, warmup, pk):
    """The tiny configuration (64 tokens, K = N = 256, fp32 activations with 1% of
    channels x20): quantize + GEMM on the 4-bit and the exact 8-bit routes."""
    p = wl.TINY.chain[0]
    x = torch.from_numpy(p.activations(64, 0, wl.CFG_TINY, bf16=False)).to(dev)
    wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch.from_numpy(p.weights(0, wl.CFG_TINY)).to(dev))
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(wq, wd)
    y = torch.empty((64, p.N), device=dev)
    out = []
    for bits in (4, 8):
        q = h32.h32_quantize_act_q4_tc if bits == 4 else h32.h32_quantize_act_q8_tc
        g = h32.q4_0_x_q4_gemm_tc if bits == 4 else h32.q4_0_x_q8_gemm_tc
        xw = torch.empty((64, p.K * bits // 4), dtype=torch.uint8, device=dev)
        xdt = torch.zeros((p.K // 32, 64), dtype=torch.float32, device=dev)

        def step():
            q(x, xw=xw, xdt=xdt, stream=stream)
            g(wp, wsc, xw, xdt, M=64, y=y, stream=stream, workspace=TC_WS)
        ms_eager = _events_time(torch, step, steps, warmup, stream)
        # the same two launches captured once in a CUDA graph and replayed: the
        # step's device time without the binding's per-call host work between them
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            step()
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            step()
        ms = _events_time(torch, graph.replay, steps, warmup, stream)
        if h32.h32_device_status(stream) != 0:
            raise RuntimeError("device status not OK after the tiny configuration")
        ints, alu, nbytes = chain_work([p], 64, bits)
        nbytes += 64 * p.K * 2   # fp32 activations: twice the bf16 bytes counted
        out.append({"suite": f"tiny_64x256x256_q{bits}", "value": round(64 / (ms / 1e3), 1),
                    "unit": UNIT, "ms_per_step": round(ms, 5),
                    "ms_per_step_eager": round(ms_eager, 5),
                    **pk.fields(ms, ints, alu, nbytes),
                    "note": "quantize + GEMM captured in a CUDA graph and replayed; eager: "
                            "each call through the Python binding"})
    return out


def suite_chain_routes(torch, h32, dev, stream, steps, warmup, pk):
    """The pp512 chain on the exact 8-bit route (tensor-core form and Q4_0-direct),
    on the unrotated 4-bit route (tensor-core form) and on the rotated 4-bit route
    with the Q4_0-direct GEMM and with the GEMM that widens the Q4_0 planes in
    shared memory."""
    out = []
    for route in ("q8_rotated_tc", "q8_rotated_q4_0_direct", "q4_unrotated",
                  "q4_rotated_q4_0_direct", "q4_rotated_widen"):
        rot = route != "q4_unrotated"
        tc = route in ("q4_unrotated", "q8_rotated_tc")
        bufs = []
        for p in CHAIN:
            cid = wl.CFG_ATTN if p is wl.ATTN else wl.CFG_FFN
            wq, wd = h32.h32_rotate_quantize_weights_q4_0(
                torch.from_numpy(p.weights(0, cid)).to(dev), rotate=rot)
            if tc:
                wq, wd = h32.h32_prepack_weights_q4_0_tc(wq, wd)
            x = torch.from_numpy(p.activations(M_TOKENS, 0, cid).view(np.int16)).view(
                torch.bfloat16).to(dev)
            bufs.append((wq, wd, x, torch.empty((M_TOKENS, p.N), device=dev)))

        def step():
            for wq, wd, x, y in bufs:
                if route == "q8_rotated_tc":
                    xw8, xdt = h32.h32_quantize_act_q8_tc(x, rotate=rot, stream=stream)
                    h32.q4_0_x_q8_gemm_tc(wq, wd, xw8, xdt, M=M_TOKENS, y=y, stream=stream,
                                          workspace=TC_WS)
                elif route.startswith("q8"):
                    xq, xd = h32.h32_quantize_act_q8(x, rotate=rot, stream=stream)
                    h32.q4_0_x_q8_gemm(wq, wd, xq, xd, y=y, stream=stream)
                elif tc:
                    xw, xdt = h32.h32_quantize_act_q4_tc(x, rotate=rot, stream=stream)
                    h32.q4_0_x_q4_gemm_tc(wq, wd, xw, xdt, M=M_TOKENS, y=y, stream=stream,
                                          workspace=TC_WS)
                elif route == "q4_rotated_widen":
                    xw, xdt = h32.h32_quantize_act_q4_tc_e5m2(x, rotate=rot, stream=stream)
                    h32.q4_0_x_q4_gemm_tc_widen(wq, wd, xw, xdt, M=M_TOKENS, y=y, stream=stream)
                else:
                    xq, xd = h32.h32_quantize_act_q4(x, rotate=rot, stream=stream)
                    h32.q4_0_x_q4_gemm(wq, wd, xq, xd, y=y, stream=stream)
        ms = _events_time(torch, step, steps, warmup, stream)
        ints, alu, nbytes = chain_work(CHAIN, M_TOKENS, 8 if route.startswith("q8") else 4)
        out.append({"suite": f"pp512_chain_{route}", "value": round(M_TOKENS / (ms / 1e3), 1),
                    "unit": UNIT, "ms_per_step": round(ms, 4), **pk.fields(ms, ints, alu, nbytes)})
        del bufs
    return out


def suite_rotations(torch, h32, dev, stream, steps, warmup):
    """Rotation size A/B on the tensor-core-form 4-bit route: the pp512 chain's
    throughput with no rotation and with 32-, 64- and 128-point rotations, and the
    error of the attention projection's output against the exact fp64 product
    x . W^T on 64 sampled token rows (the accuracy side of the pages' claim)."""
    out = []
    p0 = wl.ATTN
    x_att = p0.activations(M_TOKENS, 0, wl.CFG_ATTN)
    w_att = p0.weights(0, wl.CFG_ATTN)
    rows = np.random.default_rng(4).choice(M_TOKENS, 64, replace=False)
    exact = wl.bf16_bits_to_f32(x_att[rows]).astype(np.float64) @ w_att.astype(np.float64).T
    for rot in (0, 32, 64, 128):
        bufs = []
        for p in CHAIN:
            cid = wl.CFG_ATTN if p is wl.ATTN else wl.CFG_FFN
            wq, wd = h32.h32_rotate_quantize_weights_q4_0(
                torch.from_numpy(p.weights(0, cid)).to(dev), rotate=rot)
            wp, wsc = h32.h32_prepack_weights_q4_0_tc(wq, wd)
            del wq, wd
            x = torch.from_numpy(p.activations(M_TOKENS, 0, cid).view(np.int16)).view(
                torch.bfloat16).to(dev)
            bufs.append((wp, wsc, x, torch.empty((M_TOKENS, p.N), device=dev)))

        def step():
            for wp, wsc, x, y in bufs:
                xw, xdt = h32.h32_quantize_act_q4_tc(x, rotate=rot, stream=stream)
                h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M_TOKENS, y=y, stream=stream,
                                      workspace=TC_WS)
        ms = _events_time(torch, step, steps, warmup, stream)
        y_att = bufs[0][3][torch.from_numpy(rows).to(dev)].cpu().numpy().astype(np.float64)
        rel = float(np.linalg.norm(y_att - exact) / np.linalg.norm(exact))
        out.append({"suite": f"pp512_chain_q4_rotation_{rot}", "value": round(M_TOKENS / (ms / 1e3), 1),
                    "unit": UNIT, "ms_per_step": round(ms, 4),
                    "attn_output_rel_error_vs_exact_fp64": round(rel, 5)})
        del bufs
    return out


def suite_fused_producer(torch, h32, dev, stream, steps, warmup):
    """The attention projection (512 x 5120 x 5120) followed by the quantization of
    its output for the next projection: separately (GEMM writes y, the quantizer
    reads it back) and fused into the GEMM's epilogue (with and without y), next to
    the GEMM alone."""
    p = wl.ATTN
    wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch.from_numpy(p.weights(0, wl.CFG_ATTN)).to(dev))
    wp, wsc = h32.h32_prepack_weights_q4_0_tc(wq, wd)
    x = torch.from_numpy(p.activations(M_TOKENS, 0, wl.CFG_ATTN).view(np.int16)).view(
        torch.bfloat16).to(dev)
    xw, xdt = h32.h32_quantize_act_q4_tc(x)
    y = torch.empty((M_TOKENS, p.N), device=dev)
    xn = torch.empty((M_TOKENS, p.N), dtype=torch.uint8, device=dev)
    xnd = torch.zeros((p.N // 32, M_TOKENS), dtype=torch.float32, device=dev)

    def separate():
        h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M_TOKENS, y=y, stream=stream, workspace=TC_WS)
        h32.h32_quantize_act_q4_tc(y, xw=xn, xdt=xnd, stream=stream)

    def fused_y():
        h32.q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=M_TOKENS, y=y, xw_next=xn,
                                         xdt_next=xnd, stream=stream)

    def fused():
        h32.q4_0_x_q4_gemm_tc_quant_next(wp, wsc, xw, xdt, M=M_TOKENS, want_y=False, xw_next=xn,
                                         xdt_next=xnd, stream=stream)

    def gemm_alone():
        h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=M_TOKENS, y=y, stream=stream, workspace=TC_WS)
    out = {}
    for name, fn in (("gemm_alone", gemm_alone), ("separate", separate), ("fused_with_y", fused_y),
                     ("fused", fused)):
        out[name] = round(_events_time(torch, fn, steps, warmup, stream), 4)
    return [{"suite": "attn_gemm_then_next_quantization_pp512", "unit": "ms", "ms": out,
             "value": out["fused"]}]


def suite_moe(torch, h32, dev, stream, steps, warmup, pk):
    """One 1024-token MoE micro-batch: quantize, expert gate/up GEMM, quantize the
    down input, expert down GEMM (routing, SwiGLU and combine are outside the path)."""
    cfg = wl.MOE
    row_idx, off, _ = wl.moe_routing(cfg)
    x_gu, x_dn = wl.moe_inputs(cfg)
    w_gu, w_dn = wl.moe_weights(cfg)
    R = int(off[-1])

    def prep(w):
        E, N, K = w.shape
        wq, wd = h32.h32_rotate_quantize_weights_q4_0(torch.from_numpy(w.reshape(E * N, K)).to(dev))
        return wq.view(E, N, K // 2), wd.view(E, N, K // 32)
    wq_gu, wd_gu = prep(w_gu)
    wq_dn, wd_dn = prep(w_dn)
    xg = torch.from_numpy(x_gu.view(np.int16)).view(torch.bfloat16).to(dev)
    xn = torch.from_numpy(x_dn.view(np.int16)).view(torch.bfloat16).to(dev)
    ridx = torch.from_numpy(row_idx).to(dev)
    offs = torch.from_numpy(off).to(dev)
    y_gu = torch.empty((R, wq_gu.shape[1]), device=dev)
    y_dn = torch.empty((R, wq_dn.shape[1]), device=dev)
    times = {}

    def step():
        xq, xd = h32.h32_quantize_act_q4(xg, stream=stream)
        h32.q4_0_x_q4_gemm_experts(wq_gu, wd_gu, xq, xd, ridx, offs, R, y=y_gu, stream=stream)
        xq2, xd2 = h32.h32_quantize_act_q4(xn, stream=stream)
        h32.q4_0_x_q4_gemm_experts(wq_dn, wd_dn, xq2, xd2, None, offs, R, y=y_dn, stream=stream)
    ms = _events_time(torch, step, steps, warmup, stream)
    xq, xd = h32.h32_quantize_act_q4(xg, stream=stream)
    times["gate_up_ms"] = _events_time(torch, lambda: h32.q4_0_x_q4_gemm_experts(
        wq_gu, wd_gu, xq, xd, ridx, offs, R, y=y_gu, stream=stream), steps, warmup, stream)
    xq2, xd2 = h32.h32_quantize_act_q4(xn, stream=stream)
    times["down_ms"] = _events_time(torch, lambda: h32.q4_0_x_q4_gemm_experts(
        wq_dn, wd_dn, xq2, xd2, None, offs, R, y=y_dn, stream=stream), steps, warmup, stream)
    ops = 2 * R * (wq_gu.shape[1] * cfg.hidden + wq_dn.shape[1] * cfg.ffn)
    out = [{"suite": "moe_1024_tokens_top8_128_experts_q4_0_direct",
            "value": round(cfg.T / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
            "gemm_ms": {k: round(v, 4) for k, v in times.items()},
            "gemm_eff_TOPS": round(ops / ((times["gate_up_ms"] + times["down_ms"]) / 1e3) / 1e12, 1)}]

    # tensor-core form: repacked experts, the gate/up input quantized straight into
    # grouped order (row gather), the down input already grouped
    N_gu, N_dn = wq_gu.shape[1], wq_dn.shape[1]
    wp_gu, ws_gu = h32.h32_prepack_weights_q4_0_tc(wq_gu.reshape(-1, wq_gu.shape[2]),
                                                    wd_gu.reshape(-1, wd_gu.shape[2]))
    wp_dn, ws_dn = h32.h32_prepack_weights_q4_0_tc(wq_dn.reshape(-1, wq_dn.shape[2]),
                                                    wd_dn.reshape(-1, wd_dn.shape[2]))
    xw_gu = torch.empty((R, cfg.hidden), dtype=torch.uint8, device=dev)
    xt_gu = torch.zeros((cfg.hidden // 32, R), dtype=torch.float32, device=dev)
    xw_dn = torch.empty((R, cfg.ffn), dtype=torch.uint8, device=dev)
    xt_dn = torch.zeros((cfg.ffn // 32, R), dtype=torch.float32, device=dev)

    def step_tc():
        h32.h32_quantize_act_q4_tc_gather(xg, ridx, xw=xw_gu, xdt=xt_gu, stream=stream)
        h32.q4_0_x_q4_gemm_tc_experts(wp_gu, ws_gu, xw_gu, xt_gu, offs, N_gu, R=R, y=y_gu,
                                      stream=stream)
        h32.h32_quantize_act_q4_tc(xn, xw=xw_dn, xdt=xt_dn, stream=stream)
        h32.q4_0_x_q4_gemm_tc_experts(wp_dn, ws_dn, xw_dn, xt_dn, offs, N_dn, R=R, y=y_dn,
                                      stream=stream)
    ms = _events_time(torch, step_tc, steps, warmup, stream)
    tt = {"gate_up_ms": _events_time(torch, lambda: h32.q4_0_x_q4_gemm_tc_experts(
              wp_gu, ws_gu, xw_gu, xt_gu, offs, N_gu, R=R, y=y_gu, stream=stream), steps, warmup,
              stream),
          "down_ms": _events_time(torch, lambda: h32.q4_0_x_q4_gemm_tc_experts(
              wp_dn, ws_dn, xw_dn, xt_dn, offs, N_dn, R=R, y=y_dn, stream=stream), steps, warmup,
              stream)}
    E = cfg.E
    moe_alu = 2 * R * (N_gu * (cfg.hidden // 32) + N_dn * (cfg.ffn // 32))
    moe_bytes = int(E * (N_gu * cfg.hidden + N_dn * cfg.ffn) * 0.5625        # Q4_0 experts
                    + cfg.T * cfg.hidden * 2 + R * cfg.ffn * 2                # bf16 inputs
                    + 2 * R * (cfg.hidden + cfg.ffn) * 0.625                  # codes + scales, out and in
                    + R * (N_gu + N_dn) * 4)                                  # fp32 outputs
    out.append({"suite": "moe_1024_tokens_top8_128_experts",
                "value": round(cfg.T / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
                "operand_form": "tc", "gemm_ms": {k: round(v, 4) for k, v in tt.items()},
                "gemm_eff_TOPS": round(ops / ((tt["gate_up_ms"] + tt["down_ms"]) / 1e3) / 1e12, 1),
                "weight_bytes": int(E * (N_gu * cfg.hidden + N_dn * cfg.ffn) * 1.125),
                **pk.fields(ms, ops, moe_alu, moe_bytes)})

    # the same expert GEMMs on the experts' Q4_0 planes themselves, widened into
    # tensor-core bytes in shared memory (half the weight bytes of the repacked form)
    wq_gu2, wd_gu2 = wq_gu.reshape(-1, wq_gu.shape[2]), wd_gu.reshape(-1, wd_gu.shape[2])
    wq_dn2, wd_dn2 = wq_dn.reshape(-1, wq_dn.shape[2]), wd_dn.reshape(-1, wd_dn.shape[2])

    def gu_widen():
        h32.q4_0_x_q4_gemm_tc_widen_experts(wq_gu2, wd_gu2, xw_gu, xt_gu, offs, N_gu, R=R,
                                            y=y_gu, stream=stream)

    def dn_widen():
        h32.q4_0_x_q4_gemm_tc_widen_experts(wq_dn2, wd_dn2, xw_dn, xt_dn, offs, N_dn, R=R,
                                            y=y_dn, stream=stream)

    def step_widen():
        h32.h32_quantize_act_q4_tc_e5m2_gather(xg, ridx, xw=xw_gu, xdt=xt_gu, stream=stream)
        gu_widen()
        h32.h32_quantize_act_q4_tc_e5m2(xn, xw=xw_dn, xdt=xt_dn, stream=stream)
        dn_widen()
    ms = _events_time(torch, step_widen, steps, warmup, stream)   # leaves xw_* in e5m2 form
    tw = {"gate_up_ms": _events_time(torch, gu_widen, steps, warmup, stream),
          "down_ms": _events_time(torch, dn_widen, steps, warmup, stream)}
    out.append({"suite": "moe_1024_tokens_top8_128_experts_widen",
                "value": round(cfg.T / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
                "operand_form": "widen", "gemm_ms": {k: round(v, 4) for k, v in tw.items()},
                "gemm_eff_TOPS": round(ops / ((tw["gate_up_ms"] + tw["down_ms"]) / 1e3) / 1e12, 1),
                "weight_bytes": int(E * (N_gu * cfg.hidden + N_dn * cfg.ffn) * 0.5625),
                **pk.fields(ms, ops, moe_alu, moe_bytes)})

    # the whole expert layer on the GPU: the router (top 8 of the logits, their
    # weights, the grouped order), the tc-form expert GEMMs on that order and the
    # weighted combine back to token order (SwiGLU stays outside the path)
    lg = torch.from_numpy(wl.moe_logits(cfg)).to(dev)
    ids, tw, offs_r, ridx_r, row_of = h32.h32_moe_route(lg, cfg.top_k, stream=stream)
    out_t = torch.empty((cfg.T, N_dn), dtype=torch.float32, device=dev)

    def route():
        h32.h32_moe_route(lg, cfg.top_k, topk_id=ids, topk_w=tw, expert_off=offs_r,
                          row_idx=ridx_r, row_of=row_of, stream=stream)

    def combine():
        h32.h32_moe_combine(y_dn, row_of, tw, out=out_t, stream=stream)

    def step_layer():
        route()
        h32.h32_quantize_act_q4_tc_gather(xg, ridx_r, xw=xw_gu, xdt=xt_gu, stream=stream)
        h32.q4_0_x_q4_gemm_tc_experts(wp_gu, ws_gu, xw_gu, xt_gu, offs_r, N_gu, R=R, y=y_gu,
                                      stream=stream)
        h32.h32_quantize_act_q4_tc(xn, xw=xw_dn, xdt=xt_dn, stream=stream)
        h32.q4_0_x_q4_gemm_tc_experts(wp_dn, ws_dn, xw_dn, xt_dn, offs_r, N_dn, R=R, y=y_dn,
                                      stream=stream)
        combine()
    ms = _events_time(torch, step_layer, steps, warmup, stream)
    # the router's and the combine's device time inside the layer: events around
    # them on every step of a second pass (a call timed alone in a loop would
    # measure the host's launch rate, not the kernels)
    evs = []
    with torch.cuda.stream(stream):
        for i in range(warmup + steps):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(stream)
            route()
            e[1].record(stream)
            h32.h32_quantize_act_q4_tc_gather(xg, ridx_r, xw=xw_gu, xdt=xt_gu, stream=stream)
            h32.q4_0_x_q4_gemm_tc_experts(wp_gu, ws_gu, xw_gu, xt_gu, offs_r, N_gu, R=R, y=y_gu,
                                          stream=stream)
            h32.h32_quantize_act_q4_tc(xn, xw=xw_dn, xdt=xt_dn, stream=stream)
            h32.q4_0_x_q4_gemm_tc_experts(wp_dn, ws_dn, xw_dn, xt_dn, offs_r, N_dn, R=R, y=y_dn,
                                          stream=stream)
            e[2].record(stream)
            combine()
            e[3].record(stream)
            if i >= warmup:
                evs.append(e)
    stream.synchronize()
    t_route = sum(e[0].elapsed_time(e[1]) for e in evs) / len(evs)
    t_comb = sum(e[2].elapsed_time(e[3]) for e in evs) / len(evs)
    comb_bytes = R * N_dn * 4 + cfg.T * N_dn * 4 + R * 8
    out.append({"suite": "moe_layer_1024_tokens_route_experts_combine",
                "value": round(cfg.T / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 4),
                "operand_form": "tc", "route_ms": round(t_route, 4), "combine_ms": round(t_comb, 4),
                "combine_GBps": round(comb_bytes / (t_comb / 1e3) / 1e9, 1),
                "combine_note": "grouped rows L2-resident, as right after the down GEMM"})
    return out


def suite_long(torch, h32, dev, stream, steps, warmup, pk):
    """The chain on long prompts, in 1024-token micro-batches."""
    out = []
    projs = [wl.LONG_ATTN, wl.LONG_GATE_UP, wl.LONG_DOWN]
    weights = []
    for p in projs:
        wq, wd = h32.h32_rotate_quantize_weights_q4_0(
            torch.from_numpy(p.weights(0, wl.CFG_LONG)).to(dev))
        weights.append(h32.h32_prepack_weights_q4_0_tc(wq, wd))
        del wq, wd
    mb = 1024
    for M in wl.LONG_MS:
        xs = [torch.from_numpy(p.activations(M, 0, wl.CFG_LONG).view(np.int16)).view(
            torch.bfloat16).to(dev) for p in projs]
        ys = [torch.empty((mb, p.N), device=dev) for p in projs]

        def step():
            for s0 in range(0, M, mb):
                m = min(mb, M - s0)
                for (wp, wsc), x, y in zip(weights, xs, ys):
                    xw, xdt = h32.h32_quantize_act_q4_tc(x[s0:s0 + m], stream=stream)
                    h32.q4_0_x_q4_gemm_tc(wp, wsc, xw, xdt, M=m, y=y[:m], stream=stream,
                                          workspace=TC_WS)
        ms = _events_time(torch, step, max(1, steps // max(1, M // 1024)), max(1, warmup // 4),
                          stream)
        ints, alu, nbytes = 0, 0, 0
        for s0 in range(0, M, mb):
            i_, a_, b_ = chain_work(projs, min(mb, M - s0))
            ints, alu, nbytes = ints + i_, alu + a_, nbytes + b_
        out.append({"suite": f"long_prompt_{M}_tokens_1024_microbatches",
                    "value": round(M / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms, 3),
                    **pk.fields(ms, ints, alu, nbytes)})
        del xs, ys
    return out


def suite_quant_stream(torch, h32, dev, stream, steps, warmup, peaks):
    """The rotate+quantize kernel streaming a large activation matrix (16384 x 17408 bf16)."""
    M, K = 16384, 17408
    g = torch.Generator(device=dev).manual_seed(0)
    x = torch.randn((M, K), device=dev, generator=g).to(torch.bfloat16)
    out = []
    for bits in (4, 8):
        xq = torch.empty((M, K // 2 if bits == 4 else K), dtype=torch.uint8, device=dev)
        xd = torch.empty((M, K // 32), dtype=torch.float32, device=dev)
        fn = h32.h32_quantize_act_q4 if bits == 4 else h32.h32_quantize_act_q8
        ms = _events_time(torch, lambda: fn(x, xq=xq, xd=xd, stream=stream), steps, warmup, stream)
        nbytes = M * K * 2 + xq.numel() + xd.numel() * 4
        gbs = nbytes / (ms / 1e3) / 1e9
        out.append({"suite": f"quantize_q{bits}_stream_16384x17408_bf16", "value": round(gbs, 1),
                    "unit": "GB/s", "ms_per_call": round(ms, 4),
                    "hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "bytes_per_call": nbytes})
    # the tensor-core form: one byte (4-bit) or two bytes (8-bit) per code,
    # scales block-major
    for bits in (4, 8):
        xw = torch.empty((M, K * (bits // 4)), dtype=torch.uint8, device=dev)
        xdt = torch.zeros((K // 32, M), dtype=torch.float32, device=dev)
        fn = h32.h32_quantize_act_q4_tc if bits == 4 else h32.h32_quantize_act_q8_tc
        ms = _events_time(torch, lambda: fn(x, xw=xw, xdt=xdt, stream=stream), steps, warmup, stream)
        nbytes = M * K * 2 + xw.numel() + xdt.numel() * 4
        gbs = nbytes / (ms / 1e3) / 1e9
        out.append({"suite": f"quantize_q{bits}_tc_stream_16384x17408_bf16", "value": round(gbs, 1),
                    "unit": "GB/s", "ms_per_call": round(ms, 4),
                    "hbm_frac": round(gbs / peaks["hbm_gbs"], 4), "bytes_per_call": nbytes})
    return out


def run_suite(args, only_moe=False):
    import torch
    import hadamard_rotated_bit_gb300 as h32
    from hadamard_rotated_bit_gb300 import _build
    _build.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    peaks, _ = load_peaks()
    pk = Peaks(torch, dev)
    steps, warmup = args.steps, args.warmup
    lines = [{"suite": "peaks", "fp32_T_lane_ops": round(pk.fp32, 2), "fp8_tensor_TOPS": round(pk.fp8, 1),
              "hbm_GBps": pk.hbm_gbs, "sms": pk.sms, "hbm_source": pk.hbm_source,
              "rates_source": pk.rate_source}]
    if only_moe:
        lines += suite_moe(torch, h32, dev, stream, steps, warmup, pk)
        if h32.h32_device_status(stream) != 0:
            raise RuntimeError("device status not OK after the MoE lines")
        return lines
    lines += suite_tiny(torch, h32, dev, stream, steps, warmup, pk)
    lines += suite_quant_stream(torch, h32, dev, stream, steps, warmup, peaks)
    lines += suite_chain_routes(torch, h32, dev, stream, steps, warmup, pk)
    lines += suite_rotations(torch, h32, dev, stream, steps, warmup)
    lines += suite_fused_producer(torch, h32, dev, stream, steps, warmup)
    lines += suite_moe(torch, h32, dev, stream, steps, warmup, pk)
    lines += suite_long(torch, h32, dev, stream, steps, warmup, pk)
    if h32.h32_device_status(stream) != 0:
        raise RuntimeError("device status not OK after the suite")
    return lines


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["h32", "reference"], default="h32")
    ap.add_argument("--form", choices=list(FORMS), default="tc",
                    help="operand form of the chain (default: tensor-core form)")
    ap.add_argument("--cpu-tokens", type=int, default=24)
    ap.add_argument("--ref-tokens", type=int, default=None,
                    help="tokens per reference step (default: sized so that the whole "
                         "reference run takes about two minutes)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-split", action="store_true",
                    help="tc GEMMs without the K split of the last wave (schedule comparison)")
    ap.add_argument("--suite", action="store_true",
                    help="measure the other configurations (8-bit and unrotated routes, MoE, "
                         "long prompts, streaming quantizer), one JSON line each")
    ap.add_argument("--only-gemm", choices=[p.name for p in CHAIN] + ["moe_gate_up", "moe_down"],
                    default=None,
                    help="time one projection's GEMM alone (a small case for profilers)")
    ap.add_argument("--only-quant", choices=["q4", "q8", "q4_tc", "q8_tc"], default=None,
                    help="time the activation quantizer alone on a 16384 x 17408 bf16 matrix "
                         "(a streaming case for profilers)")
    ap.add_argument("--peaks", action="store_true",
                    help="run the rate microbenchmarks behind the rooflines (fp32 pipe, tensor "
                         "cores, TMEM, shared memory, mbarrier), one JSON line each")
    ap.add_argument("--only-moe", action="store_true",
                    help="the MoE micro-batch lines of --suite alone (expert GEMMs, and the "
                         "whole layer with the router and the combine)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    global TC_WS
    TC_WS = False if args.no_split else None
    if args.peaks:
        for ln in run_peaks(args):
            print(json.dumps(ln), flush=True)
        return
    if args.suite or args.only_moe:
        for ln in run_suite(args, only_moe=args.only_moe):
            print(json.dumps(ln), flush=True)
        return
    if args.only_gemm:
        line = run_only_gemm(args)
    elif args.only_quant:
        line = run_only_quant(args)
    elif args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
