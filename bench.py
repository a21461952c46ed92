#!/usr/bin/env python3
"""Benchmark of the routed-expert FFN layer on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|verify|small|prefill|tiny]

A step is one pass of the whole layer (router, top-k, bucketing, gate/up,
SwiGLU, down, shared expert, combine) over every layer of the workload, each
layer on its own synthetic batch: for the default ``decode`` workload that is
36 independent gpt-oss-120B-shaped MoE layers (T=1, d=ffn=2880, E=128, k=4,
MXFP4 experts) back to back. The metric is MoE-layer tokens per second
(T * layers * steps / time) with the achieved HBM GB/s over the algorithmic
bytes beside it.

``--impl ours`` (default): inputs resident in HBM, the layers captured in one
CUDA graph, K timed replays between CUDA events after W warm-up replays. The
weights a step touches exceed the 129 MB L2, so no flush is needed. Also
reported: the per-kernel roofline of the dominant kernel (CUDA events the
library records at its phase boundaries), an end-to-end number through the
host-buffer entry point, the CPU oracle on a bounded sample, and SM clocks
sampled during the timed region.

``--impl reference``: the CPU oracle (plain fp64 C) as the reference arm on
all host cores (one single-token layer evaluation per core and step).

By default the line carries, besides the main workload (``--workload``,
default decode), the other three full-size workloads under ``workloads``
(``--extra-workloads``), each with its own timing, roofline and e2e, and the
measured rate of the block-scaled MMA kind the expert GEMMs issue.

Under torchrun each rank runs its own replica of the workload on its own GPU
(independent batches, no collective on the data path); rank 0 prints the
whole-job number (units of all ranks over the slowest rank's time).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import re
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE layer tokens/s (achieved HBM GB/s alongside)"
UNIT = "tokens/s"


# ---------------------------------------------------------------- algorithmic work (per layer)

def expert_bytes(wl: synth.Workload, f: int | None = None) -> int:
    """Stored bytes of one expert of ffn f in the workload's format (MXFP4 or affine group-64)."""
    return wl.affine_bytes(f) if wl.affine_bits else wl.expert_bytes(f)


def layer_bytes(wl: synth.Workload, U: int, T: int) -> int:
    """Bytes the method must move for one layer call: the U distinct routed experts
    (+ the shared expert), router weights (+ bias), x in and y out (bf16)."""
    b = U * expert_bytes(wl) + wl.E * wl.d * 4 + 2 * T * wl.d + 2 * T * wl.d
    if wl.shared_ffn:
        b += expert_bytes(wl, wl.shared_ffn)
    if wl.zipf_bias:
        b += 4 * wl.E
    return b


def phase_bytes(wl: synth.Workload, U: int, T: int) -> dict:
    d, F, S = wl.d, wl.ffn, wl.shared_ffn
    # gate/up holds 2/3 of an expert's bytes, down 1/3, in either format
    gu = U * 2 * expert_bytes(wl) // 3 + (2 * expert_bytes(wl, S) // 3 if S else 0) + 2 * T * d
    dn = U * expert_bytes(wl) // 3 + (expert_bytes(wl, S) // 3 if S else 0)
    route = wl.E * d * 4 + (4 * wl.E if wl.zipf_bias else 0) + 2 * T * d
    # "layer" is the fused single-kernel path (T <= 16): every byte of the layer in one launch;
    # "panels" (tcgen05 path) reads x once
    return {"route": route, "panels": 2 * T * d, "gateup": gu, "down": dn, "combine": 2 * T * d,
            "layer": layer_bytes(wl, U, T)}


def layer_flops(wl: synth.Workload, T: int) -> int:
    return 2 * T * wl.E * wl.d + 2 * T * wl.k * 3 * wl.d * wl.ffn + 2 * T * 3 * wl.d * wl.shared_ffn


def phase_flops(wl: synth.Workload, T: int) -> dict:
    """Algorithmic flops of the phases: the router, the gate/up and down GEMMs (2 flops per multiply-add)."""
    P = T * wl.k
    gu = 2 * P * 2 * wl.ffn * wl.d + 2 * T * 2 * wl.shared_ffn * wl.d
    dn = 2 * P * wl.ffn * wl.d + 2 * T * wl.shared_ffn * wl.d
    return {"route": 2 * T * wl.E * wl.d, "gateup": gu, "down": dn, "layer": layer_flops(wl, T)}


# dense FP4 / FP8 tensor rates of the GB300 (nominal 13.5 and 4.5 PFLOP/s): the FP4 peak is the
# measured rate of the FP8-rate MMA kind times this ratio
FP4_OVER_FP8 = 3.0


# ---------------------------------------------------------------- clocks (NVML via ctypes; nvidia-smi fallback)

class ClockSampler:
    """Samples SM clock and throttle reasons on a thread while running."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap",
               0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle", 0x2: "applications_clocks_setting"}

    def __init__(self, device_index: int, interval_s: float = 0.002):
        self.dev = device_index
        self.interval = interval_s
        self.samples: list[tuple[int, int]] = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._th = None
        self._nvml = None
        self._h = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(h)) == 0:
                    self._nvml, self._h = nv, h
                    mx = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM = 1
                        self.max_mhz = mx.value
        except OSError:
            self._nvml = None

    def _sample(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        nv, h = self._nvml, self._h
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(self.interval)

    def start(self):
        if self._nvml is not None:
            self._th = threading.Thread(target=self._sample, daemon=True)
            self._th.start()

    def stop(self) -> dict:
        if self._th is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable: NVML not loadable"]}
        self._stop.set()
        self._th.join()
        mhz = [s[0] for s in self.samples]
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ---------------------------------------------------------------- helpers

# moe_forward_host writes y in place into a page-locked mapped buffer, and reads x in place too for
# single-launch calls on at most this many bytes of x (include/moe.h)
MAPPED_X_BYTES = 16384


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


_COMMENT_OR_STRING = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'', re.S)


def code_text(src: str) -> str:
    """C/CUDA source with its comments removed and whitespace collapsed (string and character
    literals kept): what the compiler sees of it, so comment-only edits keep a capture's key."""
    out = _COMMENT_OR_STRING.sub(lambda mt: " " if mt.group(0)[0] == "/" else mt.group(0), src)
    return " ".join(out.split())


def kernel_source_hash(sources) -> str:
    """Hash of the code of the files (repo-relative paths) that one kernel is compiled from."""
    h = hashlib.sha256()
    for rel in sorted(sources):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(rel.encode() + b"\0" + code_text(f.read()).encode() + b"\0")
    return h.hexdigest()[:16]


def ncu_traffic(phase: str, workload: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on the current code of the
    kernel's translation unit (its .cu file and the headers it includes, listed with the entry)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(workload, {}).get(phase)
    if not ent or not ent.get("sources") or ent.get("source_hash") != kernel_source_hash(ent["sources"]):
        return None
    return ent.get("dram_bytes_per_launch")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(ws: int, units_per_rank: int, seconds_max: float) -> float:
    """Units of every rank over the slowest rank's time (weak scaling: each rank has its own batch)."""
    return ws * units_per_rank / seconds_max


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def rank_x(wl: synth.Workload, layer: int, rank: int) -> np.ndarray:
    """x of one layer for one rank (rank 0 uses the layer's own x)."""
    seed = wl.seed(layer) if rank == 0 else wl.seed(layer) + 1_000_003 * rank
    return synth.gen_x(seed, wl.T, wl.d)


# ---------------------------------------------------------------- CPU oracle timing

def oracle_sample(wl: synth.Workload, budget_s: float, max_rounds: int, threads: int, first_round: int = 0):
    """Time the CPU oracle, as it stands, on whole-layer evaluations of single tokens of the
    workload's layer 0 (router over all experts, top-k, the k experts, the shared expert,
    combine; fp64), `threads` tokens per round on `threads` host threads, until budget_s of
    wall time is spent or max_rounds rounds ran. Each token is a fresh seeded draw from the
    workload's x distribution; the layer's weights are generated once, outside the timed region."""
    import oracle
    L = synth.gen_layer(wl, 0, T=1)
    done, spent, rounds = 0, 0.0, 0
    for r in range(max_rounds):
        x = synth.gen_x(wl.seed(0) + 7_919 * (first_round + r + 1), threads, wl.d)
        t0 = time.perf_counter()
        oracle.layer_tokens_parallel(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, x, L["w_router"], L["bias"],
                                     L["codes"], L["scales"], threads=threads)
        spent += time.perf_counter() - t0
        done += threads
        rounds += 1
        if spent >= budget_s:
            break
    return done, spent, rounds


def cpu_sample_text(wl: synth.Workload, n: int, spent: float, threads: int) -> str:
    return (f"{n} whole-layer evaluations of single tokens (fresh seeded x) through layer 0 of the '{wl.name}' "
            f"workload (router over all {wl.E} experts, top-{wl.k}, the selected experts"
            f"{', the shared expert' if wl.shared_ffn else ''}, combine; fp64), {threads} tokens at a time on "
            f"{threads} host threads, {spent:.1f} s")


# ---------------------------------------------------------------- reference arm

def run_reference(args, wl):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    threads = oracle.host_threads()
    for i in range(args.warmup):
        oracle_sample(wl, 0.0, 1, threads, first_round=i)
    times = []
    n_tot = 0
    for i in range(args.steps):
        n, spent, _ = oracle_sample(wl, 0.0, 1, threads, first_round=args.warmup + i)
        times.append(spent)
        n_tot += n
    total = sum(times)
    value = n_tot / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "per step: " + cpu_sample_text(wl, threads, total / args.steps, threads)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(wl: synth.Workload, args, layers: int | None = None) -> dict:
    nl = args.layers if layers is None else layers
    return {"workload": f"{wl.name}: MoE layer T={wl.T}, d={wl.d}, ffn={wl.ffn}, E={wl.E}, k={wl.k}, "
                        f"shared_ffn={wl.shared_ffn}, zipf_bias={wl.zipf_bias}, layers={nl}, "
                        + (f"{wl.affine_bits}-bit affine group-64 experts" if wl.affine_bits else "MXFP4 experts"),
            "T": wl.T, "d": wl.d, "ffn": wl.ffn, "n_experts": wl.E, "top_k": wl.k, "shared_ffn": wl.shared_ffn,
            "layers": nl, "zipf_bias": wl.zipf_bias, "parallelism": f"replica x{args.gpus}",
            "l2": "inputs larger than L2: each step streams every layer's routed experts from HBM; no flush"}


# ---------------------------------------------------------------- our arm

def measure_workload(args, wl: synth.Workload, nl: int, m, torch, ws: int, rank: int, local: int,
                     peaks: dict) -> dict:
    """All layers of one workload resident; graph-timed value, per-phase roofline, e2e."""
    T = wl.T
    if wl.affine_bits:
        shape = m.LayerShape(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, t_max=T, flags=args.flags & ~4,
                             weight_format=m.MOE_FORMAT_AFFINE64, weight_bits=wl.affine_bits)
        codes_h = torch.empty((wl.total_affine_bytes,), dtype=torch.uint8, pin_memory=True)
        scales_h = None
    else:
        shape = m.LayerShape(wl.d, wl.ffn, wl.E, wl.k, wl.shared_ffn, t_max=T, flags=args.flags)
        codes_h = torch.empty((wl.total_code_bytes,), dtype=torch.uint8, pin_memory=True)
        scales_h = torch.empty((wl.total_scale_bytes,), dtype=torch.uint8, pin_memory=True)
    layers, xs, outs, xh, oh = [], [], [], [], []
    t_gen = time.perf_counter()
    for l in range(nl):
        L = synth.gen_layer(wl, l, with_experts=False)
        lay = m.MoeLayer(shape, device=local)
        if wl.affine_bits:
            synth.gen_experts_affine(wl, wl.seed(l), codes_h.numpy())
            lay.load_affine(L["w_router"], L["bias"], codes_h)
        else:
            synth.gen_experts(wl, wl.seed(l), codes_h.numpy(), scales_h.numpy())
            lay.load(L["w_router"], L["bias"], codes_h, scales_h)
        layers.append(lay)
        x = rank_x(wl, l, rank)
        xh.append(torch.from_numpy(x.view(np.int16).copy()).pin_memory())
        xs.append(xh[-1].cuda())
        outs.append(torch.empty((T, wl.d), dtype=torch.bfloat16, device="cuda"))
        oh.append(torch.empty((T, wl.d), dtype=torch.int16, pin_memory=True))
    del codes_h, scales_h
    t_gen = time.perf_counter() - t_gen
    stream = torch.cuda.Stream()

    # routing of every layer (distinct experts U -> algorithmic bytes)
    counts = torch.empty((wl.E,), dtype=torch.int32, device="cuda")
    U = []
    with torch.cuda.stream(stream):
        for l in range(nl):
            layers[l].forward(xs[l], T, outs[l], stream)
            layers[l].routing(counts=counts, stream=stream)
            stream.synchronize()
            U.append(int((counts > 0).sum().item()))
    bytes_step = sum(layer_bytes(wl, u, T) for u in U)
    flops_step = nl * layer_flops(wl, T)

    # device-resident timing: the layers in one CUDA graph
    with torch.cuda.stream(stream):
        for _ in range(2):
            for l in range(nl):
                layers[l].forward(xs[l], T, outs[l], stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for l in range(nl):
            layers[l].forward(xs[l], T, outs[l], stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()
    bad = [lay.status() for lay in layers]
    if any(bad):
        raise RuntimeError(f"{wl.name}: device status after warm-up: {bad[:4]}... (a bounded device wait gave up)")
    clocks = ClockSampler(local)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(ws)
    ms_local = e0.elapsed_time(e1) / args.steps
    ms = reduce_max(ms_local, ws)
    value = whole_job_value(ws, T * nl, ms / 1000.0)
    status = max(lay.status() for lay in layers)
    del graph

    # per-kernel timing: the library records events at its phase boundaries
    phases = m.moe_forward_phases(layers[0].ctx, T)
    ksteps = max(1, args.kernel_steps)
    ev = [[[torch.cuda.Event(enable_timing=True) for _ in range(len(phases) + 1)] for _ in range(nl)]
          for _ in range(ksteps)]
    with torch.cuda.stream(stream):
        for s_ev in ev:  # torch creates the CUDA event at its first record
            for l_ev in s_ev:
                for e_ in l_ev:
                    e_.record(stream)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for s in range(ksteps):
            for l in range(nl):
                m.moe_profile_events(layers[l].ctx, ev[s][l])
                layers[l].forward(xs[l], T, outs[l], stream)
        for l in range(nl):
            m.moe_profile_events(layers[l].ctx, None)
    torch.cuda.synchronize()
    ph_ms = {p: 0.0 for p in phases}
    for s in range(ksteps):
        for l in range(nl):
            for i, p in enumerate(phases):
                ph_ms[p] += ev[s][l][i].elapsed_time(ev[s][l][i + 1])
    ph_bytes = {p: 0 for p in phases}
    ph_flops = {p: 0 for p in phases}
    for u in U:
        pb = phase_bytes(wl, u, T)
        pf = phase_flops(wl, T)
        for p in phases:
            ph_bytes[p] += pb.get(p, 0) * ksteps
            ph_flops[p] += pf.get(p, 0) * ksteps
    dom = max(phases, key=lambda p: ph_ms[p])
    launches = ksteps * nl
    if len(phases) == 1:
        # a one-launch layer: the timed region's graph replays hold that kernel alone, so its
        # average launch duration is the timed region's time per layer (no eager gaps)
        ph_ms = {dom: ms / nl * launches}
    achieved = ph_bytes[dom] / (ph_ms[dom] / 1000.0) / 1e9
    traffic = ncu_traffic(dom, wl.name)

    # end to end through the host-buffer entry point (pinned x in, result out, every layer)
    with torch.cuda.stream(stream):
        for l in range(nl):
            layers[l].forward_host(xh[l], T, oh[l], stream, synchronize=(l == nl - 1))
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for l in range(nl):
            layers[l].forward_host(xh[l], T, oh[l], stream, synchronize=(l == nl - 1))
    t_e2e = (time.perf_counter() - t0) / args.steps
    t_e2e = reduce_max(t_e2e, ws)
    e2e_value = whole_job_value(ws, T * nl, t_e2e)

    launches_per_fwd = m.moe_launches_per_forward(layers[0].ctx, T)
    weight_bytes = layers[0].weight_bytes()
    for lay in layers:
        lay.close()
    del layers, xs, outs, xh, oh
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    hbm = ws * bytes_step / (ms / 1000.0) / 1e9
    return {
        "value": value, "ms_per_step": ms, "us_per_layer": 1000.0 * ms / nl, "layers": nl,
        "hbm_gbs": hbm, "hbm_frac_of_measured": hbm / ws / peaks["hbm_gbs"],
        "tflops": ws * flops_step / (ms / 1000.0) / 1e12,
        "bytes_per_layer": bytes_step / nl, "flops_per_layer": flops_step / nl,
        "distinct_experts_per_layer": statistics.mean(U),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured"
                     else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": ph_bytes[dom] / launches,
                     "avg_launch_us": 1000.0 * ph_ms[dom] / launches,
                     "phase_us_per_layer": {p: 1000.0 * ph_ms[p] / launches for p in phases},
                     "phase_gbs": {p: ph_bytes[p] / (ph_ms[p] / 1000.0) / 1e9 for p in phases if ph_ms[p] > 0},
                     "phase_tflops": {p: ph_flops[p] / (ph_ms[p] / 1000.0) / 1e12 for p in phases
                                      if ph_ms[p] > 0 and ph_flops[p] > 0}},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": nl * T * wl.d * 2,
                "d2h_bytes_per_step": nl * T * wl.d * 2,
                "via": "moe_forward_host (pinned host buffers; " + (
                    "the single-launch kernel reads x and writes y over the CPU-GPU link)"
                    if launches_per_fwd == 1 and T * wl.d * 2 <= MAPPED_X_BYTES
                    else "x copied into the context, y written over the CPU-GPU link by the kernels)")},
        "gpu_launches": args.steps * nl * launches_per_fwd, "launches_per_layer": launches_per_fwd,
        "clocks": clk, "device_status": status, "setup_s": t_gen, "weight_bytes_per_layer": weight_bytes,
    }


def prefill_tensor_view(res: dict, mma: dict | None, peaks: dict) -> dict:
    """The layer's algorithmic TFLOP/s against the attainable min(FP4 peak, AI x HBM), the FP4 peak, and the
    measured rate of the MMA kind the GEMMs issue (which runs at the FP8 rate on x split into two planes:
    the tensor pipe does twice the algorithmic flops of the gate/up GEMM and four times those of down)."""
    ai = res["flops_per_layer"] / res["bytes_per_layer"]
    out = {"tflops": res["tflops"], "arithmetic_intensity_flop_per_byte": ai,
           "hbm_bound_tflops": ai * peaks["hbm_gbs"] / 1000.0}
    if mma:
        fp4 = mma["fp4_peak_tflops"]
        att = min(fp4, ai * peaks["hbm_gbs"] / 1000.0)
        out.update({"fp4_peak_tflops": fp4, "attainable_tflops": att, "frac_of_attainable": res["tflops"] / att,
                    "frac_of_fp4_peak": res["tflops"] / fp4, "mxf8f6f4_tflops": mma["tflops"],
                    "frac_of_mxf8f6f4_rate": res["tflops"] / mma["tflops"]})
        ph = res["roofline"].get("phase_tflops", {})
        if "gateup" in ph:  # pipe flops = 2 x algorithmic (two planes of x)
            out["gateup_pipe_frac_of_mxf8f6f4_rate"] = 2 * ph["gateup"] / mma["tflops"]
        if "down" in ph:  # four planes of h
            out["down_pipe_frac_of_mxf8f6f4_rate"] = 4 * ph["down"] / mma["tflops"]
    return out


def provenance(peaks: dict, roofline: dict, mma) -> dict:
    """Where each figure of the line comes from: MEASURED in this run or by ncu, CALCULATED from
    measured figures, or ASSUMED (a fallback constant)."""
    return {
        "value, ms_per_step, us_per_layer, e2e, clocks, cpu_baseline": "MEASURED (CUDA events / wall clock, this run)",
        "roofline.achieved": "CALCULATED: algorithmic bytes per launch (pinned to the page's expert size) / "
                             "MEASURED average launch time",
        "roofline.peak": "MEASURED (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
                         else "ASSUMED (fallback 6.8 TB/s)",
        "roofline.traffic": "MEASURED (ncu DRAM counters on the current kernel code, profiles/traffic.json)"
                            if roofline.get("traffic") is not None else "none taken on the current kernel code",
        "mma_probe.tflops": "MEASURED (this run)" if mma else "not run",
        "mma_probe.fp4_peak_tflops": f"CALCULATED ({FP4_OVER_FP8:g} x the measured rate)" if mma else "not run",
    }


def run_ours(args, wl):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    from routed_expert_ffn_warp_gb300 import build as lib_build
    lib_build.build()
    import routed_expert_ffn_warp_gb300 as m

    peaks = measured_peaks()
    main = measure_workload(args, wl, args.layers, m, torch, ws, rank, local, peaks)

    # the block-scaled MMA rate of this GPU (the kind the expert GEMMs issue)
    mma = None
    if not args.no_mma_probe:
        tf, pms = m.moe_probe_mma_rate(local, args.mma_probe_steps)
        mma = {"kind": "tcgen05.mma kind::mxf8f6f4 (E2M1 x E4M3, UE8M0 scales), M=128 N=192 K=32",
               "tflops": tf, "ms": pms, "unit": "TFLOP/s",
               "fp4_peak_tflops": tf * FP4_OVER_FP8,
               "fp4_peak_source": f"measured mxf8f6f4 rate x {FP4_OVER_FP8:g} (nominal dense FP4 / FP8 ratio, "
                                  "13.5 / 4.5 PFLOP/s)"}

    extras = {}
    for name in [w for w in args.extra_workloads.split(",") if w and w != wl.name]:
        wx = synth.WORKLOADS[name]
        res = measure_workload(args, wx, wx.layers, m, torch, ws, rank, local, peaks)
        res["config"] = config_of(wx, args, wx.layers)
        if name.startswith("prefill"):
            res["tensor"] = prefill_tensor_view(res, mma, peaks)
        if wx.affine_bits:
            res["dtype"] = f"affine{wx.affine_bits}-f16-f32acc"
        extras[name] = res

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = oracle.host_threads()
        n, spent, _ = oracle_sample(wl, args.cpu_budget, 64, threads)
        cpu = {"value": n / spent, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": cpu_sample_text(wl, n, spent, threads)}

    if rank != 0:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    line = {
        "metric": METRIC, "value": main["value"], "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp4-f16-f32acc",
        "data": "synthetic (seeded counter-based generator; random MXFP4 weights)",
        "config": config_of(wl, args),
        "hbm_gbs": main["hbm_gbs"], "hbm_frac_of_measured": main["hbm_frac_of_measured"], "tflops": main["tflops"],
        "us_per_layer": main["us_per_layer"], "distinct_experts_per_layer": main["distinct_experts_per_layer"],
        "roofline": main["roofline"],
        "cpu_baseline": cpu,
        "e2e": main["e2e"],
        "gpu_launches": main["gpu_launches"],
        "clocks": main["clocks"],
        "device_status": main["device_status"],
        "setup_s": main["setup_s"],
        "mma_probe": mma,
        "workloads": extras,
        "provenance": provenance(peaks, main["roofline"], mma),
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default="decode")
    ap.add_argument("--layers", type=int, default=None, help="layers per step (default: the workload's)")
    ap.add_argument("--kernel-steps", type=int, default=3, help="eager steps for per-kernel event timing")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle wall time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--flags", type=int, default=0, help="moe_config.flags of every layer (e.g. 8: register-decode GEMMs instead of tcgen05)")
    ap.add_argument("--extra-workloads", default="verify,small,prefill,prefill16k,affine3",
                    help="comma-separated workloads measured after the main one and reported under 'workloads' "
                         "('' for none)")
    ap.add_argument("--no-mma-probe", action="store_true")
    ap.add_argument("--mma-probe-steps", type=int, default=200000, help="MMAs per SM of the rate probe")
    args = ap.parse_args(argv)
    wl = synth.WORKLOADS[args.workload]
    if args.layers is None:
        args.layers = wl.layers
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
