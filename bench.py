#!/usr/bin/env python
"""Benchmark of the routed-MoE expert FFN (route + gate/up + SwiGLU + down +
combine) on one GB300, through the libds4moe C ABI.

Workload (default): one DeepSeek-V4-Flash-shaped routed-MoE layer at decode
batch 1 -- d_model 4096, d_ff 2048, 256 experts, top-6 with a softmax over
the selected, gate/up/down all Q2_K, synthetic seeded weights and tokens --
with the Q2_K weights repacked once at load into the 16-row tile order
(DS4MOE_Q2_K_R16: the same bytes permuted, see include/ds4moe.h).  A step is
one pass of the whole path over one token.  Weights are replicated into 8
device copies and tokens come from 16 pre-staged slots; step i uses copy
i % 8 and slot i % 16, so consecutive steps never re-read bytes still
resident in L2 (8 copies x 2.1 GB >> 129 MB of L2).

Printed JSON line: tokens/s (value), weight-stream GB/s and its fraction of
the measured HBM peak, the dominant kernel's roofline (its average device
span per launch, %globaltimer at grid entry and exit, over CUDA-graph
replays of the timed steps), per-kernel spans, the CPU oracle as a
baseline, the end-to-end number through the C ABI with host buffers, SM
clocks sampled during the timed region (with a one-second soak of the same
replays where the region is too short to sample), and sub-records, each
with its own roofline: the same layer on plain Q2_K blocks, the 4096-token
prefill chunk (TFLOP/s against the sustained bf16 peak) and the 43-layer
stack at T = 1 (tile order).

`--workload 3` times the prefill chunk alone: 4096 tokens per step (router
with bias, top-6 of 256, Q4_1 gate/up, Q2_K down) through ds4moe_route_topk +
ds4moe_ffn_prefill, reported as tokens/s and TFLOP/s with the tensor-core
roofline of the gate/up grouped GEMM.

`--workload 4` times the 43-layer decode stack alone (every layer with its
own router and 256 Q2_K experts, 91 GB resident; residual in fp32, each
layer fed bf16 of the RMS-normalised residual) through ds4moe_stack_decode,
one CUDA graph per step; the weights are generated on all host cores into
shared memory, layer by layer (`--r16` repacks them to the tile order).

`--impl reference` times the CPU oracle itself (the program the CUDA path is
checked against) on the same metric, each step a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time
from datetime import datetime

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

N_COPIES = 8
N_SLOTS = 16
# Decode steps captured per CUDA graph (consecutive steps, each with its own
# input slot and weight copy, as a decode loop runs them); a step count that
# is not a multiple ends with one graph of the remaining steps, so exactly K
# steps run.
STEPS_PER_GRAPH = 8
METRIC = "routed-MoE tokens/s"
R16_LAYOUT = "q2_k in the 16-row tile order (DS4MOE_Q2_K_R16, repacked once at load by ds4moe_repack)"
PLAIN_LAYOUT = "q2_k plain block layout"
CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", type=int, default=1,
                    help="workload id in synth.WORKLOADS (decode: 0, 1, 2; prefill: 3)")
    ap.add_argument("--cpu-tokens", type=int, default=0, help="tokens in the CPU-baseline sample (0: 2 x cores)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--copies", type=int, default=N_COPIES,
                    help="device copies of the layer rotated across steps (profiling runs use 1)")
    ap.add_argument("--timed-only", action="store_true",
                    help="skip the per-kernel, end-to-end and CPU passes (for profiler captures)")
    ap.add_argument("--n-expert", type=int, default=0,
                    help="override the workload's expert count (smaller cases for profiler captures)")
    ap.add_argument("--quantize", choices=("q2_k", "q4_1"), default=None,
                    help="time the device float-input quantizer instead (fp32 expert matrices -> blocks, "
                         "with per-column importance)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's tokens per step (smaller cases for profiler captures)")
    ap.add_argument("--no-sub", action="store_true",
                    help="default workload: skip the sub-records (plain Q2_K layer, prefill chunk, 43-layer stack)")
    ap.add_argument("--r16", action="store_true",
                    help="single-layer or stack decode at T = 1: repack Q2_K weights into the 16-row tile order")
    ap.add_argument("--plain", action="store_true",
                    help="workload 1 alone on plain Q2_K blocks (no sub-records)")
    ap.add_argument("--prefill", action="store_true",
                    help="time the prefill path (tensor-core grouped GEMMs) on this workload's layer and formats "
                         "(--tokens sets the chunk, default 4096)")
    ap.add_argument("--shared", type=int, default=0, metavar="D_SHARED",
                    help="time the shared expert alone (bf16, d_model of the workload, this width; "
                         "--tokens sets the tokens per step, default 1)")
    return ap.parse_args(argv)


# ------------------------------------------------------------ distribution
def dist_env():
    """(rank, world, local_rank) from torchrun's environment (1 process if unset)."""
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def rank_batch_offset(rank: int) -> int:
    """Each rank draws its own tokens (weak scaling: fixed work per GPU)."""
    return 1000 * rank


def reduce_max(value: float, world: int) -> float:
    """Max over ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (every 20 ms, read
    by a background thread); region() reports the samples inside the latest
    window between mark(True) and mark(False), and nothing else."""

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                    "-i", str(gpu_index), "-lms", str(period_ms)]
        self.proc = None
        self.rows = []
        self.t0 = self.t1 = None
        self.thread = None

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            f = [c.strip() for c in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                continue
            self.rows.append((ts, f))

    def mark(self, begin: bool):
        if begin:
            self.t0, self.t1 = datetime.now(), None
        else:
            self.t1 = datetime.now()

    def region(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples_in_region": 0}
        time.sleep(0.1)  # the samples of the window's last period
        inside = [f for ts, f in list(self.rows) if self.t0 and self.t1 and self.t0 <= ts <= self.t1]
        region_ms = (self.t1 - self.t0).total_seconds() * 1000.0 if self.t0 and self.t1 else None
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in region"],
                    "samples_in_region": 0, "region_ms": region_ms}
        sm = [float(f[2]) for f in inside if f[2].replace(".", "").isdigit()]
        smax = [float(f[3]) for f in inside if f[3].replace(".", "").isdigit()]
        reasons = set()
        for f in inside:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples_in_region": len(inside), "region_ms": region_ms}

    def close(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()


# --------------------------------------------------------------- workload
# block (values, bytes) per format: Q4_1 20 B / 32, Q2_K 84 B / 256, Q4_K 144 B / 256
BLOCK = {synth.Q4_1: (32, 20), synth.Q2_K: (256, 84), synth.Q4_K: (256, 144)}


def mat_bytes(qtype: str, rows: int, cols: int) -> int:
    bv, bb = BLOCK[qtype]
    return rows * cols // bv * bb


def host_layer_blocks(w: synth.Workload, layer: int, experts, packer):
    """Experts-major block bytes of the listed experts (others zero) via `packer`."""
    out = {}
    for t in (synth.T_GATE, synth.T_UP, synth.T_DOWN):
        rows, cols = synth.matrix_shape(w, t)
        q = synth.recipe(w, t)
        per = mat_bytes(q.qtype, rows, cols)
        buf = np.zeros(w.n_expert * per, np.uint8)
        for e in experts:
            buf[e * per:(e + 1) * per] = packer(synth.matrix_fields(w, layer, t, e))
        out[t] = buf
    return out


def product_packer(M):
    def pack(f):
        if f.qtype == synth.Q4_1:
            return M.ds4moe_quantize_ref(M.DS4MOE_Q4_1, f.bits, f.group, f.codes, f.scale, f.minv)
        if f.qtype == synth.Q4_K:
            return M.ds4moe_quantize_ref(M.DS4MOE_Q4_K, 4, 256, f.codes, f.scale, f.minv, f.sc, f.mn)
        return M.ds4moe_quantize_ref(M.DS4MOE_Q2_K, 2, 256, f.codes, f.scale, f.minv, f.sc, f.mn)
    return pack


def device_layer(w: synth.Workload, M, torch):
    """All experts of layer 0 packed by the library's host packer, uploaded."""
    from bit_quantized_moe_q2_gb300.device import DeviceLayer
    qid = {synth.Q4_1: M.DS4MOE_Q4_1, synth.Q2_K: M.DS4MOE_Q2_K, synth.Q4_K: M.DS4MOE_Q4_K}
    dev = DeviceLayer.empty(w.d_model, w.d_ff, w.n_expert, qid[w.gate.qtype], qid[w.up.qtype], qid[w.down.qtype])
    pack = product_packer(M)
    names = {synth.T_GATE: "gate", synth.T_UP: "up", synth.T_DOWN: "down"}
    pinned = {}
    for e in range(w.n_expert):
        blocks = {name: pack(synth.matrix_fields(w, 0, t, e)) for t, name in names.items()}
        torch.cuda.current_stream().synchronize()      # previous expert's copies are done
        for name, b in blocks.items():
            if name not in pinned:
                pinned[name] = torch.empty(b.size, dtype=torch.uint8).pin_memory()
            pinned[name].numpy()[:] = b
            dev.expert_slice(name, e).copy_(pinned[name], non_blocking=True)
    torch.cuda.synchronize()
    return dev


def expert_bytes(w: synth.Workload) -> int:
    tot = 0
    for t in (synth.T_GATE, synth.T_UP, synth.T_DOWN):
        rows, cols = synth.matrix_shape(w, t)
        q = synth.recipe(w, t)
        tot += mat_bytes(q.qtype, rows, cols)
    return tot


def gate_up_bytes(w: synth.Workload) -> int:
    tot = 0
    for t in (synth.T_GATE, synth.T_UP):
        rows, cols = synth.matrix_shape(w, t)
        q = synth.recipe(w, t)
        tot += mat_bytes(q.qtype, rows, cols)
    return tot


# DRAM bytes per launch of the roofline kernel from an ncu capture of the
# current build (dram__bytes_read.sum + dram__bytes_write.sum), keyed by
# (workload, weight layout, kernel); a key missing here reports null.  The summaries with the commands are in profiles/.
NCU_TRAFFIC: dict = {
    # k_ffn_t1r, mean of three launches (49.63 MB read + 3 KB written), captured on the
    # 32-expert case of the same shape: a launch processes the same 6 experts' matrices
    ("flash-layer-decode-t1-q2k", R16_LAYOUT, "ffn_t1r"): 49_636_693,
}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_tensor_peak(sustained: bool):
    """Dense bf16 TFLOP/s (kind::f16 runs at the same rate)."""
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)[key]), "measured"
    except (OSError, KeyError, ValueError):
        return (1700.0 if sustained else 1900.0), "fallback"


def prefill_flops(w: synth.Workload) -> tuple[float, float]:
    """(whole step, gate/up kernel) algorithmic FLOPs: 2 * 3 * D * F per
    (token, selected expert) plus the router's 2 * D * E per token."""
    pairs = w.T * w.k
    ffn = 2.0 * 3 * w.d_model * w.d_ff * pairs
    return ffn + 2.0 * w.d_model * w.n_expert * w.T, 2.0 * 2 * w.d_model * w.d_ff * pairs


def cores_available() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------ CPU oracle
def cpu_baseline(w: synth.Workload, n_tokens: int, batch0: int) -> dict:
    """The oracle (plain C, fp64) on a bounded sample of tokens, all host cores."""
    import oracle
    cores = cores_available()
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    Wr, bias = synth.router(w)
    x = synth.activations(w, T=n_tokens, batch=batch0)
    idx, wt, _ = oracle.route(x, Wr, bias, w.k)
    blocks = host_layer_blocks(w, 0, sorted(set(idx.ravel().tolist())), oracle.pack_fields)
    qg, qu, qd = (oracle.QTYPES[w.gate.qtype], oracle.QTYPES[w.up.qtype], oracle.QTYPES[w.down.qtype])
    t0 = time.perf_counter()
    idx, wt, _ = oracle.route(x, Wr, bias, w.k)
    oracle.moe_ffn(w.d_model, w.d_ff, w.n_expert, qg, blocks[synth.T_GATE], qu, blocks[synth.T_UP], qd,
                   blocks[synth.T_DOWN], x, idx, wt)
    dt = time.perf_counter() - t0
    return {"value": n_tokens / dt, "unit": "tokens/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"{n_tokens} tokens: route + all selected expert FFNs + combine (fp64 C oracle, OpenMP over tokens)"}


# ------------------------------------------------------- reference (oracle)
def run_reference(args, w: synth.Workload):
    """The CPU oracle as the reference arm: K timed steps, each a bounded
    sample of the per-token work (rows of the selected experts' gate, up and
    down matrices), extrapolated to tokens/s by weight values processed."""
    import oracle
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cores = 1  # the row-slice sample runs on one thread
    Wr, bias = synth.router(w)
    n_tok = 4
    x = synth.activations(w, T=n_tok, batch=0)
    idx, wt, _ = oracle.route(x, Wr, bias, w.k)
    qg, qu, qd = (oracle.QTYPES[w.gate.qtype], oracle.QTYPES[w.up.qtype], oracle.QTYPES[w.down.qtype])
    experts = sorted(set(idx.ravel().tolist()))
    blocks = host_layer_blocks(w, 0, experts, oracle.pack_fields)
    D, F = w.d_model, w.d_ff
    per_g = blocks[synth.T_GATE].size // w.n_expert
    per_u = blocks[synth.T_UP].size // w.n_expert
    per_d = blocks[synth.T_DOWN].size // w.n_expert
    xs = oracle.bf16_to_f32(x).astype(np.float64)
    hs = {}
    for t in range(n_tok):
        for i in range(w.k):
            e = int(idx[t, i])
            _, h, _, _ = oracle.expert_ffn(D, F, qg, blocks[synth.T_GATE], qu, blocks[synth.T_UP], qd,
                                           blocks[synth.T_DOWN], e, x[t])
            hs[(t, i)] = oracle.bf16_to_f32(h).astype(np.float64)
    values_per_token = w.k * 3 * D * F * w.n_layers
    # size the per-step sample so that warmup + steps take ~100 s
    budget = 100.0 / max(args.steps + args.warmup, 1)
    t0 = time.perf_counter()
    oracle.matvec_rows(qg, blocks[synth.T_GATE][idx[0, 0] * per_g:(idx[0, 0] + 1) * per_g], F, D, 0, 8, xs[0])
    t_row = (time.perf_counter() - t0) / 8          # one gate row (D values)
    R = int(max(1, min(F // 2, budget / (4 * t_row))))

    def step(s):
        t, i = (s // w.k) % n_tok, s % w.k
        e = int(idx[t, i])
        r0 = (s * R) % (F - R + 1)
        oracle.matvec_rows(qg, blocks[synth.T_GATE][e * per_g:(e + 1) * per_g], F, D, r0, R, xs[t])
        oracle.matvec_rows(qu, blocks[synth.T_UP][e * per_u:(e + 1) * per_u], F, D, r0, R, xs[t])
        d0 = (s * 2 * R) % (D - 2 * R + 1)
        oracle.matvec_rows(qd, blocks[synth.T_DOWN][e * per_d:(e + 1) * per_d], D, F, d0, 2 * R, hs[(t, i)])
        return 2 * R * D + 2 * R * F

    for s in range(args.warmup):
        step(s)
    done = 0
    t0 = time.perf_counter()
    for s in range(args.steps):
        done += step(s)
    dt = time.perf_counter() - t0
    tokens = done / values_per_token
    value = tokens / dt if dt > 0 else 0.0
    sample = (f"per step {R} rows of gate, {R} of up and {2 * R} of down of one selected expert "
              f"(fp64 C oracle, one thread); tokens/s extrapolated at {values_per_token} weight values "
              f"per token ({w.n_layers} layer(s); router < 1% of the work, not sampled)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(w: synth.Workload, n_copies: int = N_COPIES) -> dict:
    return {"workload": w.name, "d_model": w.d_model, "d_ff": w.d_ff, "n_expert": w.n_expert, "top_k": w.k,
            "tokens_per_step": w.T, "gate": w.gate.qtype, "up": w.up.qtype, "down": w.down.qtype,
            "seed": w.seed, "l2": f"{n_copies} device copies of the layer x {N_SLOTS} token slots rotate per step: "
                                  "no step re-reads bytes an earlier step left in L2"}


# --------------------------------------------------------------- our arm
def init_dist(torch):
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def load_library(rank, world):
    from bit_quantized_moe_q2_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    import bit_quantized_moe_q2_gb300 as M
    return M


def gpu_index(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis.replace(",", "").isdigit():
        return int(vis.split(",")[local])
    return local


def timed_replays(torch, stream, replay, steps, world, sampler):
    """Exactly `steps` calls of replay(i) between a barrier + synchronize on
    each side, timed with CUDA events on `stream`; max over ranks (ms)."""
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark(True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(steps):
            replay(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier(world)
    return reduce_max(ev0.elapsed_time(ev1), world)


def clock_soak(torch, stream, replay, sampler, step_ms: float, seconds: float = 1.0) -> dict:
    """The same replays for about `seconds` right after a timed region too
    short for the sampler (nothing of it is timed): the clocks under this load."""
    n = int(max(1, min(200_000, seconds * 1000.0 / max(step_ms, 1e-4))))
    torch.cuda.synchronize()
    sampler.mark(True)
    with torch.cuda.stream(stream):
        for i in range(n):
            replay(i)
    torch.cuda.synchronize()
    sampler.mark(False)
    return {"steps": n}


def measure_clocks(torch, stream, replay, gpu: int, steps: int, world: int):
    """Times the region (returns ms) and samples SM clocks during it; where the
    region is shorter than the sampling period, a one-second soak of the same
    replays follows and is reported beside it."""
    sampler = ClockSampler(gpu)
    sampler.start()
    ms = timed_replays(torch, stream, replay, steps, world, sampler)
    clocks = sampler.region()
    if clocks["samples_in_region"] == 0:
        soak = clock_soak(torch, stream, replay, sampler, ms / max(steps, 1))
        soak.update(sampler.region())
        clocks["soak"] = soak
    sampler.close()
    return ms, clocks


def span_pass(M, torch, stream, replay, n: int) -> dict:
    """Per-kernel device spans (ds4moe_profile_span, %globaltimer at grid
    entry and exit) over n replays: {kernel: {avg_us, launches_per_step}}."""
    torch.cuda.synchronize()
    M.ds4moe_profile_span(1)
    try:
        with torch.cuda.stream(stream):
            for i in range(n):
                replay(i)
        stream.synchronize()
        sp = M.ds4moe_profile_span(0)
    finally:
        M.ds4moe_profile_span(0)
    return {k: {"avg_us": ns / c / 1000.0, "launches_per_step": c / n} for k, (ns, c) in sp.items()}


def launch_count(M, torch, stream, eager_step, n: int) -> dict:
    """Kernels launched per step, by name, from the library's launch record
    over n eager steps (the counts only: eager event times include host gaps)."""
    torch.cuda.synchronize()
    M.ds4moe_profile_enable(True)
    try:
        with torch.cuda.stream(stream):
            for i in range(n):
                eager_step(i)
        stream.synchronize()
        prof = M.ds4moe_profile_read()
    finally:
        M.ds4moe_profile_enable(False)
    return {k: c / n for k, (_, c) in prof.items()}


def hbm_roofline(kdesc: str, algo_bytes: float, avg_us: float, traffic) -> dict:
    peak, kind = measured_peaks()
    gbs = algo_bytes / (avg_us * 1e-6) / 1e9
    return {"kernel": kdesc, "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
            "traffic": traffic, "algorithmic_bytes_per_launch": int(algo_bytes), "avg_launch_us": avg_us,
            "timing": "device span per launch (%globaltimer, first CTA past its dependency wait to last warp "
                      "exit) over CUDA-graph replays of the timed steps",
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if kind == "measured" else "fallback 6.8 TB/s"}


def graph_schedule(steps: int, g: int, n_slots: int):
    """The timed region's graph replays for exactly `steps` steps: (graph kind,
    graph index, the step numbers it runs) -- full graphs of g consecutive
    steps (graph j holds steps j g .. j g + g - 1, j < n_slots), then, for a
    remainder r, one graph of the r steps that follow."""
    n_full, rem = divmod(steps, g)
    sched = [("full", i % n_slots, [(i % n_slots) * g + q for q in range(g)]) for i in range(n_full)]
    if rem:
        sched.append(("rest", 0, [n_full * g + q for q in range(rem)]))
    return sched


def replicate(dev, n: int):
    return [dev] + [type(dev)(dev.d_model, dev.d_ff, dev.n_expert, dev.q_gate, dev.q_up, dev.q_down,
                              dev.gate.clone(), dev.up.clone(), dev.down.clone()) for _ in range(n - 1)]


def decode_layer_record(args, M, torch, w: synth.Workload, copies, layout: str, rank: int, world: int, local: int,
                        with_e2e: bool) -> dict:
    """One layer's decode steps (route + FFN) through ds4moe_moe_decode, step i
    on copy i % len(copies) and token slot i % N_SLOTS; CUDA graphs of
    STEPS_PER_GRAPH consecutive steps (and one graph for a remainder)."""
    from bit_quantized_moe_q2_gb300.device import check_status, workspace
    dev = copies[0]
    n_copies = len(copies)
    Wr, bias = synth.router(w)
    Wr_d = torch.from_numpy(Wr).cuda()
    b_d = None if bias is None else torch.from_numpy(bias).cuda()
    T, k, D = w.T, w.k, w.d_model
    xs_host = [synth.activations(w, T=T, batch=rank_batch_offset(rank) + s) for s in range(N_SLOTS)]
    xs = [torch.from_numpy(x.view(np.int16)).cuda() for x in xs_host]
    idx = [torch.empty((T, k), dtype=torch.int32, device="cuda") for _ in range(N_SLOTS)]
    wt = [torch.empty((T, k), dtype=torch.float32, device="cuda") for _ in range(N_SLOTS)]
    out = [torch.empty((T, D), dtype=torch.float32, device="cuda") for _ in range(N_SLOTS)]
    ws = workspace(dev, T, k)
    stream = torch.cuda.Stream()

    def step(i, s=None):
        j = i % N_SLOTS
        M.ds4moe_moe_decode(copies[i % n_copies].abi, xs[j], Wr_d, b_d, k, out[j], idx[j], wt[j], ws, s)

    with torch.cuda.stream(stream):
        for i in range(2 * N_SLOTS):
            step(i, stream)
    check_status(ws, stream)
    uniq = [len(set(idx[j].cpu().numpy().ravel().tolist())) for j in range(N_SLOTS)]
    G = STEPS_PER_GRAPH
    graphs = []
    for j in range(N_SLOTS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for q in range(G):
                step(j * G + q, stream)
        graphs.append(g)
    # the timed region: exactly args.steps steps; schedule entry = (graph, its steps)
    sched = []
    for kind, j, sts in graph_schedule(args.steps, G, N_SLOTS):
        if kind == "full":
            sched.append((graphs[j], sts))
        else:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for st in sts:
                    step(st, stream)
            sched.append((g, sts))

    def replay(i):
        sched[i % len(sched)][0].replay()

    def replay_g(i):
        graphs[i % N_SLOTS].replay()

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            replay_g(i)
        for g_, _ in sched[len(sched) - 1:]:  # a remainder graph, uploaded before the timed region
            g_.replay()
    stream.synchronize()
    check_status(ws, stream)
    ms, clocks = measure_clocks(torch, stream, replay, gpu_index(local), len(sched), world)
    check_status(ws, stream)
    tokens = world * args.steps * T
    eb = expert_bytes(w)
    algo_step = [u * eb + Wr.nbytes + (0 if bias is None else bias.nbytes) + T * D * 2 + T * D * 4 for u in uniq]
    algo_bytes = sum(algo_step[st % N_SLOTS] for _, sts in sched for st in sts)
    peak, _ = measured_peaks()
    stream_gbs = algo_bytes / (ms / 1000.0) / 1e9
    rec = {"metric": METRIC, "value": tokens / (ms / 1000.0), "unit": "tokens/s", "steps": args.steps,
           "ms_per_step": ms / args.steps, "weight_stream_gbs": stream_gbs, "hbm_frac": stream_gbs / peak,
           "clocks": clocks}
    cfg = workload_config(w, n_copies)
    cfg["layout"] = layout
    cfg["steps_per_graph"] = G
    rec["config"] = cfg
    if args.timed_only:
        return rec
    kp = max(min(max(args.steps, 200), 2000) // G, 1)
    kernels = span_pass(M, torch, stream, replay_g, kp)
    for v in kernels.values():
        v["launches_per_step"] /= G
    uniq_avg = sum(uniq[((i % N_SLOTS) * G + q) % N_SLOTS] for i in range(kp) for q in range(G)) / (kp * G)
    ffn = next((n for n in ("ffn_t1r", "ffn_t1") if n in kernels), None)
    if ffn:
        algo = uniq_avg * eb + T * D * 2 + T * D * 4
        desc = ("expert FFN over the 16-row tile order (gate/up + SwiGLU + down + combine, routing fused, "
                "dequant fused)" if ffn == "ffn_t1r" else
                "expert FFN (merged gate/up + SwiGLU + down + combine, dequant fused)")
        rec["roofline"] = hbm_roofline(desc, algo, kernels[ffn]["avg_us"], NCU_TRAFFIC.get((w.name, layout, ffn)))
    else:
        gu = next((n for n in ("gate_up_mma", "gate_up_t1") if n in kernels), None)
        if gu:
            algo = uniq_avg * gate_up_bytes(w) + T * D * 2 + T * k * w.d_ff * 2
            rec["roofline"] = hbm_roofline("gate_up (fused dequant GEMV + SwiGLU)", algo, kernels[gu]["avg_us"],
                                           NCU_TRAFFIC.get((w.name, layout, gu)))
    rec["kernels"] = kernels
    counts = launch_count(M, torch, stream, lambda i: step(i, stream), 50)
    rec["launches_per_step"] = counts
    rec["gpu_launches"] = int(round(sum(counts.values()) * args.steps))
    if with_e2e:
        ke = min(args.steps, 2000)
        xh = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs_host]
        oh = torch.empty((T, D), dtype=torch.float32).pin_memory()
        x_in = torch.empty((T, D), dtype=torch.int16, device="cuda")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for i in range(ke):
                x_in.copy_(xh[i % N_SLOTS], non_blocking=True)
                M.ds4moe_moe_decode(copies[i % n_copies].abi, x_in, Wr_d, b_d, k, out[0], idx[0], wt[0], ws, stream)
                oh.copy_(out[0], non_blocking=True)
                stream.synchronize()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(e0.elapsed_time(e1), world)
        check_status(ws, stream)
        rec["e2e"] = {"value": world * ke * T / (e2e_ms / 1000.0), "unit": "tokens/s", "steps": ke,
                      "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 4,
                      "path": "pinned H2D x, ds4moe_moe_decode (eager C-ABI call), D2H out, stream sync per step"}
    return rec


def prefill_record(args, M, torch, w: synth.Workload, rank: int, world: int, local: int, with_e2e: bool) -> dict:
    """Prefill: route (with bias) + tensor-core expert FFN over T tokens per
    step.  Inputs (3.4 GB of weights at the Flash shape) far exceed L2, so no
    flush is needed."""
    from bit_quantized_moe_q2_gb300.device import check_status, workspace
    dev = device_layer(w, M, torch)
    Wr, bias = synth.router(w)
    Wr_d = torch.from_numpy(Wr).cuda()
    b_d = None if bias is None else torch.from_numpy(bias).cuda()
    T, k, D = w.T, w.k, w.d_model
    n_slots = 2
    xs_host = [synth.activations(w, T=T, batch=rank_batch_offset(rank) + s) for s in range(n_slots)]
    xs = [torch.from_numpy(x.view(np.int16)).cuda() for x in xs_host]
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, k), dtype=torch.float32, device="cuda")
    out = torch.empty((T, D), dtype=torch.float32, device="cuda")
    ws = workspace(dev, T, k, prefill=True)
    stream = torch.cuda.Stream()

    def step(i, x=None):
        xin = xs[i % n_slots] if x is None else x
        M.ds4moe_route_topk(xin, Wr_d, b_d, k, idx, wt, None, ws, stream)
        M.ds4moe_ffn_prefill(dev.abi, xin, idx, wt, out, ws, stream)

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step(i)
    stream.synchronize()
    check_status(ws, stream)
    counts = np.bincount(idx.cpu().numpy().ravel(), minlength=w.n_expert)
    steps = max(3, min(args.steps, 200))
    ms, clocks = measure_clocks(torch, stream, step, gpu_index(local), steps, world)
    check_status(ws, stream)
    flops_step, flops_gu = prefill_flops(w)
    rec = {"metric": METRIC, "value": world * steps * T / (ms / 1000.0), "unit": "tokens/s", "steps": steps,
           "ms_per_step": ms / steps, "tflops": world * steps * flops_step / (ms / 1000.0) / 1e12,
           "clocks": clocks}
    cfg = workload_config(w, 1)
    cfg["l2"] = (f"inputs larger than L2: every step streams {w.n_expert * expert_bytes(w) / 1e9:.2f} GB "
                 "of expert weights")
    rec["config"] = cfg
    if args.timed_only:
        return rec
    kernels = span_pass(M, torch, stream, step, min(steps, 10))
    peak, peak_kind = measured_tensor_peak(sustained=True)
    rec["tensor_frac"] = rec["tflops"] / peak
    if "gate_up_tc" in kernels:
        us = kernels["gate_up_tc"]["avg_us"]
        qname = synth.recipe(w, synth.T_GATE).qtype.upper()
        # experts with at most `small` pairs stream through the multi-token
        # kernels: the grouped GEMM's own flops are those of the other pairs
        small = M.ds4moe_prefill_small_pairs(dev.abi)
        tc_pairs = int(counts[counts > small].sum()) if small > 0 else w.T * w.k
        flops_tc = flops_gu * tc_pairs / (w.T * w.k)
        rec["prefill_split"] = {"small_pairs": small, "tc_pairs": tc_pairs,
                                "streamed_pairs": w.T * w.k - tc_pairs,
                                "streamed_experts": int(((counts > 0) & (counts <= small)).sum()) if small > 0 else 0}
        rec["roofline"] = {"kernel": f"gate_up_tc (tcgen05 grouped GEMM, fused {qname} dequant + SwiGLU)",
                           "bound": "tensor", "achieved": flops_tc / (us * 1e-6) / 1e12, "peak": peak,
                           "unit": "TFLOP/s", "frac": flops_tc / (us * 1e-6) / 1e12 / peak, "traffic": None,
                           "algorithmic_flops_per_launch": flops_tc, "avg_launch_us": us,
                           "timing": "device span per launch (%globaltimer, grid entry to last warp exit)",
                           "peak_source": f"{peak_kind} bf16_tflops_sustained (kind::f16 runs at the bf16 rate)"}
        if "gate_up_mma" in kernels:  # the streamed experts' gate/up, right after the grouped GEMM
            us_all = us + kernels["gate_up_mma"]["avg_us"]
            rec["gate_up_phase"] = {"kernels": "gate_up_tc + gate_up (streamed experts)", "us": us_all,
                                    "tflops": flops_gu / (us_all * 1e-6) / 1e12,
                                    "frac": flops_gu / (us_all * 1e-6) / 1e12 / peak}
    rec["kernels"] = kernels
    cnt = launch_count(M, torch, stream, step, 2)
    rec["launches_per_step"] = cnt
    rec["gpu_launches"] = int(round(sum(cnt.values()) * steps))
    rec["expert_load"] = {"max": int(counts.max()), "min": int(counts.min()), "empty": int((counts == 0).sum())}
    if with_e2e:
        ke = min(steps, 5)
        xh = [torch.from_numpy(x.view(np.int16)).pin_memory() for x in xs_host]
        oh = torch.empty((T, D), dtype=torch.float32).pin_memory()
        x_in = torch.empty((T, D), dtype=torch.int16, device="cuda")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for i in range(ke):
                x_in.copy_(xh[i % n_slots], non_blocking=True)
                step(i, x_in)
                oh.copy_(out, non_blocking=True)
                stream.synchronize()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(e0.elapsed_time(e1), world)
        rec["e2e"] = {"value": world * ke * T / (e2e_ms / 1000.0), "unit": "tokens/s", "steps": ke,
                      "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 4,
                      "path": "pinned H2D x, ds4moe_route_topk + ds4moe_ffn_prefill (C-ABI calls), D2H out, "
                              "sync per step"}
    del dev
    torch.cuda.empty_cache()
    return rec


# ------------------------------------------------------- decode stack arm
_POOL_M = None


def _pool_init():
    global _POOL_M
    import bit_quantized_moe_q2_gb300 as M
    M.lib()
    _POOL_M = M


def _pack_expert(job):
    """Pack expert e of one layer into the shared-memory tensors (worker)."""
    from multiprocessing import shared_memory
    w, layer, e, names, per = job
    pack = product_packer(_POOL_M)
    for t, name in zip((synth.T_GATE, synth.T_UP, synth.T_DOWN), names):
        shm = shared_memory.SharedMemory(name=name)
        try:
            shm.buf[e * per[t]:(e + 1) * per[t]] = pack(synth.matrix_fields(w, layer, t, e)).tobytes()
        finally:
            shm.close()
    return e


def tensor_bytes(w: synth.Workload, t: int) -> int:
    rows, cols = synth.matrix_shape(w, t)
    q = synth.recipe(w, t)
    return mat_bytes(q.qtype, rows, cols)


def start_stack_pool(w: synth.Workload):
    """Shared-memory tensors and the generator pool (spawned: it starts
    before, or independently of, any GPU call of this process)."""
    import multiprocessing as mp
    from multiprocessing import shared_memory
    per = {t: tensor_bytes(w, t) for t in (synth.T_GATE, synth.T_UP, synth.T_DOWN)}
    shms = [shared_memory.SharedMemory(create=True, size=w.n_expert * per[t])
            for t in (synth.T_GATE, synth.T_UP, synth.T_DOWN)]
    pool = mp.get_context("spawn").Pool(max(1, cores_available()), initializer=_pool_init)
    return pool, shms, per


def stack_layers(w: synth.Workload, M, torch, pool, shms, per, r16: bool):
    """All layers generated on the host cores, uploaded (and, with r16,
    repacked on the device into the 16-row tile order)."""
    from bit_quantized_moe_q2_gb300.device import DeviceLayer
    qid = {synth.Q4_1: M.DS4MOE_Q4_1, synth.Q2_K: M.DS4MOE_Q2_K, synth.Q4_K: M.DS4MOE_Q4_K}
    devs, Wrs, biases = [], [], []
    names = [sh.name for sh in shms]
    try:
        for layer in range(w.n_layers):
            pool.map(_pack_expert, [(w, layer, e, names, per) for e in range(w.n_expert)], chunksize=4)
            dev = DeviceLayer.empty(w.d_model, w.d_ff, w.n_expert, qid[w.gate.qtype], qid[w.up.qtype],
                                    qid[w.down.qtype])
            for sh, dst in zip(shms, (dev.gate, dev.up, dev.down)):
                dst.copy_(torch.frombuffer(sh.buf, dtype=torch.uint8, count=dst.numel()))
            if r16:
                dev = dev.repacked_r16()
                torch.cuda.synchronize()
            Wr, b = synth.router(w, layer)
            devs.append(dev)
            Wrs.append(torch.from_numpy(Wr).cuda())
            biases.append(None if b is None else torch.from_numpy(b).cuda())
    finally:
        pool.close()
        pool.join()
        for sh in shms:
            sh.close()
            sh.unlink()
    return devs, Wrs, biases


def stack_record(args, M, torch, w: synth.Workload, devs, Wrs, biases, layout: str, rank: int, world: int,
                 local: int, with_e2e: bool) -> dict:
    from bit_quantized_moe_q2_gb300.device import check_status, workspace
    T, k, D, L = w.T, w.k, w.d_model, w.n_layers
    bias_arg = None if biases[0] is None else biases
    x0 = [torch.from_numpy(oracle_free_bf16_to_f32(synth.activations(w, T=T, batch=rank_batch_offset(rank) + s)))
          .cuda() for s in range(N_SLOTS)]
    x_res = torch.empty((T, D), dtype=torch.float32, device="cuda")
    xb = torch.empty((T, D), dtype=torch.int16, device="cuda")
    out = torch.empty((T, D), dtype=torch.float32, device="cuda")
    idx = torch.empty((L, M.stack_ldk(T, k)), dtype=torch.int32, device="cuda")
    wt = torch.empty((L, M.stack_ldk(T, k)), dtype=torch.float32, device="cuda")
    ws = workspace(devs[0], T, k)
    abis = [d.abi for d in devs]
    stream = torch.cuda.Stream()

    def step(j, s=None):
        x_res.copy_(x0[j % N_SLOTS], non_blocking=True)
        M.ds4moe_stack_decode(abis, Wrs, bias_arg, k, x_res, xb, out, idx, wt, ws, stream=s)

    with torch.cuda.stream(stream):
        for j in range(N_SLOTS):
            step(j, stream)
    check_status(ws, stream)
    uniq = [len(set(idx[l, :T * k].cpu().numpy().ravel().tolist())) for l in range(L)]
    graphs = []
    for j in range(N_SLOTS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(j, stream)
        graphs.append(g)

    def replay(i):
        graphs[i % N_SLOTS].replay()

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            replay(i)
    stream.synchronize()
    check_status(ws, stream)
    ms, clocks = measure_clocks(torch, stream, replay, gpu_index(local), args.steps, world)
    check_status(ws, stream)
    eb = expert_bytes(w)
    algo_step = sum(u * eb for u in uniq) + L * (w.n_expert * D * 4) + T * D * 4 * 2
    peak, _ = measured_peaks()
    stream_gbs = algo_step / (ms / args.steps / 1000.0) / 1e9
    cfg = workload_config(w, 1)
    cfg["n_layers"] = L
    cfg["layout"] = layout
    cfg["l2"] = f"inputs larger than L2: every step streams {L} layers of expert weights"
    rec = {"metric": METRIC, "value": world * args.steps * T / (ms / 1000.0), "unit": "tokens/s",
           "steps": args.steps, "ms_per_step": ms / args.steps, "weight_stream_gbs": stream_gbs,
           "hbm_frac": stream_gbs / peak, "config": cfg, "clocks": clocks}
    if args.timed_only:
        return rec
    kp = min(max(args.steps, 20), 50)
    kernels = span_pass(M, torch, stream, replay, kp)
    ffn = next((n for n in ("ffn_t1r", "ffn_t1", "gate_up_mma") if n in kernels), None)
    if ffn:
        if ffn == "gate_up_mma":
            algo = sum(uniq) / L * gate_up_bytes(w) + T * D * 2 + T * k * w.d_ff * 2
            desc = "gate_up (fused dequant GEMV + SwiGLU), per layer"
        else:
            algo = sum(uniq) / L * eb + T * D * 2 + T * D * 4
            desc = ("expert FFN over the 16-row tile order, per layer" if ffn == "ffn_t1r" else
                    "expert FFN (merged gate/up + SwiGLU + down + combine), per layer")
        rec["roofline"] = hbm_roofline(desc, algo, kernels[ffn]["avg_us"], None)
    rec["kernels"] = kernels
    cnt = launch_count(M, torch, stream, lambda i: step(i, stream), 2)
    rec["launches_per_step"] = cnt
    rec["gpu_launches"] = int(round(sum(cnt.values()) * args.steps))
    if with_e2e:
        ke = min(args.steps, 50)
        xh = [x.cpu().pin_memory() for x in x0]
        oh = torch.empty((T, D), dtype=torch.float32).pin_memory()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for i in range(ke):
                x_res.copy_(xh[i % N_SLOTS], non_blocking=True)
                M.ds4moe_stack_decode(abis, Wrs, bias_arg, k, x_res, xb, out, idx, wt, ws, stream=stream)
                oh.copy_(x_res, non_blocking=True)
                stream.synchronize()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(e0.elapsed_time(e1), world)
        rec["e2e"] = {"value": world * ke * T / (e2e_ms / 1000.0), "unit": "tokens/s", "steps": ke,
                      "h2d_bytes_per_step": T * D * 4, "d2h_bytes_per_step": T * D * 4,
                      "path": f"pinned H2D x_res, ds4moe_stack_decode (eager C-ABI call, {L} layers), D2H x_res, "
                              "sync per step"}
    return rec


def oracle_free_bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a bit shift; no method arithmetic)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


def line_from(rec: dict, args, world: int, dtype: str) -> dict:
    """The contract's JSON line around a measurement record."""
    line = {"metric": rec["metric"], "value": rec["value"], "unit": rec["unit"], "n_gpus": world,
            "steps": rec["steps"], "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic", "config": rec["config"]}
    for key in ("tflops", "tensor_frac", "weight_stream_gbs", "hbm_frac", "roofline", "gate_up_phase",
                "prefill_split", "kernels", "launches_per_step", "expert_load", "cpu_baseline", "e2e",
                "gpu_launches", "clocks"):
        if key in rec:
            line[key] = rec[key]
    return line


DECODE_DTYPE = "f32 accumulate over exact 2-bit codes and bf16 activations"
PREFILL_DTYPE = "f16 tensor-core operands (exact gate/up split), f32 accumulate"


def sub_summary(rec: dict) -> dict:
    """A sub-record of the default line: the measurement without its host-side extras."""
    keep = ("metric", "value", "unit", "steps", "ms_per_step", "tflops", "tensor_frac", "weight_stream_gbs",
            "hbm_frac", "config", "roofline", "gate_up_phase", "prefill_split", "kernels", "gpu_launches", "e2e",
            "clocks", "expert_load")
    return {k: rec[k] for k in keep if k in rec}


def run_default(args, w: synth.Workload):
    """The Flash decode layer at T = 1 on tile-order weights (the line), with
    sub-records: the same layer on plain Q2_K blocks, the 4096-token prefill
    chunk and the 43-layer stack at T = 1."""
    import torch
    rank, world, local = init_dist(torch)
    M = load_library(rank, world)
    w4 = synth.WORKLOADS[4]
    sub = not args.no_sub and world == 1   # sub-records at N = 1 only
    stack_pool = start_stack_pool(w4) if sub else None  # spawned: no CUDA state inherited
    plain = device_layer(w, M, torch)
    n_copies = max(1, args.copies)
    r16 = replicate(plain.repacked_r16(), n_copies)
    torch.cuda.synchronize()
    main = decode_layer_record(args, M, torch, w, r16, R16_LAYOUT, rank, world, local, with_e2e=True)
    del r16
    torch.cuda.empty_cache()
    subs = {}
    if sub:
        rec = decode_layer_record(args, M, torch, w, replicate(plain, n_copies), PLAIN_LAYOUT, rank, world, local,
                                  with_e2e=False)
        subs["flash_layer_t1_plain_q2k"] = sub_summary(rec)
    del plain
    torch.cuda.empty_cache()
    if sub:
        subs["flash_prefill_t4096"] = sub_summary(
            prefill_record(args, M, torch, synth.WORKLOADS[3], rank, world, local, with_e2e=False))
        if stack_pool is not None:
            pool, shms, per = stack_pool
            t_gen = time.perf_counter()
            devs, Wrs, biases = stack_layers(w4, M, torch, pool, shms, per, r16=True)
            rec = stack_record(args, M, torch, w4, devs, Wrs, biases, R16_LAYOUT, rank, world, local,
                               with_e2e=False)
            rec["config"]["weights_generated_s"] = round(time.perf_counter() - t_gen, 1)
            subs["flash_stack43_t1"] = sub_summary(rec)
            del devs
            torch.cuda.empty_cache()
    if rank == 0:
        if not args.no_cpu_baseline and not args.timed_only:
            main["cpu_baseline"] = cpu_baseline(w, args.cpu_tokens or 2 * cores_available(), batch0=50_000)
        line = line_from(main, args, world, DECODE_DTYPE)
        if subs:
            line["sub"] = subs
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_decode(args, w: synth.Workload):
    """One decode workload alone (plain block layouts, or the tile order with --r16)."""
    import torch
    rank, world, local = init_dist(torch)
    M = load_library(rank, world)
    dev = device_layer(w, M, torch)
    layout = PLAIN_LAYOUT if w.gate.qtype == synth.Q2_K else "plain block layouts"
    if args.r16:
        dev = dev.repacked_r16()
        layout = R16_LAYOUT
    rec = decode_layer_record(args, M, torch, w, replicate(dev, max(1, args.copies)), layout, rank, world, local,
                              with_e2e=not args.timed_only)
    if rank == 0:
        if not args.no_cpu_baseline and not args.timed_only:
            rec["cpu_baseline"] = cpu_baseline(w, args.cpu_tokens or 2 * cores_available(), batch0=50_000)
        print(json.dumps(line_from(rec, args, world, DECODE_DTYPE)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_prefill(args, w: synth.Workload):
    import torch
    rank, world, local = init_dist(torch)
    M = load_library(rank, world)
    rec = prefill_record(args, M, torch, w, rank, world, local, with_e2e=not args.timed_only)
    if rank == 0:
        if not args.no_cpu_baseline and not args.timed_only:
            rec["cpu_baseline"] = cpu_baseline(w, args.cpu_tokens or 2 * cores_available(), batch0=50_000)
        print(json.dumps(line_from(rec, args, world, PREFILL_DTYPE)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_stack(args, w: synth.Workload):
    import torch
    rank, world, local = init_dist(torch)
    M = load_library(rank, world)
    pool, shms, per = start_stack_pool(w)  # spawned: no CUDA state inherited
    t_gen = time.perf_counter()
    r16 = args.r16 and w.T == 1
    devs, Wrs, biases = stack_layers(w, M, torch, pool, shms, per, r16=r16)
    t_gen = time.perf_counter() - t_gen
    rec = stack_record(args, M, torch, w, devs, Wrs, biases, R16_LAYOUT if r16 else PLAIN_LAYOUT, rank, world,
                       local, with_e2e=not args.timed_only)
    rec["config"]["weights_generated_s"] = round(t_gen, 1)
    if rank == 0:
        if not args.no_cpu_baseline and not args.timed_only:
            n = args.cpu_tokens or max(2, cores_available() // 2)
            cpu = cpu_baseline(w, n, batch0=50_000)
            cpu["value"] /= w.n_layers
            cpu["sample"] = (f"{n} tokens through layer 0 (route + selected expert FFNs + combine, fp64 C oracle, "
                             f"OpenMP over tokens), tokens/s divided by the {w.n_layers} layers")
            rec["cpu_baseline"] = cpu
        print(json.dumps(line_from(rec, args, world, DECODE_DTYPE)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_quantize(args, w: synth.Workload):
    """Device float-input quantizer: 16 fp32 expert matrices (d_ff x d_model,
    512 MiB, larger than L2) -> Q2_K / Q4_1 blocks with per-column
    importance; values/s and the input-read bandwidth against HBM."""
    import torch
    torch.cuda.set_device(0)
    from bit_quantized_moe_q2_gb300 import _build
    _build.build()
    import bit_quantized_moe_q2_gb300 as M
    from bit_quantized_moe_q2_gb300.device import check_status
    q = {"q2_k": M.DS4MOE_Q2_K, "q4_1": M.DS4MOE_Q4_1}[args.quantize]
    rows, cols, n_mat = w.d_ff, w.d_model, 16
    n = rows * cols * n_mat
    g = torch.Generator(device="cuda").manual_seed(w.seed)
    x = torch.randn(n, device="cuda", generator=g) * 0.02
    imp = torch.rand(cols, device="cuda", generator=g) ** 2
    out = torch.empty(n // M.block_values(q) * M.block_bytes(q), dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    steps = max(3, min(args.steps, 50))
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup if args.warmup < 50 else 3)):
            M.ds4moe_quantize_f32(q, x, imp, out, ws, cols=cols, stream=stream)
    check_status(ws, stream)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps):
            M.ds4moe_quantize_f32(q, x, imp, out, ws, cols=cols, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1) / steps
    check_status(ws, stream)
    peak, kind = measured_peaks()
    gbs = (n * 4 + out.numel()) / (ms / 1000) / 1e9
    print(json.dumps({"metric": "quantized values/s", "value": n / (ms / 1000), "unit": "values/s", "n_gpus": 1,
                      "steps": steps, "ms_per_step": ms, "higher_is_better": True, "dtype": "f32",
                      "data": "synthetic", "config": {"workload": f"quantize-{args.quantize}-16x{rows}x{cols}",
                                                       "importance": True, "l2": "512 MiB input per step"},
                      "roofline": {"kernel": "quantize_f32", "bound": "hbm", "achieved": gbs, "peak": peak,
                                   "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                                   "algorithmic_bytes_per_launch": n * 4 + out.numel(),
                                   "peak_source": kind}}), flush=True)


def run_shared(args, w: synth.Workload):
    """The shared expert alone (ds4moe_shared_ffn): bf16 w1, w3 [Fs, D] and w2
    [D, Fs], seeded N(0, 0.02) weights, x ~ N(0, 1) bf16, out accumulated
    into.  8 weight copies rotate (8 x 50 MB > L2 at the Flash shape).  The
    pages give no width: --shared sets it.  Up to 64 tokens: weight-stream
    GB/s against HBM; more: TFLOP/s against the sustained bf16 peak."""
    import torch
    rank, world, local = init_dist(torch)
    M = load_library(rank, world)
    from bit_quantized_moe_q2_gb300.device import check_status
    D, Fs, T = w.d_model, args.shared, max(1, args.tokens or 1)
    g = torch.Generator(device="cuda").manual_seed(w.seed)
    bits = lambda shape: (torch.randn(shape, device="cuda", generator=g) * 0.02).to(torch.bfloat16).view(torch.int16)
    n_copies = 8
    W = [(bits((Fs, D)), bits((Fs, D)), bits((D, Fs))) for _ in range(n_copies)]
    xs = [(torch.randn((T, D), device="cuda", generator=g)).to(torch.bfloat16).view(torch.int16) for _ in range(2)]
    out = torch.zeros((T, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(M.ds4moe_shared_workspace_bytes(D, Fs, T), dtype=torch.uint8, device="cuda")
    M.ds4moe_workspace_init(ws)
    stream = torch.cuda.Stream()

    def step(i):
        w1, w3, w2 = W[i % n_copies]
        M.ds4moe_shared_ffn(w1, w3, w2, xs[i % 2], out, ws, accumulate=True, stream=stream)

    graphs = []
    with torch.cuda.stream(stream):
        for i in range(n_copies):
            step(i)
    stream.synchronize()
    check_status(ws, stream)
    for j in range(n_copies):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            step(j)
        graphs.append(gr)

    def replay(i):
        graphs[i % n_copies].replay()

    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            replay(i)
    stream.synchronize()
    steps = args.steps if T <= 64 else max(3, min(args.steps, 200))
    ms, clocks = measure_clocks(torch, stream, replay, gpu_index(local), steps, world)
    check_status(ws, stream)
    step_s = ms / steps / 1000.0
    kernels = span_pass(M, torch, stream, replay, min(steps, 50))
    wbytes = 3 * D * Fs * 2
    cfg = {"workload": f"shared-expert-bf16-d{D}-f{Fs}-t{T}", "d_model": D, "d_shared": Fs, "tokens_per_step": T,
           "weights": "bf16, seeded N(0, 0.02)", "l2": f"{n_copies} weight copies of {wbytes / 1e6:.0f} MB rotate"}
    line = {"metric": "shared-expert tokens/s", "value": world * T / step_s, "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 operands, f32 accumulate", "data": "synthetic",
            "config": cfg, "kernels": kernels, "clocks": clocks}
    if "shared_gate_up_tc" in kernels:
        flops = 2.0 * 3 * D * Fs * T
        us = kernels["shared_gate_up_tc"]["avg_us"] + kernels["shared_down_tc"]["avg_us"]
        peak, kind = measured_tensor_peak(sustained=True)
        line["tflops"] = flops / step_s / 1e12
        line["roofline"] = {"kernel": "shared-expert tcgen05 GEMMs (gate/up + SwiGLU, down + accumulate)",
                            "bound": "tensor", "achieved": flops / (us * 1e-6) / 1e12, "peak": peak,
                            "unit": "TFLOP/s", "frac": flops / (us * 1e-6) / 1e12 / peak, "traffic": None,
                            "algorithmic_flops_per_launch": flops, "avg_launch_us": us,
                            "timing": "device spans of the two kernels",
                            "peak_source": f"{kind} bf16_tflops_sustained"}
    else:
        algo = wbytes + T * D * 2 + 2 * T * D * 4
        peak, kind = measured_peaks()
        gbs = algo / step_s / 1e9
        line["roofline"] = {"kernel": "shared-expert GEMVs (gate/up + SwiGLU, down + accumulate), whole call",
                            "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                            "traffic": None, "algorithmic_bytes_per_launch": algo, "avg_launch_us": step_s * 1e6,
                            "timing": "CUDA events over graph replays of the call (two kernels)",
                            "peak_source": kind}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    w = synth.WORKLOADS[args.workload]
    if args.n_expert:
        w = w.replace(n_expert=args.n_expert)
    if args.tokens:
        w = w.replace(T=args.tokens)
    if args.prefill and w.path != "prefill":
        T = args.tokens or 4096
        w = w.replace(path="prefill", T=T, name=f"{w.name}@prefill-T{T}")
    if w.path not in ("decode", "prefill"):
        raise SystemExit("bench.py times workloads 0-5")
    if args.quantize:
        run_quantize(args, w)
        return
    if args.shared:
        run_shared(args, w)
        return
    default = args.workload == 1 and not args.n_expert and not args.tokens and not args.plain
    if args.impl == "reference":
        run_reference(args, w)
    elif w.n_layers > 1:
        run_stack(args, w)
    elif w.path == "prefill":
        run_prefill(args, w)
    elif default:
        run_default(args, w)
    else:
        run_decode(args, w)


if __name__ == "__main__":
    main()
