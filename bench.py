#!/usr/bin/env python
"""Benchmark of the routed-MoE expert FFN (route + gate/up + SwiGLU + down +
combine) on one GB300, through the libds4moe C ABI.

Workload (default): one DeepSeek-V4-Flash-shaped routed-MoE layer at decode
batch 1 -- d_model 4096, d_ff 2048, 256 experts, top-6 with a softmax over
the selected, gate/up/down all Q2_K, synthetic seeded weights and tokens.
A step is one pass of the whole path over one token.  Weights are
replicated into 8 device copies and tokens come from 16 pre-staged slots;
step i uses copy i % 8 and slot i % 16, so consecutive steps never re-read
bytes still resident in L2 (8 copies x 2.1 GB >> 129 MB of L2).

Printed JSON line: tokens/s (value), weight-stream GB/s and its fraction of
the measured HBM peak, the dominant kernel's roofline (gate/up GEMV, timed
with CUDA events on its launch stream), the CPU oracle as a baseline, the
end-to-end number through the C ABI with host buffers, and SM clocks sampled
during the timed region.

`--workload 3` times the prefill chunk instead: 4096 tokens per step (router
with bias, top-6 of 256, Q4_1 gate/up, Q2_K down) through ds4moe_route_topk +
ds4moe_ffn_prefill, reported as tokens/s and TFLOP/s with the tensor-core
roofline of the gate/up grouped GEMM.

`--workload 4` times the 43-layer decode stack (every layer with its own
router and 256 Q2_K experts, 91 GB resident; residual in fp32, each layer fed
bf16 of the RMS-normalised residual) through ds4moe_stack_decode, one CUDA graph per step; the
weights are generated on all host cores into shared memory, layer by layer.

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
METRIC = "routed-MoE tokens/s"
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
    """nvidia-smi sampling of SM clocks and throttle reasons."""

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                    "-i", str(gpu_index), "-lms", str(period_ms)]
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, begin: bool):
        if begin:
            self.t0 = datetime.now()
        else:
            self.t1 = datetime.now()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                continue
            rows.append((ts, f))
        inside = [f for ts, f in rows if self.t0 and self.t1 and self.t0 <= ts <= self.t1]
        use = inside if inside else [f for _, f in rows]
        sm = [float(f[2]) for f in use if f[2].replace(".", "").isdigit()]
        smax = [float(f[3]) for f in use if f[3].replace(".", "").isdigit()]
        reasons = set()
        for f in use:
            for name, v in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), f[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use), "samples_in_region": len(inside)}


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
# current build (dram__bytes_read.sum + dram__bytes_write.sum), keyed by (workload,
# kernel); a pair missing here reports null.  The summaries with the commands are in profiles/.
NCU_TRAFFIC: dict = {
    # k_ffn_t1 (merged single-token FFN grid), mean of three launches: 49.63 MB read + 46 KB written
    ("flash-layer-decode-t1-q2k", "ffn_t1"): 49_675_008,
}


def dominant_kernel(prof: dict, w: synth.Workload, uniq_avg: float):
    """The decode step's dominant kernel in the library's per-kernel timings:
    the merged single-token FFN grid where it ran (expert weights + x + out
    per launch), else the gate/up kernel (gate/up weights + x + h).
    Returns (name, description, algorithmic bytes per launch, total ms, launches)."""
    T, k, D = w.T, w.k, w.d_model
    if "ffn_t1" in prof:
        ms, n = prof["ffn_t1"]
        return ("ffn_t1", "expert FFN (merged gate/up + SwiGLU + down + combine, dequant fused)",
                uniq_avg * expert_bytes(w) + T * D * 2 + T * D * 4, ms, n)
    ms, n = prof.get("gate_up", prof.get("gate_up_simt", (float("nan"), 1)))
    return ("gate_up", "gate_up (fused dequant GEMV + SwiGLU)",
            uniq_avg * gate_up_bytes(w) + T * D * 2 + T * k * w.d_ff * 2, ms, n)


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
def run_ours(args, w: synth.Workload):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from bit_quantized_moe_q2_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    import bit_quantized_moe_q2_gb300 as M
    from bit_quantized_moe_q2_gb300.device import check_status, workspace

    dev = device_layer(w, M, torch)
    n_copies = max(1, args.copies)
    copies = [dev] + [type(dev)(dev.d_model, dev.d_ff, dev.n_expert, dev.q_gate, dev.q_up, dev.q_down,
                                dev.gate.clone(), dev.up.clone(), dev.down.clone()) for _ in range(n_copies - 1)]
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
        c = copies[i % n_copies]
        M.ds4moe_moe_decode(c.abi, xs[j], Wr_d, b_d, k, out[j], idx[j], wt[j], ws, s)

    with torch.cuda.stream(stream):
        for i in range(2 * N_SLOTS):
            step(i)
    check_status(ws, stream)
    # per-slot unique experts (algorithmic bytes)
    uniq = [len(set(idx[j].cpu().numpy().ravel().tolist())) for j in range(N_SLOTS)]

    # one CUDA graph per step position (slot j uses copy j % N_COPIES)
    graphs = []
    for j in range(N_SLOTS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(j)
        graphs.append(g)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % N_SLOTS].replay()
    stream.synchronize()
    check_status(ws, stream)

    # ---- timed region: exactly K steps
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else local
    sampler = ClockSampler(gpu_index)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark(True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            graphs[i % N_SLOTS].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier(world)
    clocks = sampler.stop()
    ms = reduce_max(ev0.elapsed_time(ev1), world)
    check_status(ws, stream)

    tokens = world * args.steps * T
    value = tokens / (ms / 1000.0)
    ms_per_step = ms / args.steps
    eb = expert_bytes(w)
    algo_step = [u * eb + Wr.nbytes + (0 if bias is None else bias.nbytes) + T * D * 2 + T * D * 4 for u in uniq]
    algo_bytes = sum(algo_step[i % N_SLOTS] for i in range(args.steps))
    stream_gbs = algo_bytes / (ms / 1000.0) / 1e9 / 1.0 * 1.0
    peak, peak_kind = measured_peaks()

    if args.timed_only:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": world * args.steps * T / (ms / 1000.0), "unit": "tokens/s",
                              "ms_per_step": ms / args.steps, "steps": args.steps, "note": "timed-only run"}),
                  flush=True)
        return
    # ---- per-kernel roofline: same steps, eager ABI calls with the library's
    # event profiling on (CUDA events on the launch stream around each kernel)
    kp = min(args.steps, 2000)
    M.ds4moe_profile_enable(True)
    with torch.cuda.stream(stream):
        for i in range(kp):
            step(i, stream)
    stream.synchronize()
    prof = M.ds4moe_profile_read()
    M.ds4moe_profile_enable(False)
    launches_per_step = sum(n for _, n in prof.values()) / kp
    kname, kdesc, gu_algo, gu_ms, gu_n = dominant_kernel(prof, w, sum(uniq[i % N_SLOTS] for i in range(kp)) / kp)
    gu_avg_s = gu_ms / gu_n / 1000.0
    roofline = {"kernel": kdesc, "bound": "hbm",
                "achieved": gu_algo / gu_avg_s / 1e9, "peak": peak, "unit": "GB/s",
                "frac": gu_algo / gu_avg_s / 1e9 / peak, "traffic": NCU_TRAFFIC.get((w.name, kname)),
                "algorithmic_bytes_per_launch": int(gu_algo), "avg_launch_us": gu_avg_s * 1e6,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else
                               "fallback 6.8 TB/s"}
    kernels = {n: {"avg_us": 1000 * t / c, "launches_per_step": c / kp} for n, (t, c) in prof.items()}

    # ---- end to end through the C ABI with host buffers
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
            c = copies[i % n_copies]
            M.ds4moe_moe_decode(c.abi, x_in, Wr_d, b_d, k, out[0], idx[0], wt[0], ws, stream)
            oh.copy_(out[0], non_blocking=True)
            stream.synchronize()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), world)
    e2e = {"value": world * ke * T / (e2e_ms / 1000.0), "unit": "tokens/s", "steps": ke,
           "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 4,
           "path": "pinned H2D x, ds4moe_moe_decode (eager C-ABI call), D2H out, stream sync per step"}

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        n = args.cpu_tokens or 2 * cores_available()
        cpu = cpu_baseline(w, n, batch0=50_000)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 accumulate over exact 2-bit codes and bf16 activations",
            "data": "synthetic", "config": workload_config(w, n_copies),
            "weight_stream_gbs": stream_gbs, "hbm_frac": stream_gbs / peak,
            "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(round(launches_per_step * args.steps)), "clocks": clocks}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------- prefill chunk arm
def run_ours_prefill(args, w: synth.Workload):
    """Prefill: route (with bias) + tensor-core expert FFN over T tokens per
    step.  Inputs (3.4 GB of weights) far exceed L2, so no flush is needed."""
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from bit_quantized_moe_q2_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    import bit_quantized_moe_q2_gb300 as M
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

    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else local
    sampler = ClockSampler(gpu_index)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark(True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier(world)
    clocks = sampler.stop()
    ms = reduce_max(ev0.elapsed_time(ev1), world)
    check_status(ws, stream)
    flops_step, flops_gu = prefill_flops(w)
    value = world * args.steps * T / (ms / 1000.0)
    tflops = world * args.steps * flops_step / (ms / 1000.0) / 1e12
    if args.timed_only:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "tokens/s", "tflops": tflops,
                              "ms_per_step": ms / args.steps, "steps": args.steps, "note": "timed-only run"}),
                  flush=True)
        return

    # per-kernel times (CUDA events around each launch on its stream)
    kp = min(args.steps, 10)
    M.ds4moe_profile_enable(True)
    with torch.cuda.stream(stream):
        for i in range(kp):
            step(i)
    stream.synchronize()
    prof = M.ds4moe_profile_read()
    M.ds4moe_profile_enable(False)
    launches_per_step = sum(n for _, n in prof.values()) / kp
    kernels = {n: {"avg_us": 1000 * t / c, "launches_per_step": c / kp} for n, (t, c) in prof.items()}
    gu_ms, gu_n = prof.get("gate_up_tc", (float("nan"), 1))
    gu_s = gu_ms / gu_n / 1000.0
    peak, peak_kind = measured_tensor_peak(sustained=True)
    roofline = {"kernel": "gate_up_tc (tcgen05 grouped GEMM, fused Q4_1 dequant + SwiGLU)", "bound": "tensor",
                "achieved": flops_gu / gu_s / 1e12, "peak": peak, "unit": "TFLOP/s",
                "frac": flops_gu / gu_s / 1e12 / peak, "traffic": None,
                "algorithmic_flops_per_launch": flops_gu, "avg_launch_us": gu_s * 1e6,
                "peak_source": f"{peak_kind} bf16_tflops_sustained (kind::f16 runs at the bf16 rate)"}

    # end to end with host buffers: pinned x in, out back, per step
    ke = min(args.steps, 5)
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
    e2e = {"value": world * ke * T / (e2e_ms / 1000.0), "unit": "tokens/s", "steps": ke,
           "h2d_bytes_per_step": T * D * 2, "d2h_bytes_per_step": T * D * 4,
           "path": "pinned H2D x, ds4moe_route_topk + ds4moe_ffn_prefill (C-ABI calls), D2H out, sync per step"}
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        n = args.cpu_tokens or 2 * cores_available()
        cpu = cpu_baseline(w, n, batch0=50_000)
    cfg = workload_config(w, 1)
    cfg["l2"] = "inputs larger than L2: every step streams 3.4 GB of expert weights"
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16 tensor-core operands (exact gate/up split), f32 accumulate",
            "data": "synthetic", "config": cfg, "tflops": tflops,
            "tensor_frac": tflops / peak, "roofline": roofline, "kernels": kernels,
            "expert_load": {"max": int(counts.max()), "min": int(counts.min()), "empty": int((counts == 0).sum())},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(round(launches_per_step * args.steps)),
            "clocks": clocks}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


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


def run_ours_stack(args, w: synth.Workload):
    import multiprocessing as mp
    from multiprocessing import shared_memory
    rank, world, local = dist_env()
    from bit_quantized_moe_q2_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    # the generator pool starts (spawn) before the first GPU call
    per = {t: tensor_bytes(w, t) for t in (synth.T_GATE, synth.T_UP, synth.T_DOWN)}
    shms = [shared_memory.SharedMemory(create=True, size=w.n_expert * per[t])
            for t in (synth.T_GATE, synth.T_UP, synth.T_DOWN)]
    pool = mp.get_context("spawn").Pool(max(1, cores_available()), initializer=_pool_init)
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    barrier(world)
    import bit_quantized_moe_q2_gb300 as M
    from bit_quantized_moe_q2_gb300.device import DeviceLayer, check_status, workspace
    qid = {synth.Q4_1: M.DS4MOE_Q4_1, synth.Q2_K: M.DS4MOE_Q2_K, synth.Q4_K: M.DS4MOE_Q4_K}
    t_gen = time.perf_counter()
    devs, Wrs, biases = [], [], []
    names = [sh.name for sh in shms]
    try:
        for layer in range(w.n_layers):
            pool.map(_pack_expert, [(w, layer, e, names, per) for e in range(w.n_expert)], chunksize=4)
            dev = DeviceLayer.empty(w.d_model, w.d_ff, w.n_expert, qid[w.gate.qtype], qid[w.up.qtype],
                                    qid[w.down.qtype])
            for sh, dst in zip(shms, (dev.gate, dev.up, dev.down)):
                dst.copy_(torch.frombuffer(sh.buf, dtype=torch.uint8, count=dst.numel()))
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
    t_gen = time.perf_counter() - t_gen
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
        x_res.copy_(x0[j], non_blocking=True)
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
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % N_SLOTS].replay()
    stream.synchronize()
    check_status(ws, stream)

    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").replace(",", "").isdigit() else local
    sampler = ClockSampler(gpu_index)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark(True)
    ev0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            graphs[i % N_SLOTS].replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    barrier(world)
    clocks = sampler.stop()
    ms = reduce_max(ev0.elapsed_time(ev1), world)
    check_status(ws, stream)
    value = world * args.steps * T / (ms / 1000.0)
    eb = expert_bytes(w)
    algo_step = sum(u * eb for u in uniq) + L * (w.n_expert * D * 4) + T * D * 4 * 2
    stream_gbs = algo_step / (ms / args.steps / 1000.0) / 1e9
    peak, peak_kind = measured_peaks()
    if args.timed_only:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": "tokens/s", "ms_per_step": ms / args.steps,
                              "steps": args.steps, "note": "timed-only run"}), flush=True)
        return
    kp = min(args.steps, 50)
    M.ds4moe_profile_enable(True)
    with torch.cuda.stream(stream):
        for i in range(kp):
            step(i % N_SLOTS, stream)
    stream.synchronize()
    prof = M.ds4moe_profile_read()
    M.ds4moe_profile_enable(False)
    launches_per_step = sum(n for _, n in prof.values()) / kp
    kernels = {n: {"avg_us": 1000 * t / c, "launches_per_step": c / kp} for n, (t, c) in prof.items()}
    kname, kdesc, gu_algo, gu_ms, gu_n = dominant_kernel(prof, w, sum(uniq) / L)
    gu_s = gu_ms / gu_n / 1000.0
    roofline = {"kernel": kdesc + ", per layer", "bound": "hbm",
                "achieved": gu_algo / gu_s / 1e9, "peak": peak, "unit": "GB/s", "frac": gu_algo / gu_s / 1e9 / peak,
                "traffic": None, "algorithmic_bytes_per_launch": int(gu_algo), "avg_launch_us": gu_s * 1e6,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else
                               "fallback 6.8 TB/s"}
    # end to end: pinned x in, x_res out, per step
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
    e2e = {"value": world * ke * T / (e2e_ms / 1000.0), "unit": "tokens/s", "steps": ke,
           "h2d_bytes_per_step": T * D * 4, "d2h_bytes_per_step": T * D * 4,
           "path": "pinned H2D x_res, ds4moe_stack_decode (eager C-ABI call, 43 layers), D2H x_res, sync per step"}
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        n = args.cpu_tokens or max(2, cores_available() // 2)
        cpu = cpu_baseline(w, n, batch0=50_000)
        cpu["value"] /= L
        cpu["sample"] = (f"{n} tokens through layer 0 (route + selected expert FFNs + combine, fp64 C oracle, "
                         f"OpenMP over tokens), tokens/s divided by the {L} layers")
    cfg = workload_config(w, 1)
    cfg["n_layers"] = L
    cfg["l2"] = f"inputs larger than L2: every step streams {L} layers of expert weights"
    cfg["weights_generated_s"] = round(t_gen, 1)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 accumulate over exact 2-bit codes and bf16 activations",
            "data": "synthetic", "config": cfg, "weight_stream_gbs": stream_gbs, "hbm_frac": stream_gbs / peak,
            "roofline": roofline, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(round(launches_per_step * args.steps)), "clocks": clocks}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def oracle_free_bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (a bit shift; no method arithmetic)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


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


def main(argv=None):
    args = parse_args(argv)
    w = synth.WORKLOADS[args.workload]
    if args.n_expert:
        w = w.replace(n_expert=args.n_expert)
    if args.tokens:
        w = w.replace(T=args.tokens)
    if w.path not in ("decode", "prefill"):
        raise SystemExit("bench.py times workloads 0-5")
    if args.quantize:
        run_quantize(args, w)
        return
    if args.impl == "reference":
        run_reference(args, w)
    elif w.n_layers > 1:
        run_ours_stack(args, w)
    elif w.path == "prefill":
        run_ours_prefill(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
