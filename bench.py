"""Benchmark: one single-token decode step of a Gemma-3-4B-shaped model.

step = qws_decode_chain over 34 layers (Q4_K q/k/v/o/gate/up, Q6_K down,
       sandwich rms_norms) + final rms_norm + Q4_0 lm_head (262144 x 2560).
Metric: achieved HBM GB/s of the packed-weight stream (+ vector bytes), with
microseconds per token of the 34-layer chain reported alongside.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
       [--n-layers L]   (a shorter chain, for small profiler captures only)
       [--op OP --batch B]  time one operation alone, back to back (not the
                        decode step): lm_head_q4_0 (f32 activations),
                        lm_head_q8 (quantize_q8 + Q4_0 x Q8_0 matvec),
                        lm_head_q4_k / lm_head_q6_k (the same 262144 x 2560
                        shape in Q4_K / Q6_K, f32 activations),
                        matvec_q4k (Q4_K 2560 x 2560), qkv (fused Q/K/V
                        4096 x 2560 + O 2560 x 2048), ffn (fused gate/up
                        GEGLU + Q6_K down, 2560/10240): each back to back
                        over a ring of weight copies >= 4 x L2 (a CUDA graph
                        of the calls; also launched one at a time) and
                        isolated after an L2 flush,
                        prefill (Q4_K 10240 x 2560 times --batch tokens on the
                        tensor cores; TFLOP/s),
                        kv_attention (one token over 32768 cached positions,
                        Gemma-3-4B heads: 8 query, 4 kv, head_dim 256),
                        decode_kv (all layers of a decode step over a KV
                        cache at --pos, default 1024)
For N > 1 launch with torchrun; every rank runs an independent replica of the
step on its own GPU (the path has no data exchange; "replicas only").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("Q4_K GEMV achieved HBM GB/s (% of GB300 peak); µs/token for 34-layer chain")
WORKLOAD = ("decode step, batch 1: 34-layer Gemma-3-4B chain (hidden 2560, inter 10240, q 8x256, "
            "kv 4x256; Q4_K q/k/v/o/gate/up, Q6_K down, rms_norm eps 1e-6 sandwich norms, "
            "attention at seq 1) + final rms_norm + Q4_0 lm_head 262144x2560")
N_LAYERS = 34
VOCAB = 262144
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["engine.cuh", "formats.cuh", "device_common.cuh", "chain.cu"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for n in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "quantized_weight_streaming_q4k_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense f16/bf16 tensor peak (same nominal rate for both): the measured
    cuBLAS bf16 burst figure, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured (bf16 burst; f16 has the same nominal rate)"
    return 1900.0, "fallback"


def profiled_traffic(n_layers=N_LAYERS):
    """dram bytes per chain launch from the committed ncu summary, if it was
    taken on the current kernel sources (else None).  The summary holds the
    bytes per layer of a shorter chain (traffic is per layer plus a small
    constant), scaled here by the number of layers."""
    p = os.path.join(ROOT, "profiles", "chain_kernel_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_hash():
        return None
    return float(d["bytes_per_layer"]) * n_layers


def algorithmic_bytes(dims, n_layers=N_LAYERS):
    from quantized_weight_streaming_q4k_gb300 import synth
    H, I = dims["hidden"], dims["inter"]
    qd = dims["n_q_heads"] * dims["head_dim"]
    kd = dims["n_kv_heads"] * dims["head_dim"]
    q4k = lambda r, c: synth.n_blocks(synth.Q4_K, r, c) * 144
    q6k = lambda r, c: synth.n_blocks(synth.Q6_K, r, c) * 210
    layer_w = q4k(qd + 2 * kd, H) + q4k(H, qd) + 2 * q4k(I, H) + q6k(H, I)
    norm_w = 4 * H * 4
    chain = n_layers * (layer_w + norm_w) + 2 * H * 4          # + h in and out
    lm_head = synth.n_blocks(synth.Q4_0, VOCAB, H) * 18 + H * 4 + VOCAB * 4
    final_norm = 3 * H * 4
    return chain, final_norm, lm_head


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, ident: str):
        self.ident = ident
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.ident}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_init(backend: str = "nccl"):
    """Rank, world and local rank from the torchrun environment; joins the
    process group when world > 1 (NCCL on GPUs; gloo for the CPU tests)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(v: float, world: int, device: str = "cuda") -> float:
    """The largest v over all ranks (every rank gets it)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank_step: float, ms_per_step_max: float, world: int) -> float:
    """Whole-job GB/s: every rank streams its own replica of the step, the job
    takes as long as its slowest rank."""
    return world * bytes_per_rank_step / (ms_per_step_max * 1e-3) / 1e9


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
def _oracle_layers_worker(layer_ids, barrier, out_q):
    """One host process of the all-core oracle timing: builds its layers
    (untimed), waits for the others, then runs the oracle on each layer."""
    import oracle
    from quantized_weight_streaming_q4k_gb300 import synth
    dims = synth.GEMMA3_4B
    layers = [synth.chain_layer(l % N_LAYERS, dims) for l in layer_ids]
    h = synth.normal_vector(synth.rng(synth.W_CHAIN, 99), dims["hidden"]).astype(np.float64)
    barrier.wait()
    t0 = time.time()
    for L in layers:
        h = oracle.layer_forward(L, dims, h)
    out_q.put((t0, time.time(), len(layer_ids)))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_oracle_sample(max_seconds: float = 15.0):
    """Times the oracle (as it stands) on a bounded sample of the same step:
    whole decoder layers of the chain workload.  Two figures: one host thread
    over up to 34 layers (at most ~max_seconds), and every host core at once,
    one process per core (spawned, so no process is forked from this one after
    its GPU work), each running its own layers (about max_seconds of CPU work
    in all); the all-core value is the packed bytes of all layers over the
    wall time from the common start to the last finish."""
    import multiprocessing as mp

    import oracle
    from quantized_weight_streaming_q4k_gb300 import synth
    dims = synth.GEMMA3_4B
    chain_b, _, _ = algorithmic_bytes(dims)
    per_layer = chain_b / N_LAYERS
    h = synth.normal_vector(synth.rng(synth.W_CHAIN, 99), dims["hidden"]).astype(np.float64)
    layers_done = 0
    elapsed = 0.0
    while True:
        L = synth.chain_layer(layers_done % N_LAYERS, dims)
        t1 = time.perf_counter()
        h = oracle.layer_forward(L, dims, h)
        elapsed += time.perf_counter() - t1
        layers_done += 1
        if elapsed > max_seconds or layers_done >= N_LAYERS:
            break
    single = per_layer * layers_done / elapsed / 1e9

    cores = host_cores()
    n_proc = max(1, min(cores, N_LAYERS))
    # about max_seconds of CPU work over all processes (each layer costs about
    # what it cost the single thread), at most 34 layers per process
    t_layer = elapsed / layers_done
    per_proc = int(max(1, min(N_LAYERS, round(max_seconds / (n_proc * t_layer)))))
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(n_proc)
    out_q = ctx.Queue()
    procs = [ctx.Process(target=_oracle_layers_worker,
                         args=(list(range(i * per_proc, (i + 1) * per_proc)), barrier, out_q))
             for i in range(n_proc)]
    for p in procs:
        p.start()
    res = [out_q.get(timeout=600) for _ in procs]
    for p in procs:
        p.join()
    t_start = min(r[0] for r in res)
    t_end = max(r[1] for r in res)
    n_all = sum(r[2] for r in res)
    wall = t_end - t_start
    return {"value": per_layer * n_all / wall / 1e9, "unit": "GB/s", "cores": n_proc,
            "kind": "oracle",
            "sample": f"{n_all} decoder layers of the same workload ({per_proc} per process, "
                      f"{per_layer * n_all / 1e6:.0f} MB of packed weights), f64 oracle, "
                      f"{n_proc} host processes at once ({cores} cores available), "
                      f"{wall:.1f} s wall",
            "single_thread": {"value": single, "unit": "GB/s", "cores": 1,
                              "sample": f"{layers_done} layers, {elapsed:.1f} s on 1 host "
                                        "thread"}}


def run_reference(args, world, rank):
    """The reference arm: the f64 CPU oracle, timed on the host's cores."""
    if rank != 0:
        return
    import oracle
    from quantized_weight_streaming_q4k_gb300 import synth
    dims = synth.GEMMA3_4B
    chain_b, _, _ = algorithmic_bytes(dims)
    per_layer = chain_b / N_LAYERS
    h = synth.normal_vector(synth.rng(synth.W_CHAIN, 99), dims["hidden"]).astype(np.float64)
    L = synth.chain_layer(0, dims)
    for _ in range(max(0, min(args.warmup, 1))):
        oracle.layer_forward(L, dims, h)
    times = []
    for s in range(args.steps):
        t = time.perf_counter()
        h = oracle.layer_forward(L, dims, h)
        times.append(time.perf_counter() - t)
    tot = sum(times)
    value = per_layer * len(times) / tot / 1e9
    out = {"metric": METRIC, "value": value, "unit": "GB/s", "impl": "reference",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": 1e3 * tot / len(times), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": WORKLOAD, "sample": "one decoder layer per step"},
           "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                            "sample": "one of the 34 decoder layers per step (59.8 MB of "
                                      "packed weights), f64 oracle, 1 host thread"},
           "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def run_gpu(args, world, rank, local):
    import torch

    from quantized_weight_streaming_q4k_gb300 import build, ops, synth
    build.build()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    dims = synth.GEMMA3_4B
    H = dims["hidden"]
    n_layers = args.n_layers
    chain_b, fnorm_b, lm_b = algorithmic_bytes(dims, n_layers)

    # ---- inputs, resident in HBM
    layers = []
    for l in range(n_layers):
        L = synth.chain_layer(l, dims)
        layers.append({k: (torch.from_numpy(v).to(dev) if isinstance(v, np.ndarray) else v)
                       for k, v in L.items()})
    structs = [ops.make_layer(L) for L in layers]
    g = synth.rng(synth.W_LM_HEAD, 0)
    W_lm = torch.from_numpy(synth.q4_0_matrix(g, VOCAB, H)).to(dev)
    w_final = torch.from_numpy(synth.norm_weights(synth.rng(synth.W_CHAIN, synth.T_NFINAL), H)).to(dev)
    h0 = torch.from_numpy(synth.normal_vector(synth.rng(synth.W_CHAIN, 99), H)).to(dev)
    h = torch.empty_like(h0)
    hn = torch.empty_like(h0)
    logits = torch.empty(VOCAB, device=dev)
    ws = torch.empty(ops.workspace_bytes(ops.OP_DECODE_CHAIN, 0, H, dims["inter"]),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        h.copy_(h0)
        if ev:
            ev[0].record(stream)
        # the 34 layers and the final norm (hn) in one launch
        ops.decode_chain(structs, h, dims, workspace=ws, w_final=w_final, hn=hn)
        if ev:
            ev[1].record(stream)
        ops.q4_0_matvec(W_lm, hn, VOCAB, H, out=logits)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert ops.device_error() == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
           for _ in range(min(args.steps, 500))]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    ident = (uuid if uuid.startswith("GPU-") else f"GPU-{uuid}") if uuid else str(local)
    clocks = ClockSampler(ident)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = start.elapsed_time(stop)
    assert ops.device_error() == 0
    total_ms = max_over_ranks(total_ms, world)
    # the split of a step between the chain (with the final norm) and the lm_head, from
    # a second run of steps with events between the kernels (an event there
    # keeps the lm_head's launch from overlapping the chain's last CTAs, so
    # the step itself is timed above without them)
    for i in range(len(evs)):
        step(evs[i])
    torch.cuda.synchronize()
    chain_ms = [a.elapsed_time(b) for a, b, _ in evs]
    lm_ms = [b.elapsed_time(c) for _, b, c in evs]

    # ---- end to end through host buffers (pinned): h0 in, logits out
    h_host = h0.cpu().pin_memory()
    logits_host = torch.empty(VOCAB, dtype=torch.float32).pin_memory()

    def step_e2e():
        h.copy_(h_host, non_blocking=True)
        ops.decode_chain(structs, h, dims, workspace=ws, w_final=w_final, hn=hn)
        ops.q4_0_matvec(W_lm, hn, VOCAB, H, out=logits)
        logits_host.copy_(logits, non_blocking=True)

    for _ in range(args.warmup):
        step_e2e()
    torch.cuda.synchronize()
    e_steps = max(1, min(args.steps, 200))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(e_steps):
        step_e2e()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b), world) / e_steps

    bytes_step = chain_b + fnorm_b + lm_b
    ms_step = total_ms / args.steps
    value = job_throughput(bytes_step, ms_step, world)
    chain_avg = statistics.mean(chain_ms)
    peak, peak_kind = peaks()
    achieved = chain_b / (chain_avg * 1e-3) / 1e9
    if rank != 0:
        return
    workload = WORKLOAD if n_layers == N_LAYERS else WORKLOAD.replace(
        f"{N_LAYERS}-layer", f"{n_layers}-layer (profiling case)")
    out = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded random Q4_K/Q6_K/Q4_0 blocks, Gemma-3-4B shapes)",
        "config": {"workload": workload, "n_layers": n_layers, "vocab": VOCAB, "batch": 1,
                   "l2": f"inputs larger than L2: {bytes_step / 1e9:.2f} GB of weights "
                         "streamed per step",
                   "parallelism": f"replicas x{world}"},
        "chain_us_per_token": 1e3 * chain_avg,
        "lm_head_us": 1e3 * statistics.mean(lm_ms),
        "bytes_per_step": bytes_step,
        "roofline": {"bound": "hbm", "kernel": f"chain_kernel ({n_layers}-layer decode chain + final norm)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "traffic": profiled_traffic(n_layers)},
        "e2e": {"value": job_throughput(bytes_step, e2e_ms, world), "unit": "GB/s",
                "h2d_bytes_per_step": H * 4, "d2h_bytes_per_step": VOCAB * 4,
                "ms_per_step": e2e_ms},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    if world == 1 and not args.no_cpu_baseline and n_layers == N_LAYERS:
        out["cpu_baseline"] = cpu_oracle_sample()
    print(json.dumps(out))


def run_decode_kv(args):
    """One decode step over a KV cache, all 34 Gemma-3-4B layers at position
    pos (qws_decode_kv), timed back to back; every step rewrites position pos,
    so each step does the same work.  Algorithmic bytes: the packed weights
    of every layer, the norm weights, the K and V rows of positions 0..pos
    read per layer, plus h in and out."""
    import torch

    from quantized_weight_streaming_q4k_gb300 import build, ops, synth
    build.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    dims = synth.GEMMA3_4B
    H, hd, nkv = dims["hidden"], dims["head_dim"], dims["n_kv_heads"]
    pos, max_seq = args.pos, args.pos + 64
    n_layers = args.n_layers
    layers, kcs, vcs = [], [], []
    for l in range(n_layers):
        L = synth.chain_layer(l, dims)
        layers.append({k: (torch.from_numpy(v).to(dev) if isinstance(v, np.ndarray) else v)
                       for k, v in L.items()})
        g = synth.rng(synth.W_CHAIN, 500, l)
        kcs.append(torch.from_numpy((0.5 * g.standard_normal((nkv, max_seq, hd))).astype(
            np.float32)).to(dev))
        vcs.append(torch.from_numpy(g.standard_normal((nkv, max_seq, hd)).astype(np.float32)).to(dev))
    structs = [ops.make_layer(L) for L in layers]
    h0 = torch.from_numpy(synth.normal_vector(synth.rng(synth.W_CHAIN, 99), H)).to(dev)
    h = torch.empty_like(h0)
    ws = torch.empty(ops.decode_kv_workspace_bytes(dims, max_seq), dtype=torch.uint8, device=dev)
    scale = 1.0 / np.sqrt(hd)

    def call():
        h.copy_(h0)
        ops.decode_kv(structs, h, dims, kcs, vcs, max_seq, pos, hd, 10000.0, scale, workspace=ws)

    chain_b, _, _ = algorithmic_bytes(dims, n_layers)
    kv_b = n_layers * 2 * nkv * (pos + 1) * hd * 4
    # head shapes whose attention runs inside the chain kernel: one launch per
    # group of up to 64 layers; else per layer split + merge + chain launch
    group = dims["n_q_heads"] // nkv
    if (hd == 256 and group <= 2) or (hd == 128 and group in (1, 2, 4)):
        kv_launches = -(-n_layers // 64)
        kv_kernel = ("chain_kernel with the attention inside the O phase's prologue "
                     "(one launch per token)")
    else:
        kv_launches = 1 + 3 * n_layers
        kv_kernel = ("decode_kv on the chain kernel (per layer: attention split with RoPE and "
                     "the K/V append fused in + merge + chain launch)")
    nbytes = chain_b + kv_b
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    clocks = ClockSampler((uuid if uuid.startswith("GPU-") else f"GPU-{uuid}") if uuid else "0")
    clocks.start()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(args.steps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert ops.device_error() == 0
    us = 1e3 * a.elapsed_time(b) / args.steps
    gbs = nbytes / (us * 1e-6) / 1e9
    peak, peak_kind = peaks()
    print(json.dumps({
        "metric": "decode step with KV cache: us/token and achieved HBM GB/s", "value": gbs,
        "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
        "us_per_token": us, "higher_is_better": True, "dtype": "f32",
        "data": "synthetic (seeded random blocks, random K/V cache contents)",
        "config": {"workload": f"{n_layers} Gemma-3-4B layers at position {pos} "
                               f"({pos + 1} cached positions, 4 kv heads of 256), batch 1",
                   "l2": f"{nbytes / 1e9:.2f} GB streamed per token (> L2)"},
        "roofline": {"bound": "hbm",
                     "kernel": kv_kernel,
                     "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_source": peak_kind, "traffic": None},
        "bytes_per_token": nbytes, "gpu_launches": kv_launches * args.steps,
        "clocks": clk,
    }))


def run_ring_op(args):
    """The small per-layer operations (weights smaller than L2), each timed
    back to back over a ring of distinct weight copies totalling at least four
    times the L2 size (so every call streams its weights from HBM): as a CUDA
    graph of the calls, replayed (the reported value: no host work between
    calls), and launched from the host one call at a time ("stream"); and
    isolated, one call after an L2 flush (a write of twice the L2 size),
    median over calls.  Algorithmic bytes: packed weights + activations read
    + outputs written (+ the FFN's intermediate written and read)."""
    import torch

    from quantized_weight_streaming_q4k_gb300 import build, ops, synth
    build.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 1024 * 1024)
    H, I = 2560, 10240
    qd, kd = 8 * 256, 4 * 256
    if args.batch != 1:
        raise SystemExit(f"--op {args.op} runs at batch 1")
    g = synth.rng(synth.W_LM_HEAD, 1)
    if args.op == "matvec_q4k":
        mats = [synth.q4_k_matrix(g, H, H)]
        x = torch.from_numpy(synth.normal_vector(g, H)).to(dev)
        y = torch.empty(H, device=dev)

        def call(ws):
            ops.q4k_matvec(ws[0], x, H, H, out=y)
        launches = 1
        nbytes = synth.n_blocks(synth.Q4_K, H, H) * 144 + H * 4 + H * 4
        kernel = "matvec_kernel<UnitQ4K, EpiStore>"
        workload = f"Q4_K matvec {H}x{H}, batch 1"
    elif args.op == "qkv":
        mats = [synth.q4_k_matrix(g, qd, H), synth.q4_k_matrix(g, kd, H),
                synth.q4_k_matrix(g, kd, H), synth.q4_k_matrix(g, H, qd)]
        x = torch.from_numpy(synth.normal_vector(g, H)).to(dev)
        a = torch.from_numpy(synth.normal_vector(g, qd)).to(dev)
        q = torch.empty(qd, device=dev)
        k = torch.empty(kd, device=dev)
        v = torch.empty(kd, device=dev)
        o = torch.empty(H, device=dev)

        def call(ws):
            ops.q4k_qkv_proj(ws[0], ws[1], ws[2], x, H, qd, kd, out=(q, k, v))
            ops.q4k_matvec(ws[3], a, H, qd, out=o)
        launches = 2
        nbytes = (synth.n_blocks(synth.Q4_K, qd + 2 * kd, H) * 144 + H * 4 + (qd + 2 * kd) * 4
                  + synth.n_blocks(synth.Q4_K, H, qd) * 144 + qd * 4 + H * 4)
        kernel = "matvec_kernel<UnitQ4K, EpiStore> (QKV: three segments in one launch; then O)"
        workload = (f"fused QKV Q4_K {qd}+{kd}+{kd} x {H} and O projection {H}x{qd}, batch 1")
    elif args.op == "ffn":
        gl = synth.rng(synth.W_FFN, 0)
        mats = [synth.q4_k_matrix(gl, I, H), synth.q4_k_matrix(gl, I, H),
                synth.q6_k_matrix(gl, H, I)]
        x = torch.from_numpy(synth.unit_rms_vector(gl, H)).to(dev)
        y = torch.empty(H, device=dev)
        wsp = torch.empty(ops.workspace_bytes(ops.OP_FFN, 0, H, I), dtype=torch.uint8, device=dev)

        def call(ws):
            ops.q4k_ffn_gate_up_geglu_down(ws[0], ws[1], ws[2], ops.Q6_K, x, H, I, workspace=wsp,
                                           out=y)
        launches = 2
        nbytes = (2 * synth.n_blocks(synth.Q4_K, I, H) * 144 + synth.n_blocks(synth.Q6_K, H, I) * 210
                  + H * 4 + 2 * I * 4 + H * 4)
        kernel = ("matvec_kernel<UnitQ4K, EpiGeglu> (gate+up) + matvec_kernel<UnitQ6K, EpiStore> "
                  "(down)")
        workload = f"fused FFN hidden {H} inter {I}, Q4_K gate/up, GEGLU, Q6_K down, batch 1"
    else:
        raise SystemExit(f"unknown --op {args.op}")
    wbytes = sum(m.nbytes for m in mats)
    n_copies = max(2, -(-4 * l2 // wbytes))
    base = [torch.from_numpy(m).to(dev) for m in mats]
    ring = [base] + [[t.clone() for t in base] for _ in range(n_copies - 1)]
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for i in range(max(3, args.warmup)):
        call(ring[i % n_copies])
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    # isolated: one call after an L2 flush, median over calls
    n_iso = min(200, max(20, args.steps // 10))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_iso)]
    for i, (ea, eb) in enumerate(evs):
        flush.zero_()
        ea.record(stream)
        call(ring[i % n_copies])
        eb.record(stream)
    torch.cuda.synchronize()
    iso_us = statistics.median(1e3 * ea.elapsed_time(eb) for ea, eb in evs)
    # back to back over the ring, launched from the host one call at a time
    uuid = str(getattr(props, "uuid", "") or "")
    clocks = ClockSampler((uuid if uuid.startswith("GPU-") else f"GPU-{uuid}") if uuid else "0")
    clocks.start()
    ta, tb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ta.record(stream)
    for i in range(args.steps):
        call(ring[i % n_copies])
    tb.record(stream)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    us_stream = 1e3 * ta.elapsed_time(tb) / args.steps
    # back to back over the ring as a CUDA graph (the same calls captured once,
    # replayed): no host work between calls
    per_graph = n_copies * max(1, -(-32 // n_copies))
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(per_graph):
            call(ring[i % n_copies])
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for i in range(per_graph):
            call(ring[i % n_copies])
    reps = max(3, -(-args.steps // per_graph))
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    ta.record(stream)
    for _ in range(reps):
        graph.replay()
    tb.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert ops.device_error() == 0
    us = 1e3 * ta.elapsed_time(tb) / (reps * per_graph)
    gbs = nbytes / (us * 1e-6) / 1e9
    peak, peak_kind = peaks()
    print(json.dumps({
        "metric": f"{args.op} achieved HBM GB/s", "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "us_per_call": us,
        "higher_is_better": True, "dtype": "f32", "data": "synthetic (seeded random blocks)",
        "config": {"workload": workload, "batch": 1,
                   "l2": f"back to back over a ring of {n_copies} distinct weight copies "
                         f"({n_copies * wbytes / 1e6:.0f} MB >= 4 x L2 of {l2 / 1e6:.0f} MB)",
                   "method": f"CUDA graph of {per_graph} calls over the ring, replayed {reps} "
                             f"times"},
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": gbs, "peak": peak,
                     "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_kind,
                     "traffic": None},
        "isolated": {"us_per_call": iso_us, "gbs": nbytes / (iso_us * 1e-6) / 1e9,
                     "frac": nbytes / (iso_us * 1e-6) / 1e9 / peak,
                     "method": f"one call after a {2 * l2 / 1e6:.0f} MB L2 flush, median of "
                               f"{n_iso}"},
        "stream": {"us_per_call": us_stream, "gbs": nbytes / (us_stream * 1e-6) / 1e9,
                   "frac": nbytes / (us_stream * 1e-6) / 1e9 / peak,
                   "method": "the same calls launched from the host one at a time"},
        "bytes_per_call": nbytes, "gpu_launches": launches * reps * per_graph, "clocks": clk,
    }))


def run_op(args):
    """One operation timed alone, back to back (weights > L2, so every call
    streams them from HBM).  Algorithmic bytes: packed weights + activations
    read + outputs written."""
    import torch

    from quantized_weight_streaming_q4k_gb300 import build, ops, synth
    build.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    H, I, B = 2560, 10240, args.batch
    g = synth.rng(synth.W_LM_HEAD, 0)
    launches = 1
    if args.op in ("lm_head_q4_k", "lm_head_q6_k"):
        fmt = synth.Q4_K if args.op == "lm_head_q4_k" else synth.Q6_K
        W = torch.from_numpy(synth.matrix(fmt, g, VOCAB, H)).to(dev)
        x = torch.from_numpy(synth.normal_vector(g, H, B if B > 1 else None)).to(dev)
        y = torch.empty((B, VOCAB) if B > 1 else (VOCAB,), device=dev)
        ws = None
        if B * H // 64 > 320:
            raise SystemExit("batch too large for one pass at hidden 2560")

        def call():
            ops.matvec(fmt, W, x, VOCAB, H, B, 1, ws, out=y)
        nbytes = synth.n_blocks(fmt, VOCAB, H) * synth.BLOCK_BYTES[fmt] + B * H * 4 + B * VOCAB * 4
        kernel = f"matvec_kernel<{'UnitQ4K' if fmt == synth.Q4_K else 'UnitQ6K'}> (f32 activations)"
        if fmt == synth.Q4_K and 2 <= B <= 8:
            kernel = "batch_q4_matvec_kernel<12> (f32 activations, decode once for all vectors)"
        workload = f"matvec {VOCAB}x{H} {'Q4_K' if fmt == synth.Q4_K else 'Q6_K'}, batch {B}"
    elif args.op in ("lm_head_q4_0", "lm_head_q8"):
        W = torch.from_numpy(synth.q4_0_matrix(g, VOCAB, H)).to(dev)
        x = torch.from_numpy(synth.normal_vector(g, H, B if B > 1 else None)).to(dev)
        y = torch.empty((B, VOCAB) if B > 1 else (VOCAB,), device=dev)
        wbytes = synth.n_blocks(synth.Q4_0, VOCAB, H) * 18
        if args.op == "lm_head_q4_0":
            split = 0
            ws = None
            if B * H // 64 > 320:
                nbytes = ops.workspace_bytes(ops.OP_MATVEC, VOCAB, H, 0, B, 0)
                ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)

            def call():
                ops.q4_0_matvec(W, x, VOCAB, H, B, split, ws, out=y)
            nbytes = wbytes + B * H * 4 + B * VOCAB * 4
            kernel = ("batch_q4_matvec_kernel<2> (f32 activations, decode once for all vectors)"
                      if 2 <= B <= 8 else "matvec_kernel<UnitQ40> (f32 activations)")
        else:
            xq = torch.empty((B, H // 32 * 34) if B > 1 else (H // 32 * 34,), dtype=torch.uint8,
                             device=dev)

            def call():
                ops.quantize_q8_0(x, H, B, out=xq)
                ops.q8_matvec(ops.Q4_0, W, xq, VOCAB, H, B, out=y)
            launches = 2
            # quantize reads x, writes xq; the matvec reads W and xq, writes y
            nbytes = wbytes + B * H * 4 + 2 * B * (H // 32 * 34) + B * VOCAB * 4
            kernel = ("quantize_q8_0_kernel + batch_q4_matvec_kernel<102> (decode once for all "
                      "vectors)" if 2 <= B <= 8 else
                      "quantize_q8_0_kernel + matvec_kernel<UnitQ40xQ8>")
        workload = f"lm_head {VOCAB}x{H} Q4_0, batch {B}"
    elif args.op == "kv_attention":
        nq, nkv, hd, L = 8, 4, 256, 32768
        gk = synth.rng(synth.W_CHAIN, 7)
        kc = torch.from_numpy(gk.standard_normal((nkv, L, hd)).astype(np.float32)).to(dev)
        vc = torch.from_numpy(gk.standard_normal((nkv, L, hd)).astype(np.float32)).to(dev)
        x = torch.from_numpy(gk.standard_normal((nq, hd)).astype(np.float32)).to(dev)
        y = torch.empty((nq, hd), device=dev)
        ws = torch.empty(ops.workspace_bytes(ops.OP_KV_ATTENTION, L, hd, nq, nkv),
                         dtype=torch.uint8, device=dev)

        def call():
            ops.kv_attention(x, kc, vc, nq, nkv, hd, L, L, 1.0 / 16, workspace=ws, out=y)
        launches = 2
        nbytes = 2 * nkv * L * hd * 4 + 2 * nq * hd * 4
        kernel = "kv_attention_split_kernel<8> + kv_attention_merge_kernel"
        workload = f"kv_attention, {L} positions, {nq} query / {nkv} kv heads of {hd}"
        if B != 1:
            raise SystemExit("--op kv_attention runs one query token")
    elif args.op == "prefill":
        rows, N = I, B
        W = torch.from_numpy(synth.q4_k_matrix(g, rows, H)).to(dev)
        x = torch.from_numpy(synth.normal_vector(g, H, N)).to(dev)
        y = torch.empty((N, rows), device=dev)
        ws = torch.empty(ops.workspace_bytes(ops.OP_PREFILL, 0, H, 0, N), dtype=torch.uint8,
                         device=dev)

        def call():
            ops.q4k_prefill_matmul(W, x, rows, H, N, workspace=ws, out=y)
        launches = 2
        nbytes = synth.n_blocks(synth.Q4_K, rows, H) * 144 + N * H * 4 + N * rows * 4
        flops = 2.0 * rows * H * N
        kernel = ("prefill_q4k_kernel (tcgen05 kind::f16, operands split into f16 hi + lo: "
                  "3 MMAs per product) + prefill_pack_x_kernel")
        workload = f"prefill Q4_K {rows}x{H}, {N} tokens"
    else:
        raise SystemExit(f"unknown --op {args.op}")
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    props = torch.cuda.get_device_properties(dev)
    uuid = str(getattr(props, "uuid", "") or "")
    clocks = ClockSampler((uuid if uuid.startswith("GPU-") else f"GPU-{uuid}") if uuid else "0")
    clocks.start()
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(args.steps):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert ops.device_error() == 0
    us = 1e3 * a.elapsed_time(b) / args.steps
    gbs = nbytes / (us * 1e-6) / 1e9
    peak, peak_kind = peaks()
    if args.op == "prefill":
        tfs = flops / (us * 1e-6) / 1e12
        tpeak, tkind = tensor_peak()
        print(json.dumps({
            "metric": "prefill achieved TFLOP/s", "value": tfs, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": max(3, args.warmup), "us_per_call": us,
            "higher_is_better": True,
            "dtype": "f16 hi + lo operand splits (3 tensor products each), f32 accumulation",
            "tensor_tflops_executed": 3 * tfs,
            "data": "synthetic (seeded random blocks)",
            "config": {"workload": workload, "batch": B,
                       "l2": "back to back; weights 14.7 MB (L2-resident across calls)"},
            "roofline": {"bound": "tensor", "kernel": kernel, "achieved": tfs, "peak": tpeak,
                         "unit": "TFLOP/s", "frac": tfs / tpeak, "peak_source": tkind,
                         "traffic": None},
            "hbm_gbs": gbs, "gpu_launches": launches * args.steps, "clocks": clk,
        }))
        return
    print(json.dumps({
        "metric": f"{args.op} achieved HBM GB/s", "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(3, args.warmup), "us_per_call": us,
        "higher_is_better": True, "dtype": "f32", "data": "synthetic (seeded random blocks)",
        "config": {"workload": workload, "batch": B,
                   "l2": "back to back; weights larger than L2"},
        "roofline": {"bound": "hbm", "kernel": kernel, "achieved": gbs, "peak": peak,
                     "unit": "GB/s", "frac": gbs / peak, "peak_source": peak_kind,
                     "traffic": None},
        "bytes_per_call": nbytes, "gpu_launches": launches * args.steps, "clocks": clk,
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--n-layers", type=int, default=N_LAYERS,
                    help="chain length (default 34; shorter only for profiler captures)")
    ap.add_argument("--op", default="step",
                    choices=["step", "lm_head_q4_0", "lm_head_q8", "lm_head_q4_k",
                             "lm_head_q6_k", "matvec_q4k", "qkv", "ffn", "prefill",
                             "kv_attention", "decode_kv"],
                    help="step (default): the decode step; otherwise one operation alone")
    ap.add_argument("--batch", type=int, default=1, help="activation vectors (--op only)")
    ap.add_argument("--pos", type=int, default=1024,
                    help="--op decode_kv: position of the token (pos cached positions before it)")
    args = ap.parse_args()
    if args.op in ("matvec_q4k", "qkv", "ffn"):
        run_ring_op(args)
        return
    if args.op == "decode_kv":
        run_decode_kv(args)
        return
    if args.op != "step":
        run_op(args)
        return
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
